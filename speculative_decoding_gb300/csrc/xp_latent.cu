// xp_latent.cu -- the latent stage of one Jacobi pass as three tcgen05 GEMM
// kernels with fused prologues/epilogues.
//
// Method (vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels,
// _xpress_latent_kernel): for every block n and slot b,
//   prev = b == 0 ? am1[n] : blk[n, b-1]
//   x[b]  = hcache[n, b] + E[prev] @ W_lat                    (fp32 accumulate)
//   u[b]  = sum_{j <= b} L[b, j, :] * x[j]                    (per channel)
//   ub    = bf16(u);  g = ub @ Wg;  v = ub @ Wu;  m = bf16(g * sigmoid(g) * v)
//   lat[n, b-1] = bf16(u[b] + m @ Wd)                         (b = 1..B-1)
//
// GB300 design.  The pages' kernel runs one program per block and makes one
// SM pull all the weights; here the weights are spread over the whole GPU:
//   proj_mix  : M tiles of whole blocks (128 rows) x 128 latent channels,
//               the D-long reduction split over an 8-CTA cluster.  Warps 2..5
//               gather the embedding rows of the previous tokens straight into
//               128-byte-swizzled shared memory, warp 0 streams W_lat with TMA,
//               warp 1 issues tcgen05.mma into TMEM.  The partial sums meet in
//               distributed shared memory, summed in a fixed order; each CTA
//               then adds the hidden cache and applies the causal mixer to
//               its share of the blocks and writes u (fp32) and bf16(u).
//   mlp_up    : ub @ Wg and ub @ Wu as two TMEM accumulators over the same A
//               tile; the epilogue applies SiLU(g) * v and rounds to bf16.
//   mlp_down  : m @ Wd with the H-long reduction split over a cluster; the
//               reduction adds the fp32 residual u and writes bf16 latents for
//               slots 1..B-1.
// The three launches are chained with programmatic dependent launch.
#include "xp_common.cuh"
#include "xp_internal.h"
#include "xp_ptx.cuh"
#include "xp_tma.cuh"

namespace xp {

constexpr int LT_BM = 128;                          // rows per M tile
constexpr int LT_BK = 64;                           // K per chunk (one 128-byte swizzle row)
constexpr int LT_THREADS = 192;                     // warp 0 TMA, warp 1 MMA, warps 2..5 workers
constexpr uint32_t LT_A_CHUNK = LT_BM * LT_BK * 2;  // 16 KB
constexpr uint32_t LT_BOX = 64 * 64 * 2;            // one 64 x 64 bf16 box (8 KB)
constexpr int LT_MAX_B = 16;
constexpr int LT_MAX_S = 8;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// bf16 bits -> float
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// ============================================================================
// proj_mix: x = hcache + E[prev] @ W_lat, then the causal mixer
// ============================================================================
struct ProjParams {
  const int64_t* blk;
  const int64_t* am1;
  const uint16_t* hcache;
  const uint16_t* E;
  const float* L;
  float* u;
  uint16_t* ub;
  WsHeader* hdr;
  int32_t N, B, V, D, R, bpt, tn, S, chunks, ntiles, stages;
};

__global__ void __launch_bounds__(LT_THREADS, 1)
proj_mix_kernel(const __grid_constant__ CUtensorMap mapWlat, const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t b_bytes = (uint32_t)p.tn * LT_BK * 2;
  const uint32_t stage_bytes = LT_A_CHUNK + b_bytes;
  const int red_ld = p.tn + 1;  // padded row of the partial-sum buffer
  const size_t ring = (size_t)p.stages * stage_bytes;
  const size_t red_bytes = (size_t)LT_BM * red_ld * 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (ring > red_bytes ? ring : red_bytes));
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  float* red = reinterpret_cast<float*>(smem);  // reuses the ring once the MMAs are done

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = (int)(blockIdx.x % p.S);
  const int nt = (int)((blockIdx.x / p.S) % p.ntiles);
  const int mt = (int)(blockIdx.x / (p.S * p.ntiles));
  const int c0 = (int)((int64_t)ks * p.chunks / p.S);
  const int nck = (int)((int64_t)(ks + 1) * p.chunks / p.S) - c0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 2);  // the gathering warp + the W_lat TMA
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // blk may have been written by the preceding pass

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&mapWlat);
      for (int i = 0; i < nck; ++i) {
        const uint32_t s = i % p.stages, k = i / p.stages;
        if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) {
          flag_error(p.hdr, XP_DEVERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], b_bytes);
        uint8_t* dst = smem + (size_t)s * stage_bytes + LT_A_CHUNK;
        for (int bx = 0; bx < p.tn / 64; ++bx)
          tma_load_2d(dst + bx * LT_BOX, &mapWlat, nt * p.tn + bx * 64, (c0 + i) * LT_BK, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(LT_BM, p.tn, 0, 1);
      bool dead = false;
      for (int i = 0; i < nck; ++i) {
        const uint32_t s = i % p.stages, k = i / p.stages;
        if (!mbar_wait(&full[s], k & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + (size_t)s * stage_bytes);
        const uint32_t b_base = a_base + LT_A_CHUNK;
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk) {
          const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(b_base + kk * 2048, LT_BOX, 1024);
          tc_mma_f16(tmem, adesc, bdesc, idesc, (i | kk) != 0);
        }
        tc_commit(&empty[s]);
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      tc_commit(acc_full);
    }
  } else {
    // gather: warp gw fills chunks i = gw, gw+4, ...; lane owns rows lane+32j
    const int gw = warp - 2;
    int64_t prev[4];
    bool valid[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = lane + 32 * j;
      const int bl = r / p.B, b = r - bl * p.B;
      const int n = mt * p.bpt + bl;
      valid[j] = bl < p.bpt && n < p.N;
      prev[j] = 0;
      if (valid[j]) {
        int64_t t = (b == 0) ? p.am1[n] : p.blk[(int64_t)n * p.B + b - 1];
        if (t < 0 || t >= p.V) {
          flag_error(p.hdr, XP_DEVERR_TOKEN);
          t = t < 0 ? 0 : p.V - 1;
        }
        prev[j] = t;
      }
    }
    for (int i = gw; i < nck; i += 4) {
      const uint32_t s = i % p.stages, k = i / p.stages;
      if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) {
        flag_error(p.hdr, XP_DEVERR_TIMEOUT);
        break;
      }
      uint8_t* dst = smem + (size_t)s * stage_bytes;
      const int kel0 = (c0 + i) * LT_BK;
      uint4 v[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          v[j][c] = make_uint4(0, 0, 0, 0);
          if (valid[j] && kel0 + 8 * c < p.D)
            v[j][c] = *reinterpret_cast<const uint4*>(p.E + prev[j] * p.D + kel0 + 8 * c);
        }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = v[j][c];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[s]);
    }
  }

  // ---- epilogue 1: the partial sums TMEM -> shared memory (warps 2..5)
  if (warp >= 2) {
    if (!mbar_wait(acc_full, 0)) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    tc_fence_after();
    const int q = warp & 3, row = q * 32 + lane;
    for (int c = 0; c < p.tn / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) red[row * red_ld + c * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  cluster_sync();

  // ---- epilogue 2: sum the cluster's partials, add hcache, causal mixer
  if (threadIdx.x >= 64) {
    const int c = threadIdx.x - 64;
    const int col = nt * p.tn + c;
    if (c < p.tn && col < p.R) {
      for (int bl = ks; bl < p.bpt; bl += p.S) {
        const int n = mt * p.bpt + bl;
        if (n >= p.N) break;
        // all of the block's partial sums are requested before any is used,
        // so the distributed-shared-memory latencies overlap
        float v[LT_MAX_B][LT_MAX_S];
#pragma unroll
        for (int b = 0; b < LT_MAX_B; ++b)
#pragma unroll
          for (int q = 0; q < LT_MAX_S; ++q)
            v[b][q] = (b < p.B && q < p.S) ? ld_dsmem_f32(&red[(bl * p.B + b) * red_ld + c], (uint32_t)q) : 0.f;
        float x[LT_MAX_B];
#pragma unroll
        for (int b = 0; b < LT_MAX_B; ++b) {
          x[b] = 0.f;
          if (b < p.B) {
            float acc = v[b][0];
#pragma unroll
            for (int q = 1; q < LT_MAX_S; ++q) acc += v[b][q];
            x[b] = bf2f(p.hcache[((int64_t)n * p.B + b) * p.R + col]) + acc;
          }
        }
#pragma unroll
        for (int b = 0; b < LT_MAX_B; ++b) {
          if (b < p.B) {
            float uu = 0.f;
#pragma unroll
            for (int j = 0; j <= b; ++j) uu = fmaf(p.L[((int64_t)b * p.B + j) * p.R + col], x[j], uu);
            const int64_t o = ((int64_t)n * p.B + b) * p.R + col;
            p.u[o] = uu;
            p.ub[o] = (uint16_t)(f32x2_to_bf16x2(uu, 0.f) & 0xffffu);
          }
        }
      }
    }
  }
  cluster_sync();  // the peers have finished reading this CTA's partials
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ============================================================================
// mlp_up: m = bf16(silu(ub @ Wg) * (ub @ Wu)), 64 hidden columns per CTA
// ============================================================================
struct UpParams {
  uint16_t* m;
  WsHeader* hdr;
  int32_t rows, H, chunks, htiles, stages;
};

__global__ void __launch_bounds__(LT_THREADS, 1)
mlp_up_kernel(const __grid_constant__ CUtensorMap mapUb, const __grid_constant__ CUtensorMap mapWg,
              const __grid_constant__ CUtensorMap mapWu, const UpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  constexpr uint32_t stage_bytes = LT_A_CHUNK + 2 * LT_BOX;  // 32 KB
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * stage_bytes);
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ht = (int)(blockIdx.x % p.htiles);
  const int mt = (int)(blockIdx.x / p.htiles);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);  // g: columns [0, 64), v: [64, 128)
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // ub comes from proj_mix

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&mapUb);
      prefetch_tensormap(&mapWg);
      prefetch_tensormap(&mapWu);
      for (int i = 0; i < p.chunks; ++i) {
        const uint32_t s = i % p.stages, k = i / p.stages;
        if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) {
          flag_error(p.hdr, XP_DEVERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        uint8_t* dst = smem + (size_t)s * stage_bytes;
        tma_load_2d(dst, &mapUb, i * LT_BK, mt * LT_BM, &full[s]);
        tma_load_2d(dst + LT_A_CHUNK, &mapWg, ht * 64, i * LT_BK, &full[s]);
        tma_load_2d(dst + LT_A_CHUNK + LT_BOX, &mapWu, ht * 64, i * LT_BK, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(LT_BM, 64, 0, 1);
      bool dead = false;
      for (int i = 0; i < p.chunks; ++i) {
        const uint32_t s = i % p.stages, k = i / p.stages;
        if (!mbar_wait(&full[s], k & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + (size_t)s * stage_bytes);
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk) {
          const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t gdesc = smem_desc_sw128(a_base + LT_A_CHUNK + kk * 2048, LT_BOX, 1024);
          const uint64_t vdesc = smem_desc_sw128(a_base + LT_A_CHUNK + LT_BOX + kk * 2048, LT_BOX, 1024);
          tc_mma_f16(tmem, adesc, gdesc, idesc, (i | kk) != 0);
          tc_mma_f16(tmem + 64, adesc, vdesc, idesc, (i | kk) != 0);
        }
        tc_commit(&empty[s]);
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      tc_commit(acc_full);
    }
  } else {
    if (!mbar_wait(acc_full, 0)) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    tc_fence_after();
    const int q = warp & 3;
    const int row = mt * LT_BM + q * 32 + lane;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t g[32], v[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, g);
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + 64 + c * 32, v);
      tmem_ld_wait();
      if (row < p.rows) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float g0 = __uint_as_float(g[2 * e]), g1 = __uint_as_float(g[2 * e + 1]);
          const float m0 = g0 / (1.f + expf(-g0)) * __uint_as_float(v[2 * e]);
          const float m1 = g1 / (1.f + expf(-g1)) * __uint_as_float(v[2 * e + 1]);
          w[e] = f32x2_to_bf16x2(m0, m1);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.m + (int64_t)row * p.H + ht * 64 + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ============================================================================
// mlp_down: lat = bf16(u + m @ Wd) for slots 1..B-1
// ============================================================================
struct DownParams {
  const float* u;
  uint16_t* lat;
  WsHeader* hdr;
  int32_t N, B, R, tn, S, chunks, ntiles, stages;
};

__global__ void __launch_bounds__(LT_THREADS, 1)
mlp_down_kernel(const __grid_constant__ CUtensorMap mapM, const __grid_constant__ CUtensorMap mapWd,
                const DownParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t b_bytes = (uint32_t)p.tn * LT_BK * 2;
  const uint32_t stage_bytes = LT_A_CHUNK + b_bytes;
  const int red_ld = p.tn + 1;
  const size_t ring = (size_t)p.stages * stage_bytes;
  const size_t red_bytes = (size_t)LT_BM * red_ld * 4;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (ring > red_bytes ? ring : red_bytes));
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  float* red = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = (int)(blockIdx.x % p.S);
  const int nt = (int)((blockIdx.x / p.S) % p.ntiles);
  const int mt = (int)(blockIdx.x / (p.S * p.ntiles));
  const int c0 = (int)((int64_t)ks * p.chunks / p.S);
  const int nck = (int)((int64_t)(ks + 1) * p.chunks / p.S) - c0;
  const int rows = p.N * p.B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();  // m comes from mlp_up

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&mapM);
      prefetch_tensormap(&mapWd);
      for (int i = 0; i < nck; ++i) {
        const uint32_t s = i % p.stages, k = i / p.stages;
        if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) {
          flag_error(p.hdr, XP_DEVERR_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        uint8_t* dst = smem + (size_t)s * stage_bytes;
        tma_load_2d(dst, &mapM, (c0 + i) * LT_BK, mt * LT_BM, &full[s]);
        for (int bx = 0; bx < p.tn / 64; ++bx)
          tma_load_2d(dst + LT_A_CHUNK + bx * LT_BOX, &mapWd, nt * p.tn + bx * 64, (c0 + i) * LT_BK, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(LT_BM, p.tn, 0, 1);
      bool dead = false;
      for (int i = 0; i < nck; ++i) {
        const uint32_t s = i % p.stages, k = i / p.stages;
        if (!mbar_wait(&full[s], k & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + (size_t)s * stage_bytes);
        const uint32_t b_base = a_base + LT_A_CHUNK;
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk) {
          const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(b_base + kk * 2048, LT_BOX, 1024);
          tc_mma_f16(tmem, adesc, bdesc, idesc, (i | kk) != 0);
        }
        tc_commit(&empty[s]);
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      tc_commit(acc_full);
    }
  } else {
    if (!mbar_wait(acc_full, 0)) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    tc_fence_after();
    const int q = warp & 3, row = q * 32 + lane;
    for (int c = 0; c < p.tn / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) red[row * red_ld + c * 32 + e] = __uint_as_float(r[e]);
    }
  }
  tc_fence_before();
  cluster_sync();

  // ---- sum the cluster's partials, add the residual, write slots 1..B-1
  if (threadIdx.x >= 64) {
    const int c = threadIdx.x - 64;
    const int col = nt * p.tn + c;
    if (c < p.tn && col < p.R) {
      const int r0 = ks * LT_BM / p.S, r1 = (ks + 1) * LT_BM / p.S;
      // rows in groups of 8, every partial of a group requested before use
      for (int g0 = r0; g0 < r1; g0 += 8) {
        float v[8][LT_MAX_S];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int q = 0; q < LT_MAX_S; ++q)
            v[i][q] = (g0 + i < r1 && q < p.S) ? ld_dsmem_f32(&red[(g0 + i) * red_ld + c], (uint32_t)q) : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = g0 + i;
          const int grow = mt * LT_BM + row;
          if (row >= r1 || grow >= rows) break;
          const int n = grow / p.B, b = grow - n * p.B;
          if (b == 0) continue;
          float acc = v[i][0];
#pragma unroll
          for (int q = 1; q < LT_MAX_S; ++q) acc += v[i][q];
          const float y = p.u[(int64_t)grow * p.R + col] + acc;
          p.lat[((int64_t)n * (p.B - 1) + b - 1) * p.R + col] = (uint16_t)(f32x2_to_bf16x2(y, 0.f) & 0xffffu);
        }
      }
    }
  }
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ============================================================================
// host side
// ============================================================================
namespace {

bool g_lt_attr[64];

cudaError_t launch_ex(const void* kernel_fn, dim3 grid, size_t smem, cudaStream_t stream, int cluster, void** args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = cluster;
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.gridDim = grid;
  cfg.blockDim = dim3(LT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelExC(&cfg, kernel_fn, args);
}

int pick_stages(uint32_t stage_bytes, int chunks_per_cta, size_t min_ring) {
  int st = chunks_per_cta < 6 ? chunks_per_cta : 6;
  if (st < 2) st = 2;
  while ((size_t)st * stage_bytes < min_ring) ++st;
  return st;
}

}  // namespace

// The latent's tile width over R: 128 channels, or R rounded up to 64 when R
// is smaller (the TMA zero-fills the missing weight columns).
static int latent_tn(int64_t R) { return R >= 128 ? 128 : 64; }

xp_status launch_latent(const int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
                        const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
                        const uint16_t* Wd, uint16_t* lat_out, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R,
                        int64_t H, void* ws, cudaStream_t stream) {
  if (N <= 0) return XP_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return XP_ERR_LAUNCH;
  if (!g_lt_attr[dev]) {
    int max_smem = 0;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return XP_ERR_LAUNCH;
    if (cudaFuncSetAttribute(proj_mix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(mlp_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) != cudaSuccess ||
        cudaFuncSetAttribute(mlp_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem) !=
            cudaSuccess)
      return XP_ERR_LAUNCH;
    g_lt_attr[dev] = true;
  }
  const LatentWsLayout lay = latent_ws_layout(N, B, R, H);
  char* w = static_cast<char*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  float* u = reinterpret_cast<float*>(w + lay.u);
  uint16_t* ub = reinterpret_cast<uint16_t*>(w + lay.ub);
  uint16_t* m = reinterpret_cast<uint16_t*>(w + lay.m);
  const int tn = latent_tn(R);
  const int ntiles = (int)((R + tn - 1) / tn);
  const int rows = (int)(N * B);

  // ---- proj_mix
  {
    ProjParams p;
    p.blk = blk;
    p.am1 = am1;
    p.hcache = hcache;
    p.E = E;
    p.L = L;
    p.u = u;
    p.ub = ub;
    p.hdr = hdr;
    p.N = (int32_t)N;
    p.B = (int32_t)B;
    p.V = (int32_t)V;
    p.D = (int32_t)D;
    p.R = (int32_t)R;
    p.bpt = (int32_t)(LT_BM / B);
    p.tn = tn;
    p.chunks = (int32_t)((D + LT_BK - 1) / LT_BK);
    p.S = p.chunks < LT_MAX_S ? p.chunks : LT_MAX_S;
    p.ntiles = ntiles;
    const uint32_t stage_bytes = LT_A_CHUNK + (uint32_t)tn * LT_BK * 2;
    const int per_cta = (p.chunks + p.S - 1) / p.S;
    p.stages = pick_stages(stage_bytes, per_cta, (size_t)LT_BM * (tn + 1) * 4);
    const size_t smem = 1024 + (size_t)p.stages * stage_bytes + 8 * (2 * p.stages + 1) + 16;
    const int mtiles = (int)((N + p.bpt - 1) / p.bpt);
    CUtensorMap mapWlat;
    if (!cached_map_bf16_2d(&mapWlat, W_lat, (uint64_t)R, (uint64_t)D, (uint64_t)R, 64, LT_BK)) return XP_ERR_LAUNCH;
    void* args[] = {&mapWlat, &p};
    if (launch_ex((const void*)proj_mix_kernel, dim3((unsigned)(mtiles * ntiles * p.S)), smem, stream, p.S, args) !=
        cudaSuccess)
      return XP_ERR_LAUNCH;
  }
  // ---- mlp_up
  {
    UpParams p;
    p.m = m;
    p.hdr = hdr;
    p.rows = rows;
    p.H = (int32_t)H;
    p.chunks = (int32_t)((R + LT_BK - 1) / LT_BK);
    p.htiles = (int32_t)(H / 64);
    p.stages = pick_stages(LT_A_CHUNK + 2 * LT_BOX, p.chunks, 0);
    const size_t smem = 1024 + (size_t)p.stages * (LT_A_CHUNK + 2 * LT_BOX) + 8 * (2 * p.stages + 1) + 16;
    const int mtiles = (rows + LT_BM - 1) / LT_BM;
    CUtensorMap mapUb, mapWg, mapWu;
    if (!cached_map_bf16_2d(&mapUb, ub, (uint64_t)R, (uint64_t)rows, (uint64_t)R, LT_BK, LT_BM) ||
        !cached_map_bf16_2d(&mapWg, Wg, (uint64_t)H, (uint64_t)R, (uint64_t)H, 64, LT_BK) ||
        !cached_map_bf16_2d(&mapWu, Wu, (uint64_t)H, (uint64_t)R, (uint64_t)H, 64, LT_BK))
      return XP_ERR_LAUNCH;
    void* args[] = {&mapUb, &mapWg, &mapWu, &p};
    if (launch_ex((const void*)mlp_up_kernel, dim3((unsigned)(mtiles * p.htiles)), smem, stream, 1, args) !=
        cudaSuccess)
      return XP_ERR_LAUNCH;
  }
  // ---- mlp_down
  {
    DownParams p;
    p.u = u;
    p.lat = lat_out;
    p.hdr = hdr;
    p.N = (int32_t)N;
    p.B = (int32_t)B;
    p.R = (int32_t)R;
    p.tn = tn;
    p.chunks = (int32_t)(H / LT_BK);
    p.S = p.chunks < LT_MAX_S ? p.chunks : LT_MAX_S;
    p.ntiles = ntiles;
    const uint32_t stage_bytes = LT_A_CHUNK + (uint32_t)tn * LT_BK * 2;
    const int per_cta = (p.chunks + p.S - 1) / p.S;
    p.stages = pick_stages(stage_bytes, per_cta, (size_t)LT_BM * (tn + 1) * 4);
    const size_t smem = 1024 + (size_t)p.stages * stage_bytes + 8 * (2 * p.stages + 1) + 16;
    const int mtiles = (rows + LT_BM - 1) / LT_BM;
    CUtensorMap mapM, mapWd;
    if (!cached_map_bf16_2d(&mapM, m, (uint64_t)H, (uint64_t)rows, (uint64_t)H, LT_BK, LT_BM) ||
        !cached_map_bf16_2d(&mapWd, Wd, (uint64_t)R, (uint64_t)H, (uint64_t)R, 64, LT_BK))
      return XP_ERR_LAUNCH;
    void* args[] = {&mapM, &mapWd, &p};
    if (launch_ex((const void*)mlp_down_kernel, dim3((unsigned)(mtiles * ntiles * p.S)), smem, stream, p.S, args) !=
        cudaSuccess)
      return XP_ERR_LAUNCH;
  }
  return XP_OK;
}

}  // namespace xp
