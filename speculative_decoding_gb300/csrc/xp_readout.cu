// xp_readout.cu -- the readout matmul x @ W2 with the add of the base logits,
// the bf16 rounding and the vocab-wide argmax fused into its epilogue.
//
// Method (vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels): the
// module docstring's "readout logits = base + x @ W2" followed by
// fused_add_argmax_to_blk; the caller's matmul yields a bf16 bias, so the
// accumulator is rounded to bf16 first, then added to base and rounded again
// (the sum is cast to bf16 before the compare, per
// _xpress_add_argmax_partial_kernel).  The [rows, V] bias and logits never
// reach memory.
//
// GB300 design (tcgen05 + TMA):
//   * one CTA per SM; CTA (m, j) owns M tile m (128 draft rows) and a
//     contiguous range of 256-wide vocab tiles;
//   * warp 0 (one thread) loads the CTA's 128 x R slice of lat ONCE into
//     shared memory (it stays resident) and then streams W2 in 64 x 256
//     K-chunks through a ring of stages, all with TMA (128-byte swizzle);
//   * warp 1 (one thread) issues tcgen05.mma M=128 N=256 K=16 (bf16 in, fp32
//     accumulate) into one of two 256-column TMEM accumulators, so the
//     epilogue of tile t overlaps the MMAs of tile t+1;
//   * warps 2..9 drain the accumulator with tcgen05.ld (thread = one row,
//     warp = a 32-lane quadrant and a 128-column half), round to bf16, add
//     the base logits (prefetched one tile ahead into registers), and keep a
//     running (max, first column) per row across the CTA's tiles (tiles and
//     columns ascend, so a strict '>' keeps the lowest index);
//   * each row's per-CTA winner is folded into a 64-bit (value, lowest
//     index) key with atomicMax; the last CTA to finish writes blk, counts the
//     changed slots and re-zeroes the keys.
#include "xp_common.cuh"
#include "xp_internal.h"
#include "xp_ptx.cuh"
#include "xp_tma.cuh"

namespace xp {

constexpr int RO_BM = 128;
constexpr int RO_BN = 256;
constexpr int RO_BK = 64;
constexpr int RO_EPI_WARPS = 8;
constexpr int RO_THREADS = (2 + RO_EPI_WARPS) * 32;
constexpr uint32_t RO_A_CHUNK = RO_BM * RO_BK * 2;    // 16 KB per 64-wide K chunk
constexpr uint32_t RO_B_STAGE = RO_BK * RO_BN * 2;    // 32 KB per stage
constexpr uint32_t RO_B_BOX = RO_BK * 64 * 2;         // one 64 x 64 TMA box, 8 KB
constexpr int RO_MAX_KCH = 8;                         // R <= 512

struct ReadoutParams {
  const uint16_t* base;
  int64_t ld_base;
  int32_t rows, V, kch, mt, nt, per, stages, B;
  int64_t* blk;
  int32_t* changed;
  unsigned long long* keys;
  WsHeader* hdr;
};

// One 32-column chunk of one row: acc (fp32) -> bias = bf16(acc);
// s = bf16(base + bias); update the running (best, first column).
__device__ __forceinline__ void ro_chunk(const uint32_t (&r)[32], const uint4 (&bw)[4], int col0, int V,
                                         bool all_valid, float& best, int& bidx) {
  uint32_t s2[16];
  uint32_t m2 = 0xff80ff80u;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t w[4] = {bw[v].x, bw[v].y, bw[v].z, bw[v].w};
    const bool ok = all_valid || (col0 + 8 * v < V);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int q = 4 * v + k;
      const uint32_t bias2 = f32x2_to_bf16x2(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]));
      s2[q] = bf16x2_add(w[k], bias2);
      if (ok) m2 = bf16x2_max(m2, s2[q]);
    }
  }
  const float m = fmaxf(bf16lo_to_f32(m2), bf16hi_to_f32(m2));
  if (m > best || bidx < 0) {
    int cand = -1;
#pragma unroll
    for (int q = 15; q >= 0; --q) {
      const bool ok = all_valid || (col0 + 2 * q < V);
      if (ok && bf16hi_to_f32(s2[q]) == m) cand = 2 * q + 1;
      if (ok && bf16lo_to_f32(s2[q]) == m) cand = 2 * q;
    }
    if (cand >= 0) {
      best = m;
      bidx = col0 + cand;
    }
  }
}

// base[row, n0 .. n0+127] -> 16 x 16 bytes (vectors past V are not read)
__device__ __forceinline__ void ro_load_base(uint4 (&dst)[16], const uint16_t* brow, int n0, int V, bool row_ok) {
#pragma unroll
  for (int v = 0; v < 16; ++v) {
    if (row_ok && n0 + 8 * v < V)
      dst[v] = ld_stream_v4(brow + n0 + 8 * v);
    else
      dst[v] = make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(RO_THREADS, 1)
readout_argmax_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                      const ReadoutParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)p.kch * RO_A_CHUNK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)p.stages * RO_B_STAGE);
  uint64_t* a_full = bars;
  uint64_t* b_full = bars + 1;
  uint64_t* b_empty = b_full + p.stages;
  uint64_t* acc_full = b_empty + p.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x % p.mt;
  const int jslot = blockIdx.x / p.mt;
  const int n_begin = (int)((int64_t)jslot * p.nt / p.per);
  const int n_end = (int)((int64_t)(jslot + 1) * p.nt / p.per);
  const int ntiles = n_end - n_begin;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], RO_EPI_WARPS);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      prefetch_tensormap(&mapA);
      prefetch_tensormap(&mapB);
      mbar_arrive_expect_tx(a_full, (uint32_t)p.kch * RO_A_CHUNK);
      for (int kc = 0; kc < p.kch; ++kc) tma_load_2d(sA + (size_t)kc * RO_A_CHUNK, &mapA, kc * RO_BK, m_tile * RO_BM, a_full);
      uint32_t it = 0;
      bool dead = false;
      for (int t = 0; t < ntiles && !dead; ++t) {
        const int n0 = (n_begin + t) * RO_BN;
        for (int kc = 0; kc < p.kch; ++kc, ++it) {
          const uint32_t s = it % p.stages, k = it / p.stages;
          if (k >= 1 && !mbar_wait(&b_empty[s], (k - 1) & 1)) {
            dead = true;
            flag_error(p.hdr, XP_DEVERR_TIMEOUT);
            break;
          }
          mbar_arrive_expect_tx(&b_full[s], RO_B_STAGE);
          uint8_t* dst = sB + (size_t)s * RO_B_STAGE;
#pragma unroll
          for (int nb = 0; nb < RO_BN / 64; ++nb) tma_load_2d(dst + nb * RO_B_BOX, &mapB, n0 + nb * 64, kc * RO_BK, &b_full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(RO_BM, RO_BN, 0, 1);
      bool dead = !mbar_wait(a_full, 0);
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      tc_fence_after();
      uint32_t it = 0;
      for (int t = 0; t < ntiles && !dead; ++t) {
        const uint32_t a = t & 1, u = t >> 1;
        if (u >= 1 && !mbar_wait(&acc_empty[a], (u - 1) & 1)) {
          dead = true;
          flag_error(p.hdr, XP_DEVERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + a * RO_BN;
        for (int kc = 0; kc < p.kch; ++kc, ++it) {
          const uint32_t s = it % p.stages, k = it / p.stages;
          if (!mbar_wait(&b_full[s], k & 1)) {
            dead = true;
            flag_error(p.hdr, XP_DEVERR_TIMEOUT);
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + (size_t)kc * RO_A_CHUNK);
          const uint32_t b_base = smem_u32(sB + (size_t)s * RO_B_STAGE);
#pragma unroll
          for (int kk = 0; kk < RO_BK / 16; ++kk) {
            // A: K-major, 128-byte rows, 8-row groups 1024 B apart; a K step of
            // 16 elements advances 32 bytes inside the swizzle atom.
            const uint64_t adesc = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            // B: N-major; 64-wide N blocks 8 KB apart (leading), 8-row K
            // groups 1024 B apart (stride); a K step of 16 rows is 2 KB.
            const uint64_t bdesc = smem_desc_sw128(b_base + kk * 2048, RO_B_BOX, 1024);
            tc_mma_f16(d, adesc, bdesc, idesc, (kc | kk) != 0);
          }
          tc_commit(&b_empty[s]);
        }
        if (dead) break;
        tc_commit(&acc_full[a]);
      }
      // every MMA issued above has completed once this barrier fires
      tc_commit(drain);
      (void)mbar_wait(drain, 0);
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int h = (warp - 2) >> 2;   // 128-column half of the tile
    const int row = m_tile * RO_BM + q * 32 + lane;
    const bool row_ok = row < p.rows;
    const uint16_t* brow = p.base + (int64_t)(row_ok ? row : 0) * p.ld_base;
    float best = -INFINITY;
    int bidx = -1;
    bool dead = false;
    uint4 cur[16], nxt[16];
    ro_load_base(cur, brow, n_begin * RO_BN + h * 128, p.V, row_ok);
    for (int t = 0; t < ntiles; ++t) {
      const uint32_t a = t & 1, u = t >> 1;
      const int n0 = (n_begin + t) * RO_BN + h * 128;
      if (t + 1 < ntiles) ro_load_base(nxt, brow, n0 + RO_BN, p.V, row_ok);
      if (!dead && !mbar_wait(&acc_full[a], u & 1)) {
        dead = true;
        flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      }
      tc_fence_after();
      if (!dead) {
        const bool all_valid = n0 + 128 <= p.V;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + a * RO_BN + h * 128 + c * 32, r);
          tmem_ld_wait();
          const uint4 bw[4] = {cur[4 * c], cur[4 * c + 1], cur[4 * c + 2], cur[4 * c + 3]};
          ro_chunk(r, bw, n0 + c * 32, p.V, all_valid, best, bidx);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[a]);
#pragma unroll
      for (int v = 0; v < 16; ++v) cur[v] = nxt[v];
    }
    if (row_ok && bidx >= 0 && !dead) atomicMax(&p.keys[row], make_key(best, (uint32_t)bidx));
    __threadfence();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int prev = atomicAdd(&p.hdr->done, 1u);
    s_last = (prev == gridDim.x - 1);
  }
  __syncthreads();
  if (s_last) {
    // every other CTA has folded its rows: publish the winners
    __threadfence();
    int nchanged = 0;
    for (int r = threadIdx.x; r < p.rows; r += blockDim.x) {
      const unsigned long long k = atomicExch(&p.keys[r], 0ull);
      const int64_t idx = (int64_t)key_index(k);
      const int64_t n = r / (p.B - 1), jj = r - n * (p.B - 1);
      int64_t* slot = p.blk + n * p.B + 1 + jj;
      nchanged += (*slot != idx);
      *slot = idx;
    }
    if (p.changed && nchanged) atomicAdd(p.changed, nchanged);
    __syncthreads();
    if (threadIdx.x == 0) p.hdr->done = 0u;
  }
}

size_t readout_smem_bytes(int kch, int stages) {
  return 1024 + (size_t)kch * RO_A_CHUNK + (size_t)stages * RO_B_STAGE + 8 * (2 * stages + 6) + 16;
}

xp_status launch_readout_argmax(const uint16_t* lat, const uint16_t* W2, const uint16_t* base, int64_t ld_base,
                                int64_t rows, int64_t V, int64_t R, int64_t* blk, int64_t B, int32_t* changed,
                                void* ws, cudaStream_t stream) {
  if (rows <= 0) return XP_OK;
  const int kch = (int)((R + RO_BK - 1) / RO_BK);
  if (kch > RO_MAX_KCH) return XP_ERR_SHAPE;
  int dev = 0, sms = 0, max_smem = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return XP_ERR_LAUNCH;
  int stages = 8;
  while (stages > 2 && readout_smem_bytes(kch, stages) > (size_t)max_smem) --stages;
  const size_t smem = readout_smem_bytes(kch, stages);
  if (smem > (size_t)max_smem) return XP_ERR_SHAPE;

  CUtensorMap mapA, mapB;
  if (!make_map_bf16_2d(&mapA, lat, (uint64_t)R, (uint64_t)rows, (uint64_t)R, RO_BK, RO_BM)) return XP_ERR_LAUNCH;
  if (!make_map_bf16_2d(&mapB, W2, (uint64_t)V, (uint64_t)R, (uint64_t)V, 64, RO_BK)) return XP_ERR_LAUNCH;

  ReadoutParams p;
  ArgmaxWs w = argmax_ws(ws, rows);
  p.base = base;
  p.ld_base = ld_base;
  p.rows = (int32_t)rows;
  p.V = (int32_t)V;
  p.kch = kch;
  p.mt = (int32_t)((rows + RO_BM - 1) / RO_BM);
  p.nt = (int32_t)((V + RO_BN - 1) / RO_BN);
  int per = sms / p.mt;
  if (per < 1) per = 1;
  if (per > p.nt) per = p.nt;
  p.per = per;
  p.stages = stages;
  p.B = (int32_t)B;
  p.blk = blk;
  p.changed = changed;
  p.keys = w.keys;
  p.hdr = w.hdr;
  if (cudaFuncSetAttribute(readout_argmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return XP_ERR_LAUNCH;
  readout_argmax_kernel<<<(unsigned int)(p.mt * per), RO_THREADS, smem, stream>>>(mapA, mapB, p);
  return cudaGetLastError() == cudaSuccess ? XP_OK : XP_ERR_LAUNCH;
}

}  // namespace xp
