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
//               the D-long reduction split over S ordinary CTAs (no cluster).
//               Warps 2..5 gather the embedding rows of the previous tokens
//               straight into 128-byte-swizzled shared memory, warp 0 streams
//               W_lat with TMA, warp 1 issues tcgen05.mma into TMEM.  Each CTA
//               stores its fp32 partial tile to an L2-resident buffer; the S
//               CTAs of a tile meet on an arrival counter and each sums the S
//               partials of its own column slice in a fixed order, adds the
//               hidden cache, applies the causal mixer and writes u (fp32)
//               and bf16(u).
//   mlp_up    : ub @ Wg and ub @ Wu as one N=128 MMA per K step into two
//               64-column halves of a TMEM accumulator; eight epilogue warps
//               (two per TMEM lane quadrant) apply SiLU(g) * v and round to
//               bf16.
//   mlp_down  : m @ Wd with the H-long reduction split over a cluster; the
//               reduction adds the fp32 residual u and writes bf16 latents for
//               slots 1..B-1.
// The three launches are chained with programmatic dependent launch.  One
// thread issues each kernel's MMAs, and anything else in its loop delays them
// (a barrier wait costs it about as much as three MMAs), so the issue loops
// carry the ring's stage and phase in running counters and add constants to
// per-stage descriptors instead of dividing by the stage count and rebuilding
// the descriptors for every chunk.
#include "xp_common.cuh"
#include "xp_internal.h"
#include "xp_ptx.cuh"
#include "xp_tma.cuh"
#include "xp_trace.cuh"

namespace xp {

constexpr int LT_BM = 128;                          // rows per M tile
constexpr int LT_BK = 64;                           // K per chunk (one 128-byte swizzle row)
constexpr int LT_THREADS = 192;                     // warp 0 TMA, warp 1 MMA, warps 2..5 workers (proj_mix, mlp_down)
constexpr int LT_UP_THREADS = 320;                  // mlp_up: warps 2..9 (two per TMEM lane quadrant)
constexpr uint32_t LT_A_CHUNK = LT_BM * LT_BK * 2;  // 16 KB
constexpr uint32_t LT_BOX = 64 * 64 * 2;            // one 64 x 64 bf16 box (8 KB)
constexpr int LT_MAX_B = 16;
constexpr int LT_MAX_S = 8;

// The dynamic shared-memory base rounded up to 1024 bytes, as an offset from
// the base pointer itself (not a round trip through an integer), so the
// compiler keeps knowing that the result points into shared memory and emits
// shared-memory loads and stores for every pointer derived from it.
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// bf16 bits -> float
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// ============================================================================
// proj_mix: x = hcache + E[prev] @ W_lat, then the causal mixer
// ============================================================================
// Shared memory: [0, region) is the stage ring; once the MMAs are done it holds
// the S partial-sum slices of this CTA's w columns (TMA from the partial
// buffer) and xs[128][w] (the reduced x), then the outgoing partial tile and,
// once that is stored, in the same place, the mixer output tiles us [rows][w]
// fp32 and ubs [rows][w] bf16 (TMA-stored); that place is sized for the
// larger of the two.  After it: Ls (the mixer weights of those
// columns, the [B][B] square), hcs (the hidden cache of
// those columns for the tile's 128 rows), the token table and the barriers.
//
// The S CTAs of a tile (one per slice of the D-long reduction) are ordinary
// CTAs, not a cluster: each writes its fp32 partial tile to the partial
// buffer (L2-resident), counts itself on the tile's arrival counter, waits
// (bounded) until all S have arrived, then loads the S partials of its own w
// columns and sums them in slice order.  The grid is one wave (one CTA per
// SM), so every CTA a wait depends on is resident.
struct ProjParams {
  const int64_t* blk;
  const int64_t* am1;
  const uint16_t* E;
  const float* L;
  float* u;
  uint16_t* ub;
  float* part;
  uint32_t* cnt;
  WsHeader* hdr;
  int32_t N, B, V, D, R, bpt, tn, S, w, lw, chunks, ntiles, stages;
  int32_t prow;  // rows of a partial tile that are stored and summed (128, or fewer for a lone M tile)
  int64_t rows_pad, r_pad;
  uint32_t region, hc_off, tok_off, bar_off;
  const uint32_t* skip;  // nullable: see pass_skipped
};


// kHalfL: the mixer weights of half the CTA's columns at a time (lw = w / 2)
template <bool kHalfL>
__global__ void __launch_bounds__(LT_THREADS, 1)
proj_mix_kernel(const __grid_constant__ CUtensorMap mapWlat, const __grid_constant__ CUtensorMap mapHc,
                const __grid_constant__ CUtensorMap mapPart, const __grid_constant__ CUtensorMap mapPartSt,
                const __grid_constant__ CUtensorMap mapL, const __grid_constant__ CUtensorMap mapU,
                const __grid_constant__ CUtensorMap mapUb, const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  if (pass_skipped(p.skip, true)) return;  // the first kernel of a pass
  if (threadIdx.x == 0) XP_TRACE_MARK(0);
  if (threadIdx.x == 0) XP_TRACE_SM(15);
  uint8_t* smem = align1024(smem_raw);
  const uint32_t b_bytes = (uint32_t)p.tn * LT_BK * 2;
  const uint32_t stage_bytes = LT_A_CHUNK + b_bytes;
  float* slices = reinterpret_cast<float*>(smem);     // [S][128][w]
  float* xs = slices + (size_t)p.S * LT_BM * p.w;     // [128][w]
  // this CTA's partial tile on its way out: tn/32 boxes of [128][32] fp32,
  // 128-byte swizzled (1024-byte aligned, after slices and xs)
  uint8_t* pst = smem + (((size_t)(p.S + 1) * LT_BM * p.w * 4 + 1023) & ~size_t(1023));
  float* Ls = reinterpret_cast<float*>(smem + p.region);
  const uint16_t* hcs = reinterpret_cast<const uint16_t*>(smem + p.hc_off);
  int64_t* tok = reinterpret_cast<int64_t*>(smem + p.tok_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint64_t* aux_full = acc_full + 1;    // Ls and hcs landed
  uint64_t* slice_full = aux_full + 1;  // the S partial slices landed
  uint64_t* ls_full = slice_full + 1;   // the second round of mixer weights landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ls_full + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = (int)(blockIdx.x % p.S);
  const int nt = (int)((blockIdx.x / p.S) % p.ntiles);
  const int mt = (int)(blockIdx.x / (p.S * p.ntiles));
  const int tile = mt * p.ntiles + nt;
  const int c0 = (int)((int64_t)ks * p.chunks / p.S);
  const int nck = (int)((int64_t)(ks + 1) * p.chunks / p.S) - c0;
  const int c_lo = ks * p.w;                   // this CTA's columns of the tile: [c_lo, c_lo + w)
  const int col0 = nt * p.tn + c_lo;           // ... as latent channels
  const int nbl = min(p.bpt, p.N - mt * p.bpt);  // blocks of this M tile
  // channels of this CTA's slice that exist (R is a multiple of 16, the
  // slice starts at a multiple of 8): 0 or a multiple of 8
  const int wv = max(0, min(p.w, p.R - col0));

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 4 + 1);  // the four gathering warps + the W_lat TMA
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(aux_full, 1);
    mbar_init(slice_full, 1);
    mbar_init(ls_full, 1);
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
  if (threadIdx.x == 0) XP_TRACE_MARK(1);
  pdl_launch_dependents();
  // copies requested, for the drain before exit after a timed-out wait
  int timed_out = 0, issued = 0;
  bool aux_issued = false, slices_issued = false, ls_issued = false;

  if (warp == 0) {
    // Nothing this warp reads is written by the preceding kernels, so it
    // starts before the dependency wait: the W_lat ring, then the hidden-cache
    // slice (one tensor box) and the mixer weights (one bulk copy per (b, j)
    // pair of the lower triangle: the slice's wv channels).  The copy engine
    // serves requests in order, so the epilogue's operands (needed only after
    // the MMAs) go after the first W_lat stages.  Lane 0 waits for a stage and
    // arms its barrier; lanes 0..tn/64-1 issue one W_lat box each (a single
    // thread issues tiled copies slowly).
    // two boxes: the hidden-cache slice and the mixer weights of the slice
    // (the whole [B][B] square of L for these w channels)
    auto aux_copies = [&]() {
      aux_issued = true;
      if (lane == 0) mbar_arrive_expect_tx(aux_full, (uint32_t)(p.B * p.B * p.lw * 4) + (uint32_t)(LT_BM * p.w * 2));
      __syncwarp();
      if (lane == 0) tma_load_2d(smem + p.hc_off, &mapHc, col0, mt * p.bpt * p.B, aux_full);
      if (lane == 1) tma_load_2d(Ls, &mapL, col0, 0, aux_full);
      __syncwarp();
    };
    const uint64_t pol = policy_evict_last();  // every pass re-reads W_lat
    if (lane == 0) {
      prefetch_tensormap(&mapWlat);
      prefetch_tensormap(&mapHc);
      prefetch_tensormap(&mapPart);
      prefetch_tensormap(&mapL);
    }
    for (int i = 0; i < nck; ++i) {
      if (i == 1) aux_copies();
      const uint32_t s = i % p.stages, k = i / p.stages;
      int ok = 1;
      if (lane == 0) {
        if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) ok = 0;
        else mbar_arrive_expect_tx(&full[s], b_bytes);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        timed_out = 1;
        if (lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
        break;
      }
      issued = i + 1;
      if (lane < p.tn / 64)
        tma_load_2d_hint(smem + (size_t)s * stage_bytes + LT_A_CHUNK + lane * LT_BOX, &mapWlat,
                         nt * p.tn + lane * 64, (c0 + i) * LT_BK, &full[s], pol);
    }
    if (nck <= 1 && !timed_out) aux_copies();
    if (lane == 0) XP_TRACE_MARK(3);
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(LT_BM, p.tn, 0, 1);
      bool dead = false;
      // stage 0's descriptors; a stage adds its offset and a K step of 16
      // adds 32 bytes to A and 16 rows (2 KB) to B (address field: 16-byte units)
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem) + LT_A_CHUNK, LT_BOX, 1024);
      uint32_t s = 0, ph = 0, soff = 0;
      for (int i = 0; i < nck; ++i) {
        if (!mbar_wait(&full[s], ph)) {
          dead = true;
          break;
        }
        tc_fence_after();
        if (i == 0) XP_TRACE_MARK(7);
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk)
          tc_mma_f16(tmem, adesc0 + soff + (uint64_t)(kk * 2), bdesc0 + soff + (uint64_t)(kk * 128), idesc, (i | kk) != 0);
        tc_commit(&empty[s]);
        if (++s == (uint32_t)p.stages) {
          s = 0;
          ph ^= 1;
          soff = 0;
        } else {
          soff += stage_bytes >> 4;
        }
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      timed_out = dead;
      tc_commit(acc_full);
      XP_TRACE_MARK(8);
    }
  } else {
    const int et = threadIdx.x - 64;  // 0..127
    pdl_wait();  // blk may have been written by the preceding pass
    if (et == 0) XP_TRACE_MARK(2);
    // token of every row of the tile (-1: no block there)
    {
      const int bl = et / p.B, b = et - bl * p.B, n = mt * p.bpt + bl;
      int64_t t = -1;
      if (bl < nbl) {
        t = (b == 0) ? p.am1[n] : p.blk[(int64_t)n * p.B + b - 1];
        if (t < 0 || t >= p.V) {
          flag_error(p.hdr, XP_DEVERR_TOKEN);
          t = t < 0 ? 0 : p.V - 1;
        }
      }
      tok[et] = t;
    }
    named_barrier_sync(1, 128);
    if (et == 0) XP_TRACE_MARK(4);
    // gather: every warp fills its 32 rows of every stage.  Eight lanes cover
    // one 128-byte row piece, so each copy instruction reads four whole
    // rows; a stage's copies form one cp.async group, and a warp hands a
    // stage over (wait for its group, proxy fence, arrive) only when it is
    // LAG = stages - 1 stages ahead, so the whole ring is in flight.
    const int gw = warp - 2, rsub = lane >> 3, piece = lane & 7;
    bool dead = false;
    auto hand_over = [&](int i) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[i % p.stages]);
      if (lane == 0 && i == 0) XP_TRACE_MARK(5);
      if (lane == 0 && i == nck - 1) XP_TRACE_MARK(6);
    };
    const int lag = p.stages - 1;  // 1..5
    for (int i = 0; i < nck; ++i) {
      const int s = i % p.stages, k = i / p.stages;
      if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) {
        dead = true;
        break;
      }
      uint8_t* dst = smem + (size_t)s * stage_bytes;
      const int kel = (c0 + i) * LT_BK + piece * 8;
      const bool kin = kel < p.D;  // D is a multiple of 8: a piece is wholly in or out
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int r = gw * 32 + it * 4 + rsub;
        const int64_t t = tok[r];
        const bool ok = kin && t >= 0;
        cp_async_16(dst + r * 128 + ((piece ^ (r & 7)) << 4), ok ? p.E + t * p.D + kel : p.E, ok ? 16u : 0u);
      }
      cp_async_commit();
      if (lane == 0 && gw == 0 && i == 0) XP_TRACE_MARK(26);
      if (i >= lag) {
        if (lane == 0 && gw == 0 && i == lag) XP_TRACE_MARK(27);
        cp_async_wait_group_n(lag);
        hand_over(i - lag);
      }
    }
    if (dead) {
      timed_out = 1;
      flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      cp_async_wait_all();
    } else {
      cp_async_wait_all();
      for (int i = max(0, nck - lag); i < nck; ++i) hand_over(i);
    }
  }

  // ---- epilogue 1: this CTA's fp32 partial tile TMEM -> shared memory (one
  // row per thread, 128-byte swizzle: conflict-free) -> TMA stores into the
  // partial buffer
  if (warp >= 2) {
    if (!mbar_wait(acc_full, 0)) {
      timed_out = 1;
      flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    }
    tc_fence_after();
    if (threadIdx.x == 64) XP_TRACE_MARK(9);
    const int q = warp & 3, row = q * 32 + lane;
    for (int c = 0; c < p.tn / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, r);
      tmem_ld_wait();
      uint8_t* box = pst + (size_t)c * (LT_BM * 128) + (size_t)row * 128;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        *reinterpret_cast<uint4*>(box + ((e ^ (row & 7)) << 4)) = make_uint4(r[4 * e], r[4 * e + 1], r[4 * e + 2], r[4 * e + 3]);
    }
    fence_proxy_async_smem();
    named_barrier_sync(1, 128);
    // one 32-column box per thread (a thread issues tiled copies ~0.27 us
    // apart), each waited for by the thread that issued it
    const int c = threadIdx.x - 64;
    if (c < p.tn / 32) {
      tma_store_2d(&mapPartSt, pst + (size_t)c * (LT_BM * 128), nt * p.tn + c * 32,
                   (int)((int64_t)ks * p.rows_pad + (int64_t)mt * LT_BM));
      bulk_commit();
      bulk_wait_all();  // this box of the partial tile is in global memory
      if (c == 0) XP_TRACE_MARK(10);
    }
  }
  tc_fence_before();
  __syncthreads();  // the partial tile of this CTA is stored
  if (warp == 0) {
    // publish this CTA's partial, wait for the other S-1, then fetch the S
    // partials of this CTA's w columns (one TMA box each, lanes in parallel)
    int ok = 1;
    if (lane == 0) {
      fence_proxy_async_global();
      (void)atom_add_acq_rel_gpu(&p.cnt[2 * tile], 1u);  // releases this CTA's stored partial
      const unsigned long long t0 = globaltimer();
      while (ld_acquire_gpu(&p.cnt[2 * tile]) < (uint32_t)p.S) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
      fence_proxy_async_global();
      if (ok) mbar_arrive_expect_tx(slice_full, (uint32_t)(p.S * p.prow * p.w * 4));
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
      timed_out = 1;
      if (lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    } else {
      slices_issued = true;
      if (lane < p.S)
        tma_load_2d(slices + (size_t)lane * LT_BM * p.w, &mapPart, col0,
                    (int)((int64_t)lane * p.rows_pad + (int64_t)mt * LT_BM), slice_full);
      // once the slices are here this CTA is done with the partial buffer:
      // the last of the S to get there resets the tile's counters
      if (lane == 0 && mbar_wait(slice_full, 0)) {
        if (atomicAdd(&p.cnt[2 * tile + 1], 1u) == (uint32_t)p.S - 1) {
          p.cnt[2 * tile] = 0u;
          p.cnt[2 * tile + 1] = 0u;
        }
      }
    }
    if (lane == 0) XP_TRACE_MARK(11);
  }

  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    if (!mbar_wait(slice_full, 0) || !mbar_wait(aux_full, 0)) {
      timed_out = 1;
      flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    }
    if (et == 127) XP_TRACE_MARK(28);
    // ---- epilogue 2: x = hcache + sum of the S partials (slice order) for
    // this CTA's columns of all rows, four columns per item
    // w is a power of two (a power-of-two split of 64 or 128 channels): the
    // item index splits by shifts, and the tile's rows that hold blocks are
    // the first nbl * B
    const int wq = p.w / 4, items = LT_BM * wq, wq_sh = __ffs(wq) - 1, live_rows = nbl * p.B;
    for (int it = et; it < items; it += 128) {
      const int rr = it >> wq_sh, gg = it & (wq - 1);
      if (rr >= live_rows) continue;
      float4 a = *reinterpret_cast<const float4*>(slices + rr * p.w + 4 * gg);
      for (int q = 1; q < p.S; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(slices + ((size_t)q * LT_BM + rr) * p.w + 4 * gg);
        a.x += v.x;
        a.y += v.y;
        a.z += v.z;
        a.w += v.w;
      }
      // the hidden cache of these 4 channels (zero past R: TMA fill)
      const uint2 hc = *reinterpret_cast<const uint2*>(hcs + rr * p.w + 4 * gg);
      float4 x;
      x.x = bf16lo_to_f32(hc.x) + a.x;
      x.y = bf16hi_to_f32(hc.x) + a.y;
      x.z = bf16lo_to_f32(hc.y) + a.z;
      x.w = bf16hi_to_f32(hc.y) + a.w;
      *reinterpret_cast<float4*>(xs + rr * p.w + 4 * gg) = x;
    }
    if (et == 127) XP_TRACE_MARK(12);
    named_barrier_sync(1, 128);
    // ---- the causal mixer on this CTA's columns: u[b] = sum_{j<=b} L[b,j] x[j],
    // into shared-memory tiles of the tile's rows (rows past N*B and columns
    // past R are clipped by the stores)
    float* us = reinterpret_cast<float*>(pst);                            // [bpt*B][w]
    uint16_t* ubs = reinterpret_cast<uint16_t*>(pst + (size_t)LT_BM * p.w * 4);  // [bpt*B][w]
    // the mixer on columns [cb, cb + lw) with Ls holding their weights
    auto mix = [&](const int cb, const int lw) {
      if (nbl * lw <= 16) {
        // very few (block, channel) pairs (one block, a narrow slice): one
        // output per thread, the same sum in the same order as below
        for (int it = et; it < nbl * p.B * lw; it += 128) {
          const int bb = it / lw, cl = it - bb * lw;  // bb = bl * B + b
          const int bl = bb / p.B, b = bb - bl * p.B, c = cb + cl;
          const float* Lb = Ls + (b * p.B) * lw + cl;
          const float* xc = xs + (bl * p.B) * p.w + c;
          float uu = 0.f;
          for (int j = 0; j <= b; ++j) uu = fmaf(Lb[j * lw], xc[j * p.w], uu);
          const int o = bb * p.w + c;
          us[o] = uu;
          ubs[o] = (uint16_t)(f32x2_to_bf16x2(uu, 0.f) & 0xffffu);
        }
      } else {
        const int lw_sh = __ffs(lw) - 1;  // lw is a power of two
        for (int it = et; it < nbl * lw; it += 128) {
          const int bl = it >> lw_sh, cl = it & (lw - 1), c = cb + cl;
          float x[LT_MAX_B];
#pragma unroll
          for (int j = 0; j < LT_MAX_B; ++j) x[j] = j < p.B ? xs[(bl * p.B + j) * p.w + c] : 0.f;
#pragma unroll
          for (int b = 0; b < LT_MAX_B; ++b) {
            if (b < p.B) {
              float uu = 0.f;
              const float* Lb = Ls + (b * p.B) * lw + cl;
#pragma unroll
              for (int j = 0; j <= b; ++j) uu = fmaf(Lb[j * lw], x[j], uu);
              const int o = (bl * p.B + b) * p.w + c;
              us[o] = uu;
              ubs[o] = (uint16_t)(f32x2_to_bf16x2(uu, 0.f) & 0xffffu);
            }
          }
        }
      }
    };
    if constexpr (!kHalfL) {
      mix(0, p.w);
    } else {
      // Ls holds the weights of half the columns: the second half's are
      // copied in once every thread is done with the first's
      mix(0, p.lw);
      named_barrier_sync(1, 128);
      if (et == 0) {
        mbar_arrive_expect_tx(ls_full, (uint32_t)(p.B * p.B * p.lw * 4));
        tma_load_2d(Ls, &mapL, col0 + p.lw, 0, ls_full);
        ls_issued = true;
      }
      if (!timed_out && !mbar_wait(ls_full, 0)) {
        timed_out = 1;
        flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      }
      mix(p.lw, p.lw);
    }
    if (et == 127) XP_TRACE_MARK(29);
    fence_proxy_async_smem();
    named_barrier_sync(1, 128);
    if (et < 2) {  // u and bf16(u), one thread each
      if (et == 0) XP_TRACE_MARK(30);
      if (et == 0) tma_store_2d(&mapU, us, col0, mt * p.bpt * p.B);
      else tma_store_2d(&mapUb, ubs, col0, mt * p.bpt * p.B);
      bulk_commit();
      bulk_wait_all();
      if (et == 0) XP_TRACE_MARK(13);
    }
  }
  tc_fence_before();
  // After a timed-out wait, warp 0 waits (bounded) for every copy it may
  // still have in flight into this CTA's shared memory before the CTA exits
  // (earlier phases of a ring slot are complete: a slot is re-armed only
  // after its previous phase was consumed)
  if (__syncthreads_or(timed_out) && threadIdx.x == 0) {
    for (int j = issued > p.stages ? issued - p.stages : 0; j < issued; ++j)
      (void)mbar_wait(&full[j % p.stages], (uint32_t)(j / p.stages) & 1);
    if (aux_issued) (void)mbar_wait(aux_full, 0);
    if (slices_issued) (void)mbar_wait(slice_full, 0);
  }
  if constexpr (kHalfL) {
    if (threadIdx.x == 64 && ls_issued) (void)mbar_wait(ls_full, 0);  // landed before exit (done on the normal path)
  }
  __syncthreads();
  if (threadIdx.x == 0) XP_TRACE_MARK(14);
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
  int32_t arow;  // rows per ub box: 128, or a lone M tile's rows rounded up to 8
  const uint32_t* skip;  // nullable: see pass_skipped
};

// kGemm: the GEMM schedule (g and v rounded to bf16 before the SiLU, as the
// bf16 u @ wgu_t returns them); else the in-kernel MLP (fp32 g and v)
template <bool kGemm>
__global__ void __launch_bounds__(LT_UP_THREADS, 2)
mlp_up_kernel(const __grid_constant__ CUtensorMap mapUb, const __grid_constant__ CUtensorMap mapWg,
              const __grid_constant__ CUtensorMap mapWu, const UpParams p) {
  extern __shared__ uint8_t smem_raw[];
  if (pass_skipped(p.skip, false)) return;
  if (threadIdx.x == 0) XP_TRACE_MARK(16);
  uint8_t* smem = align1024(smem_raw);
  constexpr uint32_t stage_bytes = LT_A_CHUNK + 2 * LT_BOX;  // 32 KB
  const uint32_t stage_tx = (uint32_t)p.arow * 128u + 2 * LT_BOX;  // bytes a stage's copies bring
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
  if (threadIdx.x == 0) XP_TRACE_MARK(17);
  pdl_launch_dependents();
  int timed_out = 0, issued = 0;  // for the drain before exit after a timed-out wait

  if (warp == 0) {
    // lane 0 arms the stage; lanes 0, 1, 2 issue the ub, Wg and Wu boxes.
    // The weights of the first stages are requested before the dependency
    // wait (nothing earlier in the pass writes them); ub comes from proj_mix.
    if (lane == 0) {
      prefetch_tensormap(&mapUb);
      prefetch_tensormap(&mapWg);
      prefetch_tensormap(&mapWu);
    }
    const uint64_t pol = policy_evict_last();  // every pass re-reads Wg, Wu
    const int pre = p.chunks < p.stages ? p.chunks : p.stages;
    issued = pre;
    // the first stages armed, then their Wg and Wu boxes one lane each (a
    // thread issues tiled copies one after another, ~0.27 us apiece, so one
    // lane per box keeps this ahead of the dependency wait short)
    if (lane == 0)
      for (int i = 0; i < pre; ++i) mbar_arrive_expect_tx(&full[i], stage_tx);
    __syncwarp();
    if (lane < 2 * pre) {
      const int i = lane >> 1;
      uint8_t* dst = smem + (size_t)i * stage_bytes + LT_A_CHUNK + (lane & 1) * LT_BOX;
      tma_load_2d_hint(dst, (lane & 1) ? &mapWu : &mapWg, ht * 64, i * LT_BK, &full[i], pol);
    }
    pdl_wait();
    if (lane == 0) XP_TRACE_MARK(18);
    // the first stages' ub boxes, one lane each (a single thread issues
    // tiled copies one after another, ~0.27 us apiece)
    if (lane < pre) tma_load_2d(smem + (size_t)lane * stage_bytes, &mapUb, lane * LT_BK, mt * LT_BM, &full[lane]);
    for (int i = pre; i < p.chunks; ++i) {
      const uint32_t s = i % p.stages, k = i / p.stages;
      int ok = 1;
      if (lane == 0) {
        if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) ok = 0;
        else mbar_arrive_expect_tx(&full[s], stage_tx);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        timed_out = 1;
        if (lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
        break;
      }
      issued = i + 1;
      uint8_t* dst = smem + (size_t)s * stage_bytes;
      if (lane == 0) tma_load_2d(dst, &mapUb, i * LT_BK, mt * LT_BM, &full[s]);
      if (lane == 1) tma_load_2d_hint(dst + LT_A_CHUNK, &mapWg, ht * 64, i * LT_BK, &full[s], pol);
      if (lane == 2) tma_load_2d_hint(dst + LT_A_CHUNK + LT_BOX, &mapWu, ht * 64, i * LT_BK, &full[s], pol);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // one N=128 MMA per K step computes [g | v]: the stage's Wg and Wu
      // boxes sit one box apart, which is the B descriptor's stride between
      // its two 64-wide N chunks, and TMEM columns [0, 64) / [64, 128) take
      // g / v (an N=64 MMA runs at ~64 % of the N=128 rate)
      constexpr uint32_t idesc = idesc_bf16_f32(LT_BM, 128, 0, 1);
      bool dead = false;
      // stage 0's descriptors; a stage adds its offset and a K step of 16
      // adds 32 bytes to A and 16 rows (2 KB) to B (address field: 16-byte units)
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t gvdesc0 = smem_desc_sw128(smem_u32(smem) + LT_A_CHUNK, LT_BOX, 1024);
      uint32_t s = 0, ph = 0, soff = 0;
      for (int i = 0; i < p.chunks; ++i) {
        if (!mbar_wait(&full[s], ph)) {
          dead = true;
          break;
        }
        tc_fence_after();
        if (i == 0) XP_TRACE_MARK(19);
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk)
          tc_mma_f16(tmem, adesc0 + soff + (uint64_t)(kk * 2), gvdesc0 + soff + (uint64_t)(kk * 128), idesc, (i | kk) != 0);
        tc_commit(&empty[s]);
        if (++s == (uint32_t)p.stages) {
          s = 0;
          ph ^= 1;
          soff = 0;
        } else {
          soff += stage_bytes >> 4;
        }
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      timed_out = dead;
      tc_commit(acc_full);
      XP_TRACE_MARK(20);
    }
  } else {
    pdl_wait();
    if (!mbar_wait(acc_full, 0)) {
      timed_out = 1;
      flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    }
    tc_fence_after();
    if (threadIdx.x == 64) XP_TRACE_MARK(21);
    // two warps per TMEM lane quadrant, one 32-column half of g and v each
    const int q = warp & 3;
    const int row = mt * LT_BM + q * 32 + lane;
    {
      const int c = (warp - 2) >> 2;
      uint32_t g[32], v[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, g);
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + 64 + c * 32, v);
      tmem_ld_wait();
      if (row < p.rows) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float g0 = __uint_as_float(g[2 * e]), g1 = __uint_as_float(g[2 * e + 1]);
          float v0 = __uint_as_float(v[2 * e]), v1 = __uint_as_float(v[2 * e + 1]);
          if (kGemm) {
            // the GEMM schedule's u @ wgu_t returns bf16: round g and v first
            const uint32_t gq = f32x2_to_bf16x2(g0, g1), vq = f32x2_to_bf16x2(v0, v1);
            g0 = bf16lo_to_f32(gq);
            g1 = bf16hi_to_f32(gq);
            v0 = bf16lo_to_f32(vq);
            v1 = bf16hi_to_f32(vq);
          }
          const float m0 = __fdividef(g0, 1.f + __expf(-g0)) * v0;
          const float m1 = __fdividef(g1, 1.f + __expf(-g1)) * v1;
          w[e] = f32x2_to_bf16x2(m0, m1);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.m + (int64_t)row * p.H + ht * 64 + c * 32);
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    }
    if (threadIdx.x == 64) XP_TRACE_MARK(22);
  }
  tc_fence_before();
  // after a timed-out wait: the ring's copies still in flight land before exit
  if (__syncthreads_or(timed_out) && threadIdx.x == 0)
    for (int j = issued > p.stages ? issued - p.stages : 0; j < issued; ++j)
      (void)mbar_wait(&full[j % p.stages], (uint32_t)(j / p.stages) & 1);
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// ============================================================================
// mlp_down: lat = bf16(u + m @ Wd) for slots 1..B-1
// ============================================================================
// Shared memory: [0, region) is the stage ring, then red[128][tn + 4] (this
// CTA's fp32 partial sums, read by the whole cluster) reusing it; us (the
// residual u of this CTA's w columns for the tile's 128 rows, copied by TMA
// while the MMAs run); the barriers.
struct DownParams {
  uint16_t* lat;
  WsHeader* hdr;
  int32_t N, B, R, tn, S, w, chunks, ntiles, stages;
  int32_t arow;  // rows per m / residual box: 128, or a lone M tile's rows rounded up to 8
  uint32_t region, bar_off;
  const uint32_t* skip;  // nullable: see pass_skipped
};

// kGemm: the GEMM schedule (the residual is bf16(u): addmm_ into the bf16 u);
// else the in-kernel MLP (the fp32 residual u)
template <bool kGemm>
__global__ void __launch_bounds__(LT_THREADS, 2)
mlp_down_kernel(const __grid_constant__ CUtensorMap mapM, const __grid_constant__ CUtensorMap mapWd,
                const __grid_constant__ CUtensorMap mapU, const DownParams p) {
  extern __shared__ uint8_t smem_raw[];
  if (pass_skipped(p.skip, false)) return;
  if (threadIdx.x == 0) XP_TRACE_MARK(32);
  uint8_t* smem = align1024(smem_raw);
  const uint32_t b_bytes = (uint32_t)p.tn * LT_BK * 2;
  const uint32_t stage_bytes = LT_A_CHUNK + b_bytes;
  const uint32_t stage_tx = (uint32_t)p.arow * 128u + b_bytes;  // bytes a stage's copies bring
  const int ld = p.tn + 4;  // floats per row of red (a 16-byte multiple)
  const float* us = reinterpret_cast<const float*>(smem + p.region);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint64_t* aux_full = acc_full + 1;  // us landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aux_full + 1);
  float* red = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = (int)(blockIdx.x % p.S);
  const int nt = (int)((blockIdx.x / p.S) % p.ntiles);
  const int mt = (int)(blockIdx.x / (p.S * p.ntiles));
  const int c0 = (int)((int64_t)ks * p.chunks / p.S);
  const int nck = (int)((int64_t)(ks + 1) * p.chunks / p.S) - c0;
  const int rows = p.N * p.B;
  const int c_lo = ks * p.w;          // this CTA's columns of the tile: [c_lo, c_lo + w)
  const int col0 = nt * p.tn + c_lo;  // ... as latent channels

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(aux_full, 1);
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
  if (threadIdx.x == 0) XP_TRACE_MARK(33);
  pdl_launch_dependents();
  int timed_out = 0, issued = 0;  // for the drain before exit after a timed-out wait

  if (warp == 0) {
    // lane 0 arms the stage; lane 0 issues the m box, lanes 1.. the Wd boxes.
    // The Wd boxes of the first stages are requested before the dependency
    // wait (nothing earlier in the pass writes Wd); m comes from mlp_up and
    // the residual u (one box of this CTA's columns) from proj_mix.
    if (lane == 0) {
      prefetch_tensormap(&mapM);
      prefetch_tensormap(&mapWd);
      prefetch_tensormap(&mapU);
    }
    const uint64_t pol = policy_evict_last();  // every pass re-reads Wd
    const int pre = nck < p.stages ? nck : p.stages;
    issued = pre;
    // the first stages armed, then their Wd boxes one lane each (see mlp_up)
    if (lane == 0)
      for (int i = 0; i < pre; ++i) mbar_arrive_expect_tx(&full[i], stage_tx);
    __syncwarp();
    const int bpb = p.tn / 64;  // Wd boxes per stage
    if (lane < pre * bpb) {
      const int i = lane / bpb, bx = lane - i * bpb;
      tma_load_2d_hint(smem + (size_t)i * stage_bytes + LT_A_CHUNK + bx * LT_BOX, &mapWd, nt * p.tn + bx * 64,
                       (c0 + i) * LT_BK, &full[i], pol);
    }
    pdl_wait();
    if (lane == 0) XP_TRACE_MARK(34);
    // the first stages' m boxes and the residual box, one lane each (a single
    // thread issues tiled copies one after another, ~0.27 us apiece)
    if (lane < pre)
      tma_load_2d(smem + (size_t)lane * stage_bytes, &mapM, (c0 + lane) * LT_BK, mt * LT_BM, &full[lane]);
    if (lane == 31) {
      mbar_arrive_expect_tx(aux_full, (uint32_t)(p.arow * p.w * 4));
      tma_load_2d(smem + p.region, &mapU, col0, mt * LT_BM, aux_full);
    }
    for (int i = pre; i < nck; ++i) {
      const uint32_t s = i % p.stages, k = i / p.stages;
      int ok = 1;
      if (lane == 0) {
        if (k >= 1 && !mbar_wait(&empty[s], (k - 1) & 1)) ok = 0;
        else mbar_arrive_expect_tx(&full[s], stage_tx);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        timed_out = 1;
        if (lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
        break;
      }
      issued = i + 1;
      uint8_t* dst = smem + (size_t)s * stage_bytes;
      if (lane == 0) tma_load_2d(dst, &mapM, (c0 + i) * LT_BK, mt * LT_BM, &full[s]);
      if (lane >= 1 && lane <= p.tn / 64)
        tma_load_2d_hint(dst + LT_A_CHUNK + (lane - 1) * LT_BOX, &mapWd, nt * p.tn + (lane - 1) * 64, (c0 + i) * LT_BK,
                         &full[s], pol);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(LT_BM, p.tn, 0, 1);
      bool dead = false;
      // stage 0's descriptors; a stage adds its offset and a K step of 16
      // adds 32 bytes to A and 16 rows (2 KB) to B (address field: 16-byte units)
      const uint64_t adesc0 = smem_desc_sw128(smem_u32(smem), 16, 1024);
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem) + LT_A_CHUNK, LT_BOX, 1024);
      uint32_t s = 0, ph = 0, soff = 0;
      for (int i = 0; i < nck; ++i) {
        if (!mbar_wait(&full[s], ph)) {
          dead = true;
          break;
        }
        tc_fence_after();
        if (i == 0) XP_TRACE_MARK(32 + 7);
#pragma unroll
        for (int kk = 0; kk < LT_BK / 16; ++kk)
          tc_mma_f16(tmem, adesc0 + soff + (uint64_t)(kk * 2), bdesc0 + soff + (uint64_t)(kk * 128), idesc, (i | kk) != 0);
        tc_commit(&empty[s]);
        if (++s == (uint32_t)p.stages) {
          s = 0;
          ph ^= 1;
          soff = 0;
        } else {
          soff += stage_bytes >> 4;
        }
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      timed_out = dead;
      tc_commit(acc_full);
      XP_TRACE_MARK(32 + 8);
    }
  } else {
    pdl_wait();
    if (!mbar_wait(acc_full, 0)) {
      timed_out = 1;
      flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    }
    tc_fence_after();
    if (threadIdx.x == 64) XP_TRACE_MARK(41);
    const int q = warp & 3, row = q * 32 + lane;
    for (int c = 0; c < p.tn / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, r);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(red + row * ld + c * 32);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]), __uint_as_float(r[4 * e + 2]),
                             __uint_as_float(r[4 * e + 3]));
    }
  }
  if (threadIdx.x == 64) XP_TRACE_MARK(42);
  tc_fence_before();
  cluster_sync();
  if (threadIdx.x == 64) XP_TRACE_MARK(43);

  // ---- sum the cluster's partials for this CTA's columns (fixed order), add
  // the residual u, write slots 1..B-1.  Two (row, 4 columns) items per
  // thread per round; the residual and every partial are requested first.
  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    const int wq = p.w / 4, items = LT_BM * wq;
    if (!mbar_wait(aux_full, 0)) {
      timed_out = 1;
      flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    }
    for (int i0 = et; i0 < items; i0 += 256) {
      float4 v[2][LT_MAX_S], uu[2];
      int64_t dst[2];
      bool on[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int it = i0 + h * 128;
        const int rr = it / wq, gg = it - rr * wq;
        const int grow = mt * LT_BM + rr;
        const int n = grow / p.B, b = grow - n * p.B;
        const int col = col0 + 4 * gg;
        on[h] = it < items && grow < rows && b >= 1 && col < p.R;
        dst[h] = ((int64_t)n * (p.B - 1) + b - 1) * p.R + col;
        uu[h] = on[h] ? *reinterpret_cast<const float4*>(us + rr * p.w + 4 * gg) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (kGemm) {
          const uint32_t lo = f32x2_to_bf16x2(uu[h].x, uu[h].y), hi = f32x2_to_bf16x2(uu[h].z, uu[h].w);
          uu[h] = make_float4(bf16lo_to_f32(lo), bf16hi_to_f32(lo), bf16lo_to_f32(hi), bf16hi_to_f32(hi));
        }
#pragma unroll
        for (int q = 0; q < LT_MAX_S; ++q)
          v[h][q] = (on[h] && q < p.S) ? ld_dsmem_v4(red + rr * ld + c_lo + 4 * gg, (uint32_t)q)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!on[h]) continue;
        float4 a = v[h][0];
#pragma unroll
        for (int q = 1; q < LT_MAX_S; ++q) {
          if (q < p.S) {
            a.x += v[h][q].x;
            a.y += v[h][q].y;
            a.z += v[h][q].z;
            a.w += v[h][q].w;
          }
        }
        *reinterpret_cast<uint2*>(p.lat + dst[h]) =
            make_uint2(f32x2_to_bf16x2(uu[h].x + a.x, uu[h].y + a.y), f32x2_to_bf16x2(uu[h].z + a.z, uu[h].w + a.w));
      }
    }
    if (et == 127) XP_TRACE_MARK(44);
  }
  // after a timed-out wait: the copies still in flight land before exit (the
  // residual box is always requested)
  if (__syncthreads_or(timed_out) && threadIdx.x == 0) {
    for (int j = issued > p.stages ? issued - p.stages : 0; j < issued; ++j)
      (void)mbar_wait(&full[j % p.stages], (uint32_t)(j / p.stages) & 1);
    (void)mbar_wait(aux_full, 0);
  }
  __syncwarp();
  cluster_sync_relaxed();  // the peers have finished reading this CTA's partial sums
  if (threadIdx.x == 0) XP_TRACE_MARK(45);
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
int g_lt_sms[64];  // multiprocessors of each device (read with the attributes)

cudaError_t launch_ex(const void* kernel_fn, dim3 grid, size_t smem, cudaStream_t stream, int cluster, void** args,
                      int threads = LT_THREADS) {
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
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  return cudaLaunchKernelExC(&cfg, kernel_fn, args);
}

// Largest power of two <= min(cap, x) (x >= 1): the cluster size of a split
// reduction, so every CTA's column slice of a tile is a multiple of 4 wide.
int pow2_floor(int x, int cap) {
  int s = 1;
  while (s * 2 <= x && s * 2 <= cap) s *= 2;
  return s;
}


}  // namespace

xp_status launch_latent(const int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
                        const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
                        const uint16_t* Wd, uint16_t* lat_out, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R,
                        int64_t H, void* ws, cudaStream_t stream, const uint32_t* skip, bool do_mlp) {
  if (N <= 0) return XP_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return XP_ERR_LAUNCH;
  if (!g_lt_attr[dev]) {
    int max_smem = 0;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&g_lt_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return XP_ERR_LAUNCH;
    // the largest dynamic shared memory each kernel may ask for (the opt-in
    // maximum less its static shared memory) and the largest carve-out
    auto allow = [&](const void* fn) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return false;
      return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  max_smem - (int)fa.sharedSizeBytes) == cudaSuccess &&
             cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
    };
    if (!allow((const void*)proj_mix_kernel<false>) || !allow((const void*)proj_mix_kernel<true>) ||
        !allow((const void*)mlp_up_kernel<false>) ||
        !allow((const void*)mlp_up_kernel<true>) || !allow((const void*)mlp_down_kernel<false>) ||
        !allow((const void*)mlp_down_kernel<true>))
      return XP_ERR_LAUNCH;
    g_lt_attr[dev] = true;
  }
  const LatentWsLayout lay = latent_ws_layout(N, B, D, R, H);
  char* w = static_cast<char*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  float* u = reinterpret_cast<float*>(w + lay.u);
  uint16_t* ub = reinterpret_cast<uint16_t*>(w + lay.ub);
  uint16_t* m = reinterpret_cast<uint16_t*>(w + lay.m);
  const int rows = (int)(N * B);

  // ---- proj_mix
  {
    const ProjTiling t = proj_tiling(N, B, D, R);
    ProjParams p;
    p.skip = skip;
    p.blk = blk;
    p.am1 = am1;
    p.E = E;
    p.L = L;
    p.u = u;
    p.ub = ub;
    p.part = reinterpret_cast<float*>(w + lay.part);
    p.cnt = reinterpret_cast<uint32_t*>(w + lay.cnt);
    p.hdr = hdr;
    p.N = (int32_t)N;
    p.B = (int32_t)B;
    p.V = (int32_t)V;
    p.D = (int32_t)D;
    p.R = (int32_t)R;
    p.bpt = t.bpt;
    p.tn = t.tn;
    p.chunks = t.chunks;
    p.S = t.S;
    p.w = t.w;
    p.lw = t.lw;
    p.ntiles = t.ntiles;
    p.rows_pad = t.rows_pad;
    p.r_pad = t.r_pad;
    // a lone M tile stores and sums only the rows that hold blocks
    p.prow = t.mtiles == 1 ? (int32_t)(((N * B + 7) / 8) * 8 < LT_BM ? ((N * B + 7) / 8) * 8 : LT_BM) : LT_BM;
    // the gathering warps keep stages - 1 stages in flight; as deep a ring as
    // fits (at least 2 stages)
    const int per_cta = (t.chunks + t.S - 1) / t.S;
    int st = per_cta < 6 ? (per_cta < 2 ? 2 : per_cta) : 6;
    while (st > 2 && proj_smem(t, B, st).total > kLatentSmemBudget) --st;
    const ProjSmem lay_s = proj_smem(t, B, st);
    if (lay_s.total > kLatentSmemBudget) return XP_ERR_UNSUPPORTED;  // the tiling keeps every supported shape within it
    p.stages = st;
    p.region = lay_s.region;
    p.hc_off = lay_s.hc_off;
    p.tok_off = lay_s.tok_off;
    p.bar_off = lay_s.bar_off;
    const size_t smem = lay_s.total;
    CUtensorMap mapWlat, mapHc, mapPart, mapPartSt, mapL, mapU, mapUbS;
    if (!cached_map_bf16_2d(&mapWlat, W_lat, (uint64_t)R, (uint64_t)D, (uint64_t)R, 64, LT_BK) ||
        !cached_map_plain_2d(&mapHc, hcache, 2, (uint64_t)R, (uint64_t)(N * B), (uint64_t)R, (uint32_t)t.w, LT_BM) ||
        !cached_map_plain_2d(&mapPart, p.part, 4, (uint64_t)t.r_pad, (uint64_t)(t.S * t.rows_pad), (uint64_t)t.r_pad,
                             (uint32_t)t.w, (uint32_t)p.prow) ||
        !cached_map_plain_2d(&mapPartSt, p.part, 4, (uint64_t)t.r_pad, (uint64_t)(t.S * t.rows_pad),
                             (uint64_t)t.r_pad, 32, (uint32_t)p.prow, true) ||
        !cached_map_plain_2d(&mapL, L, 4, (uint64_t)R, (uint64_t)(B * B), (uint64_t)R, (uint32_t)t.lw,
                             (uint32_t)(B * B)) ||
        !cached_map_plain_2d(&mapU, u, 4, (uint64_t)R, (uint64_t)(N * B), (uint64_t)R, (uint32_t)t.w,
                             (uint32_t)(t.bpt * B)) ||
        !cached_map_plain_2d(&mapUbS, ub, 2, (uint64_t)R, (uint64_t)(N * B), (uint64_t)R, (uint32_t)t.w,
                             (uint32_t)(t.bpt * B)))
      return XP_ERR_LAUNCH;
    void* args[] = {&mapWlat, &mapHc, &mapPart, &mapPartSt, &mapL, &mapU, &mapUbS, &p};
    const void* pm_fn = t.lw == t.w ? (const void*)proj_mix_kernel<false> : (const void*)proj_mix_kernel<true>;
    if (launch_ex(pm_fn, dim3((unsigned)(t.mtiles * t.ntiles * t.S)), smem, stream, 1, args) !=
        cudaSuccess) {
      (void)cudaGetLastError();  // a failed launch must not be reported again by a later call
      return XP_ERR_LAUNCH;
    }
  }
  // ---- mlp_up
  {
    UpParams p;
    p.skip = skip;
    p.m = m;
    p.hdr = hdr;
    p.rows = rows;
    p.H = (int32_t)H;
    p.chunks = (int32_t)((R + LT_BK - 1) / LT_BK);
    p.htiles = (int32_t)(H / 64);
    const int mtiles = (rows + LT_BM - 1) / LT_BM;
    p.arow = rows < LT_BM ? (rows + 7) / 8 * 8 : LT_BM;  // a lone partial M tile copies only its rows
    p.stages = p.chunks < 6 ? (p.chunks < 2 ? 2 : p.chunks) : 6;
    // more CTAs than SMs: a three-stage ring, so two CTAs fit on an SM and
    // the grid runs in one wave
    if ((int64_t)mtiles * p.htiles > g_lt_sms[dev] && p.stages > 3) p.stages = 3;
    const size_t smem = 1024 + (size_t)p.stages * (LT_A_CHUNK + 2 * LT_BOX) + 8 * (2 * p.stages + 1) + 16;
    CUtensorMap mapUb, mapWg, mapWu;
    if (!cached_map_bf16_2d(&mapUb, ub, (uint64_t)R, (uint64_t)rows, (uint64_t)R, LT_BK, (uint32_t)p.arow) ||
        !cached_map_bf16_2d(&mapWg, Wg, (uint64_t)H, (uint64_t)R, (uint64_t)H, 64, LT_BK) ||
        !cached_map_bf16_2d(&mapWu, Wu, (uint64_t)H, (uint64_t)R, (uint64_t)H, 64, LT_BK))
      return XP_ERR_LAUNCH;
    void* args[] = {&mapUb, &mapWg, &mapWu, &p};
    const void* up_fn = do_mlp ? (const void*)mlp_up_kernel<false> : (const void*)mlp_up_kernel<true>;
    if (launch_ex(up_fn, dim3((unsigned)(mtiles * p.htiles)), smem, stream, 1, args, LT_UP_THREADS) != cudaSuccess) {
      (void)cudaGetLastError();
      return XP_ERR_LAUNCH;
    }
  }
  // ---- mlp_down
  {
    DownParams p;
    p.skip = skip;
    p.lat = lat_out;
    p.hdr = hdr;
    p.N = (int32_t)N;
    p.B = (int32_t)B;
    p.R = (int32_t)R;
    // 64-channel tiles and a 4-way H split: half the cluster reduction
    // (distributed shared memory is the slow part here) for 1.5x the operand
    // bytes per CTA; one CTA per SM (clusters of 4 always fit the GPCs)
    const int dtn = 64;
    p.tn = dtn;
    p.chunks = (int32_t)(H / LT_BK);
    p.S = pow2_floor(p.chunks, 4);
    p.w = dtn / p.S;
    p.ntiles = (int32_t)((R + dtn - 1) / dtn);
    const uint32_t stage_bytes = LT_A_CHUNK + (uint32_t)dtn * LT_BK * 2;
    const size_t red_bytes = (size_t)LT_BM * (dtn + 4) * 4;
    auto region_of = [&](int st) {
      const size_t ring = (size_t)st * stage_bytes;
      return (ring > red_bytes ? ring : red_bytes + 1023) & ~size_t(1023);
    };
    const size_t us_bytes = (size_t)LT_BM * p.w * 4;
    // us, then full/empty per stage, acc_full, aux_full and the TMEM slot
    auto total = [&](int st) { return 1024 + region_of(st) + us_bytes + 8 * (2 * st + 2) + 16; };
    const int per_cta = (p.chunks + p.S - 1) / p.S;
    const int mtiles = (rows + LT_BM - 1) / LT_BM;
    p.arow = rows < LT_BM ? (rows + 7) / 8 * 8 : LT_BM;  // a lone partial M tile copies only its rows
    p.stages = per_cta < 6 ? (per_cta < 2 ? 2 : per_cta) : 6;
    // more CTAs than SMs: a four-stage ring, so two CTAs fit on an SM and the
    // grid runs in one wave
    if ((int64_t)mtiles * p.ntiles * p.S > g_lt_sms[dev] && p.stages > 4) p.stages = 4;
    p.region = (uint32_t)region_of(p.stages);
    p.bar_off = p.region + (uint32_t)us_bytes;
    const size_t smem = total(p.stages);
    CUtensorMap mapM, mapWd, mapU;
    if (!cached_map_bf16_2d(&mapM, m, (uint64_t)H, (uint64_t)rows, (uint64_t)H, LT_BK, (uint32_t)p.arow) ||
        !cached_map_bf16_2d(&mapWd, Wd, (uint64_t)R, (uint64_t)H, (uint64_t)R, 64, LT_BK) ||
        !cached_map_plain_2d(&mapU, u, 4, (uint64_t)R, (uint64_t)rows, (uint64_t)R, (uint32_t)p.w, (uint32_t)p.arow))
      return XP_ERR_LAUNCH;
    void* args[] = {&mapM, &mapWd, &mapU, &p};
    const void* down_fn = do_mlp ? (const void*)mlp_down_kernel<false> : (const void*)mlp_down_kernel<true>;
    if (launch_ex(down_fn, dim3((unsigned)(mtiles * p.ntiles * p.S)), smem, stream, p.S, args) != cudaSuccess) {
      (void)cudaGetLastError();
      return XP_ERR_LAUNCH;
    }
  }
  return XP_OK;
}

}  // namespace xp

XP_TRACE_READER(xp_trace_read_latent)
