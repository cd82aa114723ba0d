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
// GB300 design (tcgen05 + TMEM + TMA, CTA pairs):
//   * W2 is read vocabulary-major (W2t = W2 transposed, [V, R]), so the
//     weights of a vocab tile are one contiguous block of memory rather than
//     128-byte pieces of distant rows;
//   * CTAs work in pairs (a 2-CTA cluster): the pair owns two M tiles of 128
//     draft rows (one per CTA) and a contiguous range of 128-wide vocab tiles.
//     The leader issues tcgen05.mma.cta_group::2 with M = 256, N = 128: each
//     CTA holds its own 128 rows of the latent (the A operand) in tensor
//     memory and streams only ITS 64-vocab half of every W2 tile, yet
//     receives the full 128 x 128 accumulator for its rows.  Every W2 byte an
//     SM ingests thus serves 256 rows instead of 128, which halves the
//     per-SM W2 traffic, the limit of this stream;
//   * each CTA's 128 x R latent slice is staged ONCE into tensor memory (256
//     columns for R = 512): one round of TMA brings it into the (still empty)
//     base ring and second W2 slot, and the epilogue warps copy their rows
//     into TMEM lanes (the second slot's first W2 tile is requested after);
//   * the W2t half-tiles (64 vocab x R, up to eight 8 KB TMA boxes, one lane
//     each) go into two tile slots, refilled by two producer warps (0 and 10,
//     one slot each); the copies of both CTAs complete on the leader's
//     barrier, so one wait covers both halves; warp 11 streams the CTA's
//     128 x 128 base tiles into a 3-deep ring (128-byte swizzle throughout);
//   * the leader's warp 1 issues the MMAs of tile t into accumulator t % 2
//     (two 128-column TMEM accumulators: the epilogue of tile t overlaps the
//     MMAs of tile t+1) and commits them ONCE per tile to the barriers of
//     both CTAs: that commit both hands the accumulator to the epilogue and
//     frees the W2 slot of tile t for tile t+2 (each CTA's W2 half-tile is
//     one contiguous 64 KB block of W2t; loading and releasing it in K parts
//     was slower);
//   * warps 2..9 drain the accumulator with tcgen05.ld (thread = one row,
//     warp = a 32-lane quadrant and a 64-column half), round to bf16, add the
//     base tile from shared memory and keep a running (max, first column)
//     per row across the CTA's tiles (tiles and columns ascend, so a strict
//     '>' keeps the lowest index); both CTAs' epilogues release an
//     accumulator on the leader's barrier;
//   * each row's per-CTA winner is folded into a 64-bit (value, lowest
//     index) key with atomicMax and counted on the row's arrival counter; the
//     arrival that completes a row writes its blk slot, counts a change and
//     re-zeroes the key, so no CTA waits for the others at the end.
#include "xp_common.cuh"
#include "xp_internal.h"
#include "xp_ptx.cuh"
#include "xp_tma.cuh"
#include "xp_trace.cuh"

namespace xp {

constexpr int RO_BM = 128;                             // draft rows per CTA (M per CTA)
constexpr int RO_BN = 128;                             // vocab per tile (N of the pair's MMA)
constexpr int RO_HALF = RO_BN / 2;                     // vocab rows of W2t a CTA streams per tile
constexpr int RO_EPI_WARPS = 8;
// warp 0: W2 producer (even stages); warp 1: MMA issuer (leader); warps 2..9:
// epilogue; warp 10: W2 producer (odd stages); warp 11: latent + base producer.
constexpr int RO_WARP_W2B = 2 + RO_EPI_WARPS;
constexpr int RO_WARP_BASE = RO_WARP_W2B + 1;
constexpr int RO_THREADS = (RO_WARP_BASE + 1) * 32;
constexpr uint32_t RO_W2_BOX = 64 * RO_HALF * 2;       // 64 K x 64 vocab (8 KB)
constexpr int RO_MAX_KCH = 8;                          // R <= 512 (K chunks of 64)
constexpr uint32_t RO_W2_SLOT = RO_MAX_KCH * RO_W2_BOX;  // one tile's W2t half: 64 KB per CTA
constexpr int RO_PREFETCH_TILES = 6;                   // W2t tiles pulled into L2 early (one M tile only)
constexpr int RO_SLOTS = 2;                            // slot t % 2 holds tile t, refilled by producer t % 2
constexpr uint32_t RO_BASE_BOX = RO_BM * 64 * 2;       // base box: 128 rows x 64 cols (16 KB)
constexpr uint32_t RO_BASE_TILE = RO_BM * RO_BN * 2;   // 32 KB
constexpr int RO_NBASE = 3;
// latent boxes per staging round: the still-empty base ring's six 16 KB
// boxes and the second W2 slot's four (its first W2 tile is requested once
// the latent has been copied to TMEM), so R <= 512 stages in one round
constexpr int RO_A_IN_BASE = 2 * RO_NBASE;
constexpr int RO_A_ROUND = RO_A_IN_BASE + (int)(RO_W2_SLOT / RO_BASE_BOX);
constexpr uint32_t RO_TMEM_A = 0;                      // A: columns [0, 32*kch)
constexpr uint32_t RO_TMEM_ACC = 256;                  // accumulators: [256, 384), [384, 512)

struct ReadoutParams {
  const uint16_t* lat;
  int32_t rows, V, R, kch, mp, nt, per, B;  // kch = ceil(R / 64) K chunks (boxes) per tile
  // rows per latent / base box: 128, or the rows of a lone partial M tile
  // rounded up to 8 (fewer rows copied; the rest of the box is never read out)
  int32_t box_rows;
  int64_t* blk;
  int32_t* changed;
  unsigned long long* keys;
  unsigned int* rcnt;    // per-row arrival counters (zero between calls)
  WsHeader* hdr;
  const uint32_t* skip;  // nullable: see pass_skipped
  int32_t* passes_out;   // nullable: fixpoint pass count
  // nonzero: the while-node handle of a captured fixpoint loop; the last CTA
  // sets it to 0 after the pass that changed nothing or the max_passes-th pass
  unsigned long long cond;
  int32_t max_passes;
};

// One 32-column chunk of one row: acc (fp32) -> bias = bf16(acc);
// s = bf16(base + bias); update the running (best, first column).  Base
// columns at or past V arrive as NaN (the base tensor map's out-of-range
// fill), so their sums are NaN: max.bf16x2 ignores a NaN operand and a NaN
// never equals the maximum, so padding columns can neither raise the maximum
// nor be chosen (for an odd V the upper half of the last pair included).
__device__ __forceinline__ void ro_chunk(const uint32_t (&r)[32], const uint32_t (&bw)[16], int col0,
                                         float& best, int& bidx) {
  uint32_t s2[16];
  uint32_t m2 = 0xff80ff80u;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const uint32_t bias2 = f32x2_to_bf16x2(__uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]));
    s2[q] = bf16x2_add(bw[q], bias2);
    m2 = bf16x2_max(m2, s2[q]);
  }
  const float m = fmaxf(bf16lo_to_f32(m2), bf16hi_to_f32(m2));
  if (m > best || bidx < 0) {
    int cand = -1;
#pragma unroll
    for (int q = 15; q >= 0; --q) {
      if (bf16hi_to_f32(s2[q]) == m) cand = 2 * q + 1;
      if (bf16lo_to_f32(s2[q]) == m) cand = 2 * q;
    }
    if (cand >= 0) {
      best = m;
      bidx = col0 + cand;
    }
  }
}

__global__ void __launch_bounds__(RO_THREADS, 1)
readout_argmax_kernel(const __grid_constant__ CUtensorMap mapW2, const __grid_constant__ CUtensorMap mapBase,
                      const __grid_constant__ CUtensorMap mapLat, const ReadoutParams p) {
  extern __shared__ uint8_t smem_raw[];
  // rounded up to 1024 bytes as an offset from smem_raw, so the compiler
  // keeps the shared address space for every pointer derived from it
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sB = smem;                                                  // RO_SLOTS x 64 KB
  uint8_t* sBase = smem + (size_t)RO_SLOTS * RO_W2_SLOT;                // RO_NBASE x 32 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sBase + (size_t)RO_NBASE * RO_BASE_TILE);
  uint64_t* b_full = bars;
  uint64_t* base_full = b_full + RO_SLOTS;
  uint64_t* base_empty = base_full + RO_NBASE;
  uint64_t* acc_full = base_empty + RO_NBASE;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* a_ready = acc_empty + 2;
  uint64_t* drain = a_ready + 1;
  uint64_t* a_full = drain + 1;  // [2]: latent rounds landed in the base ring
  uint64_t* a_free = a_full + 2;  // the epilogue warps copied a round to TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(a_free + 1);
  // where latent box b of a staging round lands
  auto a_box = [&](int b) -> uint8_t* {
    return b < RO_A_IN_BASE ? sBase + (size_t)b * RO_BASE_BOX
                            : sB + RO_W2_SLOT + (size_t)(b - RO_A_IN_BASE) * RO_BASE_BOX;
  };
  if (pass_skipped(p.skip, false)) return;  // both CTAs of a pair read the same flag
  if (threadIdx.x == 0) XP_TRACE_MARK(0);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: the pair's leader
  const int pair = (int)(blockIdx.x >> 1);
  const int m_tile = 2 * (pair % p.mp) + (int)rank;
  const int jslot = pair / p.mp;
  const int n_begin = (int)((int64_t)jslot * p.nt / p.per);
  const int n_end = (int)((int64_t)(jslot + 1) * p.nt / p.per);
  const int ntiles = n_end - n_begin;

  // Barriers live at the same offsets in both CTAs.  b_full, acc_empty and
  // a_ready are used in the leader only (both CTAs count on them); acc_full
  // is arrived on in both CTAs by the leader's commits.
  if (threadIdx.x == 0) {
    for (int s = 0; s < RO_SLOTS; ++s) mbar_init(&b_full[s], 1);  // the leader's arrive_expect_tx (both halves)
    for (int s = 0; s < RO_NBASE; ++s) {
      mbar_init(&base_full[s], 1);
      mbar_init(&base_empty[s], 1);  // one arrive per CTA after the epilogue warps' barrier
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 2);  // one (release) arrive per CTA of the pair
    }
    mbar_init(a_ready, 2);  // one (release) arrive per CTA of the pair
    mbar_init(drain, 1);
    mbar_init(&a_full[0], 1);
    mbar_init(&a_full[1], 1);
    mbar_init(a_free, RO_EPI_WARPS);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) XP_TRACE_MARK(1);
  // Programmatic dependent launch: the next kernel in the stream (the next
  // pass's first latent kernel) may start its prologue as SMs free up; it
  // waits for this grid before it reads blk.  This grid, in turn, may have
  // started while the latent stage was still running: only the W2 producers
  // and the base producer's L2 prefetch (W2t and base are never written by a
  // pass) run ahead of the wait below.
  pdl_launch_dependents();
  if (warp != 0 && warp != RO_WARP_W2B && warp != RO_WARP_BASE) pdl_wait();
  // Copies this CTA requested, for the drain before exit when a wait timed
  // out (on the normal path every copy is consumed before the end)
  int timed_out = 0;      // this thread saw a wait run out
  uint32_t w2_armed = 0;  // phases of b_full[pid] a leader producer armed
  int lat_issued = 0;     // latent rounds requested
  int base_issued = 0;    // base tiles requested
  // the leader's copy of a barrier, as a shared::cluster address
  auto leader_bar = [](uint64_t* b) { return mapa_shared(smem_u32(b), 0u); };
  // arrive on the leader's copy of a barrier (locally in the leader)
  auto arrive_leader = [&](uint64_t* b) {
    if (rank == 0) mbar_arrive(b);
    else mbar_arrive_remote(leader_bar(b));
  };

  if (warp == 0 || warp == RO_WARP_W2B) {
    // ---------------- TMA producers: W2t tile slots ----------------
    // slot s = t % 2 is always refilled by producer s, after the pair's
    // commit of tile t-2 (acc_full of that slot, arrived in both CTAs) shows
    // the MMAs that read it are done.  Lane 0 waits (and, in the leader,
    // arms the pair's barrier for both halves); lanes 0..kch-1 issue one box
    // each (a single thread issues tiled copies slowly).
    const int pid = warp == 0 ? 0 : 1;
    if (pid == 0 && lane == 0) prefetch_tensormap(&mapW2);
    const uint64_t pol = policy_evict_first();  // read once per pass
    bool dead = false;
    for (int t = pid; t < ntiles; t += RO_SLOTS) {
      const int n0 = (n_begin + t) * RO_BN;
      const uint32_t u = (uint32_t)t >> 1;
      int ok = 1;
      if (lane == 0) {
        // the second slot holds latent boxes until they are in TMEM
        if (t == 1 && p.kch > RO_A_IN_BASE && !mbar_wait(a_free, 0)) ok = 0;
        else if (u >= 1 && !mbar_wait_cluster(&acc_full[pid], (u - 1) & 1)) ok = 0;
        else if (rank == 0) {
          mbar_arrive_expect_tx(&b_full[pid], 2u * (uint32_t)p.kch * RO_W2_BOX);
          ++w2_armed;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        dead = true;
        break;
      }
      // this CTA's half: vocab rows [n0 + 64 * rank, +64) of W2t
      if (lane < p.kch)
        tma_load_2d_pair(sB + (size_t)pid * RO_W2_SLOT + lane * RO_W2_BOX, &mapW2, lane * 64,
                         n0 + (int)rank * RO_HALF, leader_bar(&b_full[pid]), pol);
      if (t == 0 && p.rows <= RO_BM) {
        // A small batch (one M tile) leaves most SMs idle during the latent
        // stage, and its readout CTAs are resident early: they pull the next
        // RO_PREFETCH_TILES tiles of their W2t half into L2 meanwhile (more
        // than that measured slower: the pulls then delay the latent stage's
        // own reads)
        for (int j = lane; j < RO_PREFETCH_TILES * p.kch; j += 32) {
          const int pt = 1 + j / p.kch, bx = j - (pt - 1) * p.kch;
          if (pt < ntiles) tma_prefetch_2d(&mapW2, bx * 64, (n_begin + pt) * RO_BN + (int)rank * RO_HALF);
        }
      }
      if (t == pid) pdl_wait();  // after the first tile of this slot is requested
    }
    pdl_wait();  // returns at once if already passed above
    if (dead && lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    timed_out = dead;
    if (pid == 0 && lane == 0) XP_TRACE_MARK(7);
  } else if (warp == RO_WARP_BASE) {
    // ---------------- TMA producer: base tiles (two lanes, one box each) ----------------
    // The latent tile (A) goes first, through the still-empty base ring and
    // second W2 slot: rounds of up to RO_A_ROUND 64-column boxes (one round
    // for R <= 512), each copied to TMEM by the epilogue warps before the
    // space is reused.
    const int rounds = (p.kch + RO_A_ROUND - 1) / RO_A_ROUND;
    bool a_dead = false;
    const uint64_t pol_base = policy_evict_first();  // read once per pass
    // an M tile with no rows (the second tile of a lone pair) copies nothing:
    // its barriers complete on the arrival alone
    const bool live = m_tile * RO_BM < p.rows;
    const uint32_t box_bytes = live ? (uint32_t)p.box_rows * 128u : 0u;
    if (lane == 0) {
      prefetch_tensormap(&mapLat);
      prefetch_tensormap(&mapBase);
    }
    // the first base tiles into L2 while the latent is still being computed
    if (live && lane < 2 * RO_NBASE && lane / 2 < ntiles)
      tma_prefetch_2d(&mapBase, (n_begin + lane / 2) * RO_BN + (lane & 1) * 64, m_tile * RO_BM);
    pdl_wait();
    for (int r = 0; r < rounds && !a_dead; ++r) {
      const int nbox = p.kch - RO_A_ROUND * r < RO_A_ROUND ? p.kch - RO_A_ROUND * r : RO_A_ROUND;
      int ok = 1;
      if (lane == 0) {
        if (r >= 1 && !mbar_wait(a_free, (r - 1) & 1)) ok = 0;
        else mbar_arrive_expect_tx(&a_full[r], (uint32_t)nbox * box_bytes);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        a_dead = true;
        break;
      }
      if (live && lane < nbox)
        tma_load_2d(a_box(lane), &mapLat, (RO_A_ROUND * r + lane) * 64, m_tile * RO_BM, &a_full[r]);
      lat_issued = r + 1;
    }
    {
      int ok = 1;
      if (lane == 0 && (a_dead || !mbar_wait(a_free, (rounds - 1) & 1))) ok = 0;
      a_dead = !__shfl_sync(0xffffffffu, ok, 0);
    }
    if (a_dead) {
      timed_out = 1;
      if (lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
    } else {
      for (int t = 0; t < ntiles; ++t) {
        const int n0 = (n_begin + t) * RO_BN;
        const uint32_t bb = t % RO_NBASE, k = t / RO_NBASE;
        int ok = 1;
        if (lane == 0) {
          if (k >= 1 && !mbar_wait(&base_empty[bb], (k - 1) & 1)) ok = 0;
          else mbar_arrive_expect_tx(&base_full[bb], 2u * box_bytes);
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          timed_out = 1;
          if (lane == 0) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
          break;
        }
        base_issued = t + 1;
        if (live && lane < 2)
          tma_load_2d_hint(sBase + (size_t)bb * RO_BASE_TILE + lane * RO_BASE_BOX, &mapBase, n0 + lane * 64,
                           m_tile * RO_BM, &base_full[bb], pol_base);
      }
    }
    if (lane == 0) XP_TRACE_MARK(8);
  } else if (warp == 1) {
    // ---------------- MMA issuer (the pair's leader) ----------------
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * RO_BM, RO_BN, 0, 0);
      bool dead = !mbar_wait_cluster(a_ready, 0);
      tc_fence_after();
      const int ksteps = (p.R + 15) / 16;
      // slot 0's W2t descriptor; slot 1 adds the slot size (address field:
      // 16-byte units)
      const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sB), 16, 1024);
      for (int t = 0; t < ntiles && !dead; ++t) {
        const uint32_t a = t & 1, u = t >> 1;
        if (u >= 1 && !mbar_wait_cluster(&acc_empty[a], (u - 1) & 1)) {
          dead = true;
          break;
        }
        if (t < 16) XP_TRACE_MARK(42 + t);
        if (!mbar_wait(&b_full[a], u & 1)) {
          dead = true;
          break;
        }
        tc_fence_after();
        if (t == 0) XP_TRACE_MARK(3);
        if (t < 16) XP_TRACE_MARK(26 + t);
        const uint32_t d = tmem + RO_TMEM_ACC + a * RO_BN;
        // A: TMEM columns hold K pairs; a K step of 16 is 8 columns.
        // B: K-major (W2t rows), 128-byte rows, 8-row groups 1024 B apart;
        // a K step of 16 advances 32 bytes inside a 64-wide box.  The
        // descriptor's address field is in 16-byte units, so the steps are
        // added to the slot's descriptor directly.
        const uint64_t bdesc = bdesc0 + (uint64_t)(a * (RO_W2_SLOT >> 4));
        // R = 512 fills the tile's K: its MMAs go out without a per-MMA
        // predicate (whatever else the single issuing thread does between
        // MMAs delays them)
        if (ksteps == RO_MAX_KCH * 4) {
#pragma unroll
          for (int kk = 0; kk < RO_MAX_KCH * 4; ++kk)
            tc_mma_f16_ts_pair(d, tmem + RO_TMEM_A + kk * 8,
                               bdesc + (uint64_t)(((kk >> 2) * RO_W2_BOX + (kk & 3) * 32) >> 4), idesc, kk != 0);
        } else {
#pragma unroll
          for (int kk = 0; kk < RO_MAX_KCH * 4; ++kk) {
            if (kk < ksteps)
              tc_mma_f16_ts_pair(d, tmem + RO_TMEM_A + kk * 8,
                                 bdesc + (uint64_t)(((kk >> 2) * RO_W2_BOX + (kk & 3) * 32) >> 4), idesc, kk != 0);
          }
        }
        tc_commit_pair(&acc_full[a], 0x3);
      }
      if (dead) flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      timed_out = dead;
      XP_TRACE_MARK(4);
      tc_commit_pair(drain, 0x1);
      (void)mbar_wait(drain, 0);
    }
  } else if (warp >= 2 && warp < 2 + RO_EPI_WARPS) {
    // ---------------- epilogue warps ----------------
    const int q = warp & 3;          // TMEM lane quadrant this warp may access
    const int h = (warp - 2) >> 2;   // 64-column half of the tile
    const int rr = q * 32 + lane;    // row within the M tile
    const int row = m_tile * RO_BM + rr;
    const bool row_ok = row < p.rows;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;

    // Stage the A operand (this row of the latent, zero-padded to 64*kch)
    // into TMEM columns [0, 32*kch).  The latent arrives by TMA in the base
    // ring and the second W2 slot, 128-byte swizzled (chunk c of row rr at
    // (c ^ rr%8)*16), in rounds of up to RO_A_ROUND 64-column boxes (one
    // round when R <= 640); the two warps of a lane quadrant take alternate
    // boxes.
    {
      const int rounds = (p.kch + RO_A_ROUND - 1) / RO_A_ROUND;
      bool ok = true;
      for (int r = 0; r < rounds; ++r) {
        if (ok && !mbar_wait(&a_full[r], 0)) {
          ok = false;
          timed_out = 1;
          flag_error(p.hdr, XP_DEVERR_TIMEOUT);
        }
        if (ok && m_tile * RO_BM < p.rows) {  // an M tile with no rows leaves its A alone
#pragma unroll
          for (int j = 0; j < RO_A_ROUND / 2; ++j) {
            const int box = 2 * j + h, kc = RO_A_ROUND * r + box;
            if (kc < p.kch) {
              const uint8_t* src = a_box(box) + (size_t)rr * 128;
              uint32_t v[32];
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint4 x = *reinterpret_cast<const uint4*>(src + ((c ^ (rr & 7)) << 4));
                v[4 * c] = x.x;
                v[4 * c + 1] = x.y;
                v[4 * c + 2] = x.z;
                v[4 * c + 3] = x.w;
              }
              tmem_st_32x32b_x32(tmem + lane_addr + RO_TMEM_A + kc * 32, v);
            }
          }
          tmem_st_wait();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(a_free);  // this warp is done reading the round
      }
      tc_fence_before();
      named_barrier_sync(2, 32 * RO_EPI_WARPS);
      if (threadIdx.x == 64) {
        arrive_leader(a_ready);
        XP_TRACE_MARK(2);
      }
    }

    float best = -INFINITY;
    int bidx = -1;
    bool dead = false;
    for (int t = 0; t < ntiles; ++t) {
      const uint32_t a = t & 1, u = t >> 1;
      const uint32_t bb = t % RO_NBASE, kb = t / RO_NBASE;
      const int n0 = (n_begin + t) * RO_BN + h * 64;
      if (!dead && !mbar_wait(&base_full[bb], kb & 1)) {
        dead = true;
        timed_out = 1;
        flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      }
      if (!dead && !mbar_wait(&acc_full[a], u & 1)) {
        dead = true;
        timed_out = 1;
        flag_error(p.hdr, XP_DEVERR_TIMEOUT);
      }
      tc_fence_after();
      if (!dead) {
        // this row of the base box for columns [n0, n0+64): 128 bytes, its
        // 16-byte chunks permuted by the 128-byte swizzle (chunk ^ row%8)
        const uint8_t* brow = sBase + (size_t)bb * RO_BASE_TILE + (size_t)h * RO_BASE_BOX + (size_t)rr * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem + lane_addr + RO_TMEM_ACC + a * RO_BN + h * 64 + c * 32, r);
          uint32_t bw[16];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 x = *reinterpret_cast<const uint4*>(brow + (((4 * c + v) ^ (rr & 7)) << 4));
            bw[4 * v] = x.x;
            bw[4 * v + 1] = x.y;
            bw[4 * v + 2] = x.z;
            bw[4 * v + 3] = x.w;
          }
          tmem_ld_wait();
          ro_chunk(r, bw, n0 + c * 32, best, bidx);
        }
      }
      // the eight epilogue warps meet, then one thread releases the
      // accumulator and the base slot: a cluster-scope release arrive costs
      // a memory barrier, so one per CTA and tile instead of one per warp
      tc_fence_before();
      named_barrier_sync(2, 32 * RO_EPI_WARPS);
      if (threadIdx.x == 64) {
        arrive_leader(&acc_empty[a]);
        mbar_arrive(&base_empty[bb]);
      }
      if (threadIdx.x == 64 && t < 16) XP_TRACE_MARK(10 + t);
    }
    // Fold this (row, half) winner into the row's key, then count the
    // arrival: the 2 * per arrivals of a row (both halves of every vocab
    // range) complete it, and the thread whose arrival does publishes the row
    // and re-zeroes its key and counter; no CTA waits for the others.  A
    // thread whose wait timed out still arrives (the row completes; the
    // error bit is set).
    if (row_ok) {
      if (bidx >= 0 && !dead) atomicMax(&p.keys[row], make_key(best, (uint32_t)bidx));
      // the arrival releases this fold and, for the row's last arrival,
      // acquires every other one
      if (atom_add_acq_rel_gpu(&p.rcnt[row], 1u) == 2u * (uint32_t)p.per - 1u) {
        const unsigned long long k = atomicExch(&p.keys[row], 0ull);
        p.rcnt[row] = 0u;
        const int64_t idx = (int64_t)key_index(k);
        const int64_t n = row / (p.B - 1), jj = row - n * (p.B - 1);
        int64_t* slot = p.blk + n * p.B + 1 + jj;
        if (p.changed != nullptr || p.passes_out != nullptr) {
          if (*slot != idx) {
            if (p.changed) atomicAdd(p.changed, 1);
            if (p.passes_out) atomicAdd(&p.hdr->pass_changed, 1u);
          }
        }
        *slot = idx;
      }
    }
  }

  __syncwarp();  // lane-0 roles rejoin their warps before any .aligned op
  tc_fence_before();
  // After a timeout some copies this CTA requested may never have been
  // consumed: each producer waits (bounded) for the last phase it armed on
  // each of its barriers before the pair may exit.  Earlier phases of a
  // barrier are complete: a phase is re-armed only after its previous one
  // was consumed.  The peer's W2 halves count on the leader's b_full, and the
  // peer cannot exit before the cluster barrier below.
  if (__syncthreads_or(timed_out) && lane == 0) {
    if ((warp == 0 || warp == RO_WARP_W2B) && w2_armed > 0)
      (void)mbar_wait(&b_full[warp == 0 ? 0 : 1], (w2_armed - 1) & 1);
    if (warp == RO_WARP_BASE) {
      for (int r = 0; r < lat_issued; ++r) (void)mbar_wait(&a_full[r], 0);
      for (int t = base_issued > RO_NBASE ? base_issued - RO_NBASE : 0; t < base_issued; ++t)
        (void)mbar_wait(&base_full[t % RO_NBASE], (uint32_t)(t / RO_NBASE) & 1);
    }
  }
  __syncwarp();
  // the leader's MMAs are complete (drain) and no remote arrive is in flight
  // once both CTAs are here
  cluster_sync();
  if (threadIdx.x == 0) XP_TRACE_MARK(5);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
  // Fixpoint driver only: the last CTA to finish counts the pass, and a pass
  // that changed no slot is the last one (the passes launched after it exit
  // at once; in a captured loop, the while node stops).  Every row of the
  // pass is published by then: each CTA counts itself after its threads' rows.
  if (p.passes_out != nullptr) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(&p.hdr->done, 1u) == gridDim.x - 1) {
        __threadfence();
        const uint32_t np = p.hdr->passes + 1u;
        p.hdr->passes = np;
        *p.passes_out = (int32_t)np;
        const bool last = atomicExch(&p.hdr->pass_changed, 0u) == 0u;
        if (last) p.hdr->converged = 1u;
        p.hdr->done = 0u;
        if (p.cond != 0ull)
          cudaGraphSetConditional((cudaGraphConditionalHandle)p.cond,
                                  (!last && (int32_t)np < p.max_passes) ? 1u : 0u);
      }
    }
  }
  if (threadIdx.x == 0) XP_TRACE_MARK(6);
}

size_t readout_smem_bytes() {
  return 1024 + (size_t)RO_SLOTS * RO_W2_SLOT + (size_t)RO_NBASE * RO_BASE_TILE +
         8 * (RO_SLOTS + 2 * RO_NBASE + 9) + 16;
}

namespace {
// Work split: mp pairs of 128-row M tiles x per contiguous vocabulary ranges
// of 128-wide tiles, one CTA pair each (2 * mp * per <= SMs).
struct RoSplit {
  int32_t mp, nt, per;
};
RoSplit readout_split(int sms, int64_t rows, int64_t V) {
  RoSplit s;
  const int64_t mt = (rows + RO_BM - 1) / RO_BM;
  s.mp = (int32_t)((mt + 1) / 2);
  s.nt = (int32_t)((V + RO_BN - 1) / RO_BN);
  s.per = sms / (2 * s.mp);
  if (s.per < 1) s.per = 1;
  if (s.per > s.nt) s.per = s.nt;
  return s;
}

struct RoDevInfo {
  bool init = false;
  int sms = 0;
};
RoDevInfo g_ro_dev[64];
}  // namespace

xp_status launch_readout_argmax(const uint16_t* lat, const uint16_t* W2t, const uint16_t* base, int64_t ld_base,
                                int64_t rows, int64_t V, int64_t R, int64_t* blk, int64_t B, int32_t* changed,
                                void* ws, cudaStream_t stream, const uint32_t* skip, int32_t* passes_out,
                                unsigned long long cond, int32_t max_passes) {
  if (rows <= 0) return XP_OK;
  const int kch = (int)((R + 63) / 64);
  if (kch > RO_MAX_KCH) return XP_ERR_SHAPE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return XP_ERR_LAUNCH;
  RoDevInfo& info = g_ro_dev[dev];
  const size_t smem = readout_smem_bytes();
  if (!info.init) {
    int max_smem = 0;
    if (cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return XP_ERR_LAUNCH;
    if (smem > (size_t)max_smem) return XP_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(readout_argmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return XP_ERR_LAUNCH;
    info.init = true;
  }

  CUtensorMap mapW2, mapBase, mapLat;
  if (!cached_map_bf16_2d(&mapW2, W2t, (uint64_t)R, (uint64_t)V, (uint64_t)R, 64, RO_HALF)) return XP_ERR_LAUNCH;
  // base: columns past V read as NaN (see ro_chunk)
  // a lone partial M tile (rows < 128) copies only its rows, rounded up to 8
  const int32_t box_rows = rows < RO_BM ? (int32_t)((rows + 7) / 8 * 8) : RO_BM;
  if (!cached_map_bf16_2d(&mapBase, base, (uint64_t)V, (uint64_t)rows, (uint64_t)ld_base, 64, (uint32_t)box_rows,
                          true))
    return XP_ERR_LAUNCH;
  if (!cached_map_bf16_2d(&mapLat, lat, (uint64_t)R, (uint64_t)rows, (uint64_t)R, 64, (uint32_t)box_rows))
    return XP_ERR_LAUNCH;

  ReadoutParams p;
  ArgmaxWs w = argmax_ws(ws, rows);
  const RoSplit sp = readout_split(info.sms, rows, V);
  p.lat = lat;
  p.rows = (int32_t)rows;
  p.V = (int32_t)V;
  p.R = (int32_t)R;
  p.kch = kch;  // A staged in TMEM up to the last K chunk, zero beyond R
  p.box_rows = box_rows;
  p.mp = sp.mp;
  p.nt = sp.nt;
  p.per = sp.per;
  const int per = sp.per;
  p.B = (int32_t)B;
  p.blk = blk;
  p.changed = changed;
  p.keys = w.keys;
  p.rcnt = w.cnt;
  p.hdr = w.hdr;
  p.skip = skip;
  p.passes_out = passes_out;
  p.cond = cond;
  p.max_passes = max_passes;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3((unsigned int)(2 * p.mp * per));
  cfg.blockDim = dim3(RO_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, readout_argmax_kernel, mapW2, mapBase, mapLat, p) != cudaSuccess) {
    (void)cudaGetLastError();  // a failed launch must not be reported again by a later call
    return XP_ERR_LAUNCH;
  }
  return XP_OK;
}

}  // namespace xp

XP_TRACE_READER(xp_trace_read_readout)
