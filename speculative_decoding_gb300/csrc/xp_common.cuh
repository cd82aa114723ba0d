// xp_common.cuh -- small device helpers shared by the xpress kernels:
// packed bf16 arithmetic, the order-preserving (value, lowest index) key used
// to fold partial argmaxes across CTAs, and the workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/xpress.h"

namespace xp {

// ---------------------------------------------------------------------------
// packed bf16 arithmetic (two values per 32-bit word; the lower address is the
// low half)
// ---------------------------------------------------------------------------

// Correctly rounded (round-to-nearest-even) bf16 sum of two packed pairs.
// A single rounding of the exact sum equals rounding the fp32 sum, which is
// the rounding the method prescribes (the sum is cast back to bf16 before the
// compare).
__device__ __forceinline__ uint32_t bf16x2_add(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Lane-wise maximum of two packed pairs (inputs are finite).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two fp32 values -> packed bf16 pair, each rounded to nearest even
// (lo goes to the low half).
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ---------------------------------------------------------------------------
// (value, index) keys: a 64-bit unsigned integer whose order is "larger value
// first, then lower index", so atomicMax over keys folds partial argmaxes with
// the lowest-index tie rule in any arrival order.  -0 is mapped to +0 first
// so the two zeros tie.  Key 0 is below every real key (the empty state).
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long make_key(float val, uint32_t idx) {
  uint32_t b = __float_as_uint(val);
  if (b == 0x80000000u) b = 0u;
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xffffffffu - idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return 0xffffffffu - (uint32_t)(k & 0xffffffffull);
}

// ---------------------------------------------------------------------------
// streaming loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------------------
// workspace layout (all offsets 256-byte aligned)
//   [0, 256)            header: error bits, grid-done counters
//   keys  u64[rows]     per-row folded (value, index) key, zero between calls
//   cnt   u32[rows]     per-row arrival counter, zero between calls
//   then the latent stage's buffers (see xp_latent.cu)
// ---------------------------------------------------------------------------
struct WsHeader {
  unsigned int err;         // XP_DEVERR_* bits
  unsigned int done;          // CTAs of the current readout grid that finished (fixpoint driver)
  unsigned int pass_changed;  // slots the current pass changed (fixpoint driver)
  // xp_jacobi_fixpoint: nonzero once a pass changed no slot (the passes
  // launched after it exit at once), and the number of passes that ran
  unsigned int converged;
  unsigned int passes;
  unsigned int pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

__host__ __device__ constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct ArgmaxWs {
  WsHeader* hdr;
  unsigned long long* keys;
  unsigned int* cnt;
};

__host__ __device__ constexpr size_t argmax_ws_bytes(int64_t rows) {
  return 256 + align256(sizeof(unsigned long long) * (size_t)rows) + align256(4 * (size_t)rows);
}
__host__ inline ArgmaxWs argmax_ws(void* ws, int64_t rows) {
  char* p = (char*)ws;
  ArgmaxWs w;
  w.hdr = (WsHeader*)p;
  w.keys = (unsigned long long*)(p + 256);
  w.cnt = (unsigned int*)(p + 256 + align256(sizeof(unsigned long long) * (size_t)rows));
  return w;
}

// Tiling of the latent stage's projection x = E[prev] @ W_lat (shared by the
// kernel launch and the workspace layout): M tiles of bpt whole blocks
// (<= 128 rows), N tiles of tn latent channels, the D-long reduction split
// S ways; each split writes an fp32 partial tile that the S CTAs of the tile
// then sum in a fixed order.
struct ProjTiling {
  int32_t bpt, mtiles, tn, ntiles, chunks, S, w;
  int32_t lw;  // mixer-weight columns held at once: w, or w/2 (two rounds) when w columns do not fit
  int64_t rows_pad, r_pad;  // partial-sum buffer: [S][rows_pad][r_pad] fp32
};

// The projection kernel's dynamic shared memory for a tiling and a ring of
// `stages` stages (128-row A chunks of 64 K columns plus a tn-wide W_lat
// box each).  [0, region): the ring; after the MMAs the same place holds the
// S partial slices and xs (w columns each), then the outgoing partial tile,
// whose place the mixer's output (u fp32 and bf16(u), w columns) takes later:
// the larger of the two.  Then the mixer weights of the w columns (the whole
// [B][B] square), the hidden cache of those columns, the token table, and the
// barriers (full/empty per stage, acc_full, aux_full, slice_full, ls_full) and
// the TMEM address slot; 1024 bytes of alignment slack in front.
struct ProjSmem {
  uint32_t region, hc_off, tok_off, bar_off;
  size_t total;
};
__host__ inline ProjSmem proj_smem(const ProjTiling& t, int64_t B, int stages) {
  constexpr size_t rows = 128;
  const size_t stage_bytes = rows * 64 * 2 + (size_t)t.tn * 64 * 2;
  const size_t pst = rows * (size_t)(t.tn * 4 > t.w * 6 ? t.tn * 4 : t.w * 6);
  const size_t sl_xs = (((size_t)(t.S + 1) * rows * t.w * 4 + 1023) & ~size_t(1023)) + pst;
  const size_t ls = ((size_t)(B * B * t.lw * 4) + 127) & ~size_t(127);
  const size_t hc = (rows * t.w * 2 + 127) & ~size_t(127);
  const size_t ring = (size_t)stages * stage_bytes;
  ProjSmem m;
  m.region = (uint32_t)((ring > sl_xs ? ring : sl_xs + 1023) & ~size_t(1023));
  m.hc_off = m.region + (uint32_t)ls;
  m.tok_off = m.hc_off + (uint32_t)hc;
  m.bar_off = m.tok_off + 8 * (uint32_t)rows;
  m.total = 1024 + (size_t)m.bar_off + 8 * (2 * (size_t)stages + 4) + 16;
  return m;
}
// Dynamic shared memory a latent-stage kernel may use: the 227 KB opt-in
// maximum less the static shared memory and a margin.
constexpr size_t kLatentSmemBudget = 226 * 1024;

__host__ inline ProjTiling proj_tiling(int64_t N, int64_t B, int64_t D, int64_t R) {
  ProjTiling t;
  t.bpt = B <= 128 ? (int32_t)(128 / B) : 1;
  t.mtiles = (int32_t)((N + t.bpt - 1) / t.bpt);
  t.tn = R >= 128 ? 128 : 64;
  t.ntiles = (int32_t)((R + t.tn - 1) / t.tn);
  t.chunks = (int32_t)((D + 63) / 64);
  // as many slices as keep the grid within 128 CTAs (one wave at one CTA
  // per SM, so the S CTAs of a tile that wait for each other are resident
  // together), at most 16 and at least 8 channels per CTA
  t.S = 1;
  while (t.S * 2 <= t.chunks && t.S * 2 <= 16 && t.tn / (t.S * 2) >= 8 &&
         (int64_t)t.mtiles * t.ntiles * t.S * 2 <= 128)
    t.S *= 2;
  t.w = t.tn / t.S;
  t.lw = t.w;
  // while a CTA's share of the epilogue (partial slices, mixer tiles and
  // mixer weights) does not fit beside a two-stage ring: first hold the mixer
  // weights of half the columns at a time, then take fewer slices
  while (t.S > 1 && proj_smem(t, B, 2).total > kLatentSmemBudget) {
    if (t.lw == t.w && t.w >= 16) {
      t.lw = t.w / 2;
      continue;
    }
    t.S /= 2;
    t.w = t.tn / t.S;
    t.lw = t.w;
  }
  // with the D sum unsplit (many output tiles) a CTA mixes all its tile's
  // channels: 64-channel tiles keep its shared memory (the mixer weights
  // and the x / u / bf16(u) tiles of those channels) within budget
  if (t.S == 1 && t.tn == 128) {
    t.tn = 64;
    t.ntiles = (int32_t)((R + t.tn - 1) / t.tn);
    t.w = t.tn;
    t.lw = t.w;
  }
  t.rows_pad = (int64_t)t.mtiles * 128;
  t.r_pad = (int64_t)t.ntiles * t.tn;
  return t;
}

// Latent / full-pass workspace: the argmax part for rows = N*(B-1), then
//   u    fp32 [N*B, R]   mixer output (the MLP residual)
//   ub   bf16 [N*B, R]   bf16(u), the MLP input
//   m    bf16 [N*B, H]   bf16(silu(ub@Wg) * (ub@Wu))
//   part fp32 [S, rows_pad, r_pad]  the projection's partial sums
//   cnt  u32  [mtiles * ntiles, 2]  per projection tile: partials written,
//                                   partials read (zero between calls)
//   lat  bf16 [N*(B-1), R]  the latent read by the readout (full pass only)
struct LatentWsLayout {
  size_t u, ub, m, part, cnt, lat, total_latent, total_pass;
};
__host__ inline LatentWsLayout latent_ws_layout(int64_t N, int64_t B, int64_t D, int64_t R, int64_t H) {
  LatentWsLayout L;
  const ProjTiling t = proj_tiling(N, B, D, R);
  size_t off = argmax_ws_bytes(N * (B - 1));
  L.u = off;
  off += align256(4 * (size_t)(N * B * R));
  L.ub = off;
  off += align256(2 * (size_t)(N * B * R));
  L.m = off;
  off += align256(2 * (size_t)(N * B * H));
  L.part = off;
  off += align256(4 * (size_t)t.S * (size_t)t.rows_pad * (size_t)t.r_pad);
  L.cnt = off;
  off += align256(8 * (size_t)t.mtiles * (size_t)t.ntiles);
  L.total_latent = off;
  L.lat = off;
  off += align256(2 * (size_t)(N * (B - 1) * R));
  L.total_pass = off;
  return L;
}

__device__ __forceinline__ void flag_error(WsHeader* h, unsigned int bits) { atomicOr(&h->err, bits); }


}  // namespace xp
