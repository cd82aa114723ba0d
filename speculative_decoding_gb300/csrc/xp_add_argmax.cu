// xp_add_argmax.cu -- the fused add + vocab-wide argmax written into blk.
//
// Method (vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels,
// fused_add_argmax_to_blk with _xpress_add_argmax_partial_kernel and
// _xpress_add_argmax_reduce_to_blk_kernel): for row r = n*(B-1)+j,
// blk[n, 1+j] = lowest v maximising bf16(base[r,v] + bias[r,v]).
//
// GB300 design: one launch, HBM-bound streaming.  Each CTA owns one
// (row, CHUNK-wide vocab slice); every thread issues all of its 16-byte loads
// of base and bias up front (VEC vectors of 8 elements each, coalesced per
// vector step), adds them as packed bf16 pairs (one rounding, RNE) and keeps a
// packed running maximum.  The CTA reduces the maximum, the threads that hold
// it search their registers for its first position, and the CTA folds the
// (value, lowest index) pair into the row's 64-bit key with atomicMax.  The
// last CTA of a row (arrival counter) writes blk and re-zeroes the key and
// counter, so the workspace is clean for the next call and no second launch
// or partial buffer is needed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "xp_common.cuh"
#include "xp_internal.h"
#include "xp_ptx.cuh"

namespace xp {

template <int THREADS, int VEC>
__global__ void __launch_bounds__(THREADS)
add_argmax_kernel(const uint16_t* __restrict__ base, int64_t ld_base, const uint16_t* __restrict__ bias,
                  int64_t ld_bias, int32_t V, int32_t nchunks, int64_t* __restrict__ blk, int32_t B,
                  unsigned long long* __restrict__ keys, unsigned int* __restrict__ cnt) {
  constexpr int CHUNK = THREADS * VEC * 8;
  constexpr int WARPS = THREADS / 32;
  __shared__ float s_max[WARPS];
  __shared__ int s_idx[WARPS];

  const int t = threadIdx.x;
  const int64_t unit = blockIdx.x;
  const int64_t row = unit / nchunks;
  const int32_t chunk = (int32_t)(unit - row * nchunks);
  const uint16_t* pa = base + row * ld_base;
  const uint16_t* pb = bias + row * ld_bias;
  const int32_t v0 = chunk * CHUNK;

  // s[j][k]: packed sums of elements v0 + (j*THREADS + t)*8 + 2k, +1.
  uint32_t s[VEC][4];
  uint4 a[VEC], b[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int32_t v = v0 + (j * THREADS + t) * 8;
    if (v + 8 <= V) {
      a[j] = ld_stream_v4(pa + v);
      b[j] = ld_stream_v4(pb + v);
    } else {
      // ragged tail: element-wise, padding with -inf (never selected: the
      // search below only accepts indices < V)
      uint32_t wa[4], wb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t lo_a = 0xff80u, hi_a = 0xff80u, lo_b = 0u, hi_b = 0u;
        if (v + 2 * k < V) { lo_a = pa[v + 2 * k]; lo_b = pb[v + 2 * k]; }
        if (v + 2 * k + 1 < V) { hi_a = pa[v + 2 * k + 1]; hi_b = pb[v + 2 * k + 1]; }
        wa[k] = lo_a | (hi_a << 16);
        wb[k] = lo_b | (hi_b << 16);
      }
      a[j] = make_uint4(wa[0], wa[1], wa[2], wa[3]);
      b[j] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
    }
  }
  uint32_t m2 = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    s[j][0] = bf16x2_add(a[j].x, b[j].x);
    s[j][1] = bf16x2_add(a[j].y, b[j].y);
    s[j][2] = bf16x2_add(a[j].z, b[j].z);
    s[j][3] = bf16x2_add(a[j].w, b[j].w);
#pragma unroll
    for (int k = 0; k < 4; ++k) m2 = bf16x2_max(m2, s[j][k]);
  }
  const float mt = fmaxf(bf16lo_to_f32(m2), bf16hi_to_f32(m2));

  // CTA maximum
  float m = mt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((t & 31) == 0) s_max[t >> 5] = m;
  __syncthreads();
  float mc = s_max[0];
#pragma unroll
  for (int w = 1; w < WARPS; ++w) mc = fmaxf(mc, s_max[w]);

  // first position of the CTA maximum among this thread's elements
  // (positions increase with j, then k, then the half)
  int cand = 0x7fffffff;
  if (mt == mc) {
#pragma unroll
    for (int j = VEC - 1; j >= 0; --j) {
#pragma unroll
      for (int k = 3; k >= 0; --k) {
        const int32_t v = v0 + (j * THREADS + t) * 8 + 2 * k;
        if (bf16hi_to_f32(s[j][k]) == mc && v + 1 < V) cand = v + 1;
        if (bf16lo_to_f32(s[j][k]) == mc && v < V) cand = v;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
  if ((t & 31) == 0) s_idx[t >> 5] = cand;
  __syncthreads();
  if (t == 0) {
    int ic = s_idx[0];
#pragma unroll
    for (int w = 1; w < WARPS; ++w) ic = min(ic, s_idx[w]);
    atomicMax(&keys[row], make_key(mc, (uint32_t)ic));
    // the arrival releases this CTA's key fold and, for the last CTA of the
    // row, acquires every other CTA's
    const unsigned int arrived = atom_add_acq_rel_gpu(&cnt[row], 1u);
    if (arrived == (unsigned int)nchunks - 1u) {
      const unsigned long long k = atomicExch(&keys[row], 0ull);
      cnt[row] = 0u;
      const int64_t n = row / (B - 1), jj = row - n * (B - 1);
      blk[n * B + 1 + jj] = (int64_t)key_index(k);
    }
  }
}

// 256 threads x 4 vectors of 8 elements: 8192 columns per CTA.  Back to back
// at 480 x 152064, 128 x 8 / 256 x 4 / 256 x 8 / 512 x 4 / 512 x 2 measured
// 45.3 / 45.6 / 46.5 / 51.5 / 55.3 us, but a single cold launch (ncu) took
// 48.9 us with 128 x 8 against 47.0 with 256 x 4
constexpr int AA_THREADS = 256;
constexpr int AA_VEC = 4;

xp_status launch_add_argmax(const uint16_t* base, int64_t ld_base, const uint16_t* bias, int64_t ld_bias,
                            int64_t rows, int64_t V, int64_t* blk, int64_t B, void* ws,
                            cudaStream_t stream) {
  ArgmaxWs w = argmax_ws(ws, rows);
  if (rows <= 0) return XP_OK;
  constexpr int CHUNK = AA_THREADS * AA_VEC * 8;
  const int64_t nchunks = (V + CHUNK - 1) / CHUNK;
  const int64_t grid = rows * nchunks;
  add_argmax_kernel<AA_THREADS, AA_VEC><<<(unsigned int)grid, AA_THREADS, 0, stream>>>(
      base, ld_base, bias, ld_bias, (int32_t)V, (int32_t)nchunks, blk, (int32_t)B, w.keys, w.cnt);
  return cudaGetLastError() == cudaSuccess ? XP_OK : XP_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the keys and counters live in one fixed array of
// device memory per device instead of a caller workspace.  Its layout is the
// workspace layout of argmax_ws() for up to XP_ADD_ARGMAX_NOALLOC_MAX_ROWS rows
// (the size is taken from argmax_ws_bytes itself, so the two cannot drift).
// ---------------------------------------------------------------------------
constexpr size_t kNoallocBytes = argmax_ws_bytes(XP_ADD_ARGMAX_NOALLOC_MAX_ROWS);
static __device__ __align__(256) unsigned char g_add_argmax_scratch[kNoallocBytes];

namespace {
constexpr int kMaxDevices = 64;

// The scratch's device address belongs to the CUDA context that loaded this
// module: a device reset, or a caller that makes another context of the same
// device current, gives a different address.  So the cached address is kept
// with the id of the context it was looked up in (cuCtxGetId: unique for the
// life of the process) and looked up again when the current context differs.
struct ScratchEntry {
  unsigned long long ctx_id = 0;  // 0: nothing cached
  void* ptr = nullptr;
};
ScratchEntry g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// id of the current context, through the runtime's driver entry points (the
// library does not link libcuda); 0 when it cannot be read
unsigned long long current_ctx_id() {
  static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch in the current context: looked up with the
// device current on the first call in each (device, context) and cached.
// The first lookup may load this module's device code.
xp_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return XP_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return XP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchEntry& e = g_scratch[dev];
  unsigned long long id = current_ctx_id();  // 0 before the runtime has made a context current
  if (id == 0 || e.ctx_id != id || e.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_add_argmax_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // do not leave the lookup's error for the next call to find
      return XP_ERR_LAUNCH;
    }
    // the lookup made the device's context current if none was
    if (id == 0) id = current_ctx_id();
    e.ptr = p;
    e.ctx_id = id;  // an unreadable id (0) never matches: such calls look up again
  }
  *out = e.ptr;
  return XP_OK;
}
}  // namespace

xp_status launch_add_argmax_noalloc(const uint16_t* base, int64_t ld_base, const uint16_t* bias, int64_t ld_bias,
                                    int64_t rows, int64_t V, int64_t* blk, int64_t B, cudaStream_t stream) {
  if (rows < 0 || rows > XP_ADD_ARGMAX_NOALLOC_MAX_ROWS) return XP_ERR_SHAPE;
  if (rows == 0) return XP_OK;
  void* ws = nullptr;
  xp_status st = noalloc_scratch(&ws);
  if (st != XP_OK) return st;
  // keys and counters must start at zero; the kernel leaves them zero, but a
  // call that never completed (an error, a killed stream) could have left
  // them dirty, so clear the rows this call uses
  if (cudaMemsetAsync(ws, 0, argmax_ws_bytes(rows), stream) != cudaSuccess) return XP_ERR_LAUNCH;
  return launch_add_argmax(base, ld_base, bias, ld_bias, rows, V, blk, B, ws, stream);
}

}  // namespace xp
