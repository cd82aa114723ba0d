// xp_topc.cu -- the top-C candidate argmax: per draft slot, the argmax over C
// gathered candidates of bf16(base_c + bias_c), mapped back to a vocab id.
//
// Method (vLLM docs, vllm.v1.worker.gpu.spec_decode.xpress.kernels,
// fused_topc_argmax_to_blk / _xpress_topc_argmax_to_blk_kernel): the sum is
// rounded back to bf16 before the compare (as in the full-vocab epilogue),
// ties go to the lowest candidate position, the winner's vocab id
// cand[r, pos] is written to blk[n, 1 + j] for r = n*(B-1) + j.
//
// GB300 design: one warp per row, no workspace and no second launch.  Lanes
// stride over the row's candidates (consecutive lanes read consecutive
// elements), each keeps the 64-bit (value, lowest position) key of its best
// candidate, a shuffle max folds the 32 keys, and lane 0 gathers the vocab
// id.  The key order (larger value, then lower position; -0 == +0) is the
// one the full-vocab kernels fold with atomicMax.
#include "xp_common.cuh"
#include "xp_internal.h"

namespace xp {

constexpr int TC_WARPS = 8;  // rows per CTA

__global__ void __launch_bounds__(TC_WARPS * 32)
topc_argmax_kernel(const uint16_t* __restrict__ base_c, const uint16_t* __restrict__ bias_c,
                   const int64_t* __restrict__ cand, int64_t rows, int64_t C, int64_t* __restrict__ blk, int64_t B) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * TC_WARPS + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint16_t* a = base_c + row * C;
  const uint16_t* b = bias_c + row * C;
  unsigned long long best = 0ull;  // below every real key
  for (int64_t c = lane; c < C; c += 32) {
    // one correctly rounded bf16 add of the pair (the fp32 sum rounded to bf16)
    const uint32_t s2 = bf16x2_add((uint32_t)a[c], (uint32_t)b[c]);
    const unsigned long long k = make_key(bf16lo_to_f32(s2), (uint32_t)c);
    best = k > best ? k : best;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
    best = o > best ? o : best;
  }
  if (lane == 0) {
    const int64_t pos = (int64_t)key_index(best);
    const int64_t n = row / (B - 1), j = row - n * (B - 1);
    blk[n * B + 1 + j] = cand[row * C + pos];
  }
}

xp_status launch_topc_argmax(const uint16_t* base_c, const uint16_t* bias_c, const int64_t* cand, int64_t rows,
                             int64_t C, int64_t* blk, int64_t B, cudaStream_t stream) {
  if (rows <= 0) return XP_OK;
  const int64_t grid = (rows + TC_WARPS - 1) / TC_WARPS;
  topc_argmax_kernel<<<(unsigned)grid, TC_WARPS * 32, 0, stream>>>(base_c, bias_c, cand, rows, C, blk, B);
  return cudaGetLastError() == cudaSuccess ? XP_OK : XP_ERR_LAUNCH;
}

}  // namespace xp
