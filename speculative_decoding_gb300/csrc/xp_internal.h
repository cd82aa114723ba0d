// xp_internal.h -- launchers behind the C ABI (host side, not exported).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/xpress.h"

namespace xp {

xp_status launch_add_argmax(const uint16_t* base, int64_t ld_base, const uint16_t* bias, int64_t ld_bias,
                            int64_t rows, int64_t V, int64_t* blk, int64_t B, void* ws,
                            cudaStream_t stream);

// xp_add_argmax on the library's fixed per-device scratch (no workspace).
xp_status launch_add_argmax_noalloc(const uint16_t* base, int64_t ld_base, const uint16_t* bias, int64_t ld_bias,
                                    int64_t rows, int64_t V, int64_t* blk, int64_t B, cudaStream_t stream);

// xp_topc_argmax: one warp per row, no workspace.
xp_status launch_topc_argmax(const uint16_t* base_c, const uint16_t* bias_c, const int64_t* cand, int64_t rows,
                             int64_t C, int64_t* blk, int64_t B, cudaStream_t stream);

// skip (nullable): the pass's fixpoint flag (pass_skipped); passes_out
// (nullable): the readout's last CTA counts the pass there and sets the flag
// when the pass changed no slot.  cond (with passes_out; 0 = none): the
// handle of a captured while node, which the same CTA sets to continue while
// the pass changed a slot and fewer than max_passes passes have run.
xp_status launch_readout_argmax(const uint16_t* lat, const uint16_t* W2t, const uint16_t* base, int64_t ld_base,
                                int64_t rows, int64_t V, int64_t R, int64_t* blk, int64_t B, int32_t* changed,
                                void* ws, cudaStream_t stream, const uint32_t* skip = nullptr,
                                int32_t* passes_out = nullptr, unsigned long long cond = 0,
                                int32_t max_passes = 0);

xp_status launch_latent(const int64_t* blk, const int64_t* am1, const uint16_t* hcache, const uint16_t* E,
                        const uint16_t* W_lat, const float* L, const uint16_t* Wg, const uint16_t* Wu,
                        const uint16_t* Wd, uint16_t* lat_out, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R,
                        int64_t H, void* ws, cudaStream_t stream, const uint32_t* skip = nullptr,
                        bool do_mlp = true);

// The failure-detection self-test: a bounded wait that runs out (limit_ns).
xp_status launch_wait_timeout_probe(void* ws, unsigned long long limit_ns, cudaStream_t stream);

}  // namespace xp
