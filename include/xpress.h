/*
 * xpress.h -- C ABI of libxpress.so: one XPress Jacobi draft pass on one
 * NVIDIA GB300 (sm_103a) GPU.
 *
 * The method (vLLM docs, module "vllm.v1.worker.gpu.spec_decode.xpress.kernels",
 * module docstring): a pass over N blocks of B slots (slot 0 is the verified
 * anchor) computes
 *     latent   u[n,b,:] = causal_mix(hcache[n,b] + E[prev[n,b]] @ W_lat)
 *              x[n,b,:] = u[n,b,:] + SwiGLU_MLP(u[n,b,:])
 *     readout  logits[r,:] = base[r,:] + x[n,1+j,:] @ W2      r = n*(B-1)+j
 *     argmax   blk[n,1+j] = argmax_v logits[r,v]
 * and never stores the [N*(B-1), V] logits.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named d_* are DEVICE pointers owned by the caller.  The library
 *   allocates no device memory, never synchronises the device and only
 *   enqueues work on `stream` (0 = the legacy default stream).
 * - bf16 data is passed as xp_bf16 (the 16-bit pattern of a bfloat16).  Tokens
 *   are int64.  The mixer L is float32.
 * - Matrices are row-major; the latent-stage weights are stored [in, out]
 *   ("transposed" as on the pages: W_lat [D,R], Wg/Wu [R,H], Wd [H,R]).
 *   The readout weight is the one exception: the pages multiply by W2 [R,V],
 *   but every entry point here takes it vocabulary-major, as W2t = W2
 *   transposed, [V,R] (parameter d_W2t), so that the weights of one vocab
 *   tile are one contiguous block.  Passing W2 [R,V] itself is NOT detected
 *   (a raw pointer carries no shape) and gives wrong tokens.
 * - Alignment: every bf16 pointer must be 16-byte aligned and every leading
 *   dimension (ld_*) a multiple of 8 elements, else XP_ERR_ALIGN.  Sizes are
 *   otherwise free (V need not be a multiple of 8 for xp_add_argmax).
 * - Workspace: an opaque caller-provided device buffer of at least the bytes
 *   the matching *_workspace_size() returns, 256-byte aligned, ZEROED ONCE
 *   (e.g. cudaMemsetAsync) before its first use.  Every call leaves its
 *   reduction state zero again, so one workspace serves any number of calls,
 *   but calls that share a workspace must not overlap on the GPU (use one
 *   stream, or one workspace per stream).  A workspace sized for one entry
 *   point may serve a smaller one: xp_jacobi_workspace_size() covers
 *   xp_latent_pass and xp_readout_argmax/xp_add_argmax of the same shapes.
 * - Errors: host-side checks run before any launch and return a status
 *   without touching memory.  Device-side conditions (a token outside
 *   [0, V)) are clamped, recorded in the workspace and reported by
 *   xp_read_error(); kernels never trap.
 * - blk must not alias any other argument.  Slot 0 of blk is never written.
 */
#ifndef XPRESS_H
#define XPRESS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define XP_API __attribute__((visibility("default")))
#else
#define XP_API
#endif

typedef uint16_t xp_bf16;                 /* bfloat16 bit pattern */
typedef struct CUstream_st* xp_stream_t;  /* the same type as cudaStream_t */

typedef int32_t xp_status;
#define XP_OK 0
#define XP_ERR_NULL 1          /* a required pointer is NULL */
#define XP_ERR_SHAPE 2         /* inconsistent or out-of-range sizes */
#define XP_ERR_ALIGN 3         /* pointer or leading dimension misaligned */
#define XP_ERR_WORKSPACE 4     /* workspace missing, too small or misaligned */
#define XP_ERR_LAUNCH 5        /* a CUDA launch or driver call failed */
#define XP_ERR_UNSUPPORTED 6   /* current device is not sm_103 (GB300) */

/* Device-side error bits reported by xp_read_error(). */
#define XP_DEVERR_TOKEN 1u     /* a token in blk/am1 was outside [0, V) and was clamped */
#define XP_DEVERR_TIMEOUT 2u   /* a bounded device-side wait gave up */

/* Human-readable name of a status code (static string, never NULL). */
XP_API const char* xp_status_string(xp_status s);

/* Library version, major*10000 + minor*100 + patch. */
XP_API int32_t xp_version(void);

/* ------------------------------------------------------------------------
 * xp_add_argmax -- the fused add + vocab-wide argmax, written into blk.
 * Pages: fused_add_argmax_to_blk and its two kernels
 * (_xpress_add_argmax_partial_kernel, _xpress_add_argmax_reduce_to_blk_kernel).
 *
 *   for r in [0, rows):  n = r / (B-1), j = r % (B-1)
 *     blk[n*B + 1 + j] = min { v : s[r,v] = max_v' s[r,v'] },
 *     s[r,v] = bf16_round_nearest_even(float(base[r*ld_base+v]) + float(bias[r*ld_bias+v]))
 *
 * -0 and +0 compare equal; ties go to the lowest v.  Inputs must be finite.
 * d_base, d_bias: [rows, V] bf16 with row strides ld_base, ld_bias >= V.
 * d_blk: [N, B] int64, rows == N*(B-1), B >= 2, N >= 0 (N == 0 is a no-op).
 * V in [1, 2^30].  Workspace: xp_add_argmax_workspace_size(rows, V).
 * ---------------------------------------------------------------------- */
XP_API size_t xp_add_argmax_workspace_size(int64_t rows, int64_t V);
XP_API xp_status xp_add_argmax(const xp_bf16* d_base, int64_t ld_base, const xp_bf16* d_bias,
                        int64_t ld_bias, int64_t rows, int64_t V, int64_t* d_blk, int64_t N,
                        int64_t B, void* d_workspace, size_t workspace_bytes, xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_add_argmax_noalloc -- xp_add_argmax without a caller workspace.
 * The XPress pages have no counterpart of this call: it only changes where
 * the per-row scratch lives, not what is computed.  It is for callers that
 * cannot hand out device memory per call: a serving engine that has given
 * all free HBM to its KV-cache pool at start-up has nothing left to carve a
 * workspace from, and code that must not call cudaMalloc/cudaFree (which
 * synchronise the device and stall every other stream) cannot allocate one.
 *
 * Same arguments, result and errors as xp_add_argmax, minus the workspace.
 * The scratch (one 64-bit key and one counter per row) is a fixed array in
 * the library's device memory, sized for XP_ADD_ARGMAX_NOALLOC_MAX_ROWS rows;
 * rows above that return XP_ERR_SHAPE before anything is launched.  Each call
 * zeroes the part of the scratch it uses (cudaMemsetAsync on `stream`) and
 * then launches the add-argmax kernel; it calls no allocator.
 *
 * The first call on each device (with that device current) looks up the
 * scratch's device address, which may load the library's device code; make
 * that first call before any stream capture.  The address belongs to the
 * CUDA context it was looked up in: the cache is keyed by device and context
 * id, so after a device reset, or with another context of the device made
 * current, the next call looks it up again (that call is again a first call,
 * to be made outside capture).  Other calls only read the cached address.
 *
 * There is one scratch per device: calls that can overlap in time (on
 * different streams without ordering between them, or from several host
 * threads) race on it and corrupt each other's results.  Serialise them,
 * e.g. issue them all on one stream.
 * ---------------------------------------------------------------------- */
#define XP_ADD_ARGMAX_NOALLOC_MAX_ROWS 8192
XP_API xp_status xp_add_argmax_noalloc(const xp_bf16* d_base, int64_t ld_base, const xp_bf16* d_bias,
                                int64_t ld_bias, int64_t rows, int64_t V, int64_t* d_blk, int64_t N,
                                int64_t B, xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_topc_argmax -- the argmax over a slot's C gathered candidates, written
 * back as a vocab id.
 * Pages: fused_topc_argmax_to_blk / _xpress_topc_argmax_to_blk_kernel.
 *
 *   for r in [0, rows):  n = r / (B-1), j = r % (B-1)
 *     p* = min { p : s[r,p] = max_p' s[r,p'] },
 *     s[r,p] = bf16_round_nearest_even(float(base_c[r*C+p]) + float(bias_c[r*C+p]))
 *     blk[n*B + 1 + j] = cand[r*C + p*]
 *
 * d_base_c, d_bias_c: [rows, C] bf16, dense (2-byte aligned); d_cand:
 * [rows, C] int64 vocab ids; d_blk: [N, B] int64 with rows == N*(B-1).
 * C in [1, 2^30].  -0 and +0 compare equal; inputs must be finite.  No
 * workspace; one launch; nothing but blk[:, 1:] is written.
 * ---------------------------------------------------------------------- */
XP_API xp_status xp_topc_argmax(const xp_bf16* d_base_c, const xp_bf16* d_bias_c, const int64_t* d_cand,
                                int64_t rows, int64_t C, int64_t* d_blk, int64_t N, int64_t B,
                                xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_latent_pass -- the fused latent stage.
 * Pages: xpress_latent_pass / _xpress_latent_kernel (in-kernel MLP form).
 *
 *   prev[n,0] = am1[n], prev[n,b] = blk[n,b-1]            (b >= 1)
 *   x[n,b,:]  = float(hcache[n,b,:]) + E[prev[n,b],:] @ W_lat     (fp32 accumulate)
 *   u[n,b,r]  = sum_{j<=b} L[b,j,r] * x[n,j,r]
 *   ub = bf16(u);  g = ub @ Wg;  v = ub @ Wu;  m = bf16(g * sigmoid(g) * v)
 *   lat_out[n,b-1,:] = bf16(u[n,b,:] + m @ Wd)           (b = 1..B-1)
 *
 * d_blk [N,B] int64, d_am1 [N] int64, d_hcache [N,B,R] bf16, d_E [V,D] bf16,
 * d_W_lat [D,R] bf16, d_L [B,B,R] float32 (16-byte aligned like the bf16
 * pointers; entries above the diagonal are ignored), d_Wg/d_Wu [R,H] bf16,
 * d_Wd [H,R] bf16, d_lat_out [N,B-1,R] bf16.
 * All dense (no padding).  Constraints (else XP_ERR_SHAPE / XP_ERR_ALIGN):
 * 2 <= B <= 16; 16 <= R <= 512 with R a multiple of 16; D a multiple of 8 in
 * [8, 2^20]; H a multiple of 64 in [64, 2^16]; N*B <= 2^22; V <= 2^30.
 * Workspace: xp_latent_workspace_size(N,B,D,R,H).
 * ---------------------------------------------------------------------- */
XP_API size_t xp_latent_workspace_size(int64_t N, int64_t B, int64_t D, int64_t R, int64_t H);
XP_API xp_status xp_latent_pass(const int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache,
                         const xp_bf16* d_E, const xp_bf16* d_W_lat, const float* d_L,
                         const xp_bf16* d_Wg, const xp_bf16* d_Wu, const xp_bf16* d_Wd,
                         xp_bf16* d_lat_out, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R,
                         int64_t H, void* d_workspace, size_t workspace_bytes, xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_latent_pass_ex -- xp_latent_pass with the MLP schedule selectable.
 * Pages: xpress_latent_pass, argument do_mlp.
 *
 *   do_mlp = 1: the in-kernel MLP, exactly xp_latent_pass.
 *   do_mlp = 0: the GEMM schedule.  The kernel stops after the mixer and
 *     hands back ub = bf16(u); the caller's GEMMs then run on that bf16
 *     tensor, with [Wg | Wu] side by side as wgu_t:
 *       g = bf16(ub @ Wg);  v = bf16(ub @ Wu)                 (u @ wgu_t)
 *       m = bf16(g * sigmoid(g) * v)                           (silu_and_mul)
 *       lat_out[n,b-1,:] = bf16(float(ub) + m @ Wd)            (u.addmm_(m, wd_t))
 *     i.e. g and v are rounded before the SiLU and the residual is bf16(u).
 *   Here both schedules run in the same kernels (the roundings are applied
 *   in their epilogues); any other do_mlp value is XP_ERR_SHAPE.
 * Arguments, constraints and workspace as xp_latent_pass.
 * ---------------------------------------------------------------------- */
XP_API xp_status xp_latent_pass_ex(const int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache,
                                   const xp_bf16* d_E, const xp_bf16* d_W_lat, const float* d_L,
                                   const xp_bf16* d_Wg, const xp_bf16* d_Wu, const xp_bf16* d_Wd,
                                   xp_bf16* d_lat_out, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R,
                                   int64_t H, int32_t do_mlp, void* d_workspace, size_t workspace_bytes,
                                   xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_readout_argmax -- the readout matmul with the add + argmax fused into
 * its epilogue (the caller's `lat_out @ W2` followed by fused_add_argmax_to_blk,
 * without the bias or the logits ever reaching memory):
 *
 *   bias[r,v] = bf16(sum_k lat[r,k] * W2t[v,k])             (fp32 accumulate)
 *   s[r,v]    = bf16(float(base[r*ld_base+v]) + float(bias[r,v]))
 *   blk[n*B + 1 + j] = lowest argmax_v s[r,v]               r = n*(B-1)+j
 *
 * d_lat [rows,R] bf16 dense.  d_W2t: [V,R] bf16 dense -- the readout weight
 * W2 [R,V] of the pages stored TRANSPOSED (vocabulary-major; the layout of a
 * linear layer's weight), so one vocab tile's weights are contiguous.  d_base [rows,V] with
 * row stride ld_base.  R a multiple of 8 in [8, 512].  d_changed (nullable,
 * device int32): incremented by the number of slots whose token differs from
 * the value blk held before the call.  Workspace:
 * xp_readout_workspace_size(rows, V).
 * ---------------------------------------------------------------------- */
XP_API size_t xp_readout_workspace_size(int64_t rows, int64_t V);
XP_API xp_status xp_readout_argmax(const xp_bf16* d_lat, const xp_bf16* d_W2t, const xp_bf16* d_base,
                            int64_t ld_base, int64_t rows, int64_t V, int64_t R, int64_t* d_blk,
                            int64_t N, int64_t B, int32_t* d_changed, void* d_workspace,
                            size_t workspace_bytes, xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_jacobi_pass -- one whole pass: xp_latent_pass, then xp_readout_argmax on
 * its output (kept in the workspace), writing blk[:,1:] in place.  Repeated
 * calls iterate the Jacobi fixpoint: each pass reads the blk written by the
 * previous one (_xpress_add_argmax_reduce_to_blk_kernel docstring).
 * d_W2t: [V,R] bf16 dense -- the readout weight W2 [R,V] of the pages stored
 * TRANSPOSED (vocabulary-major), as in xp_readout_argmax.  d_changed as in
 * xp_readout_argmax.  Constraints: those of both stages.
 * Workspace: xp_jacobi_workspace_size(N,B,V,D,R,H).
 * ---------------------------------------------------------------------- */
XP_API size_t xp_jacobi_workspace_size(int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H);
XP_API xp_status xp_jacobi_pass(int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache,
                         const xp_bf16* d_E, const xp_bf16* d_W_lat, const float* d_L,
                         const xp_bf16* d_Wg, const xp_bf16* d_Wu, const xp_bf16* d_Wd,
                         const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base, int64_t N,
                         int64_t B, int64_t V, int64_t D, int64_t R, int64_t H,
                         int32_t* d_changed, void* d_workspace, size_t workspace_bytes,
                         xp_stream_t stream);

/* xp_jacobi_pass_ex -- xp_jacobi_pass with the latent stage's MLP schedule
 * selectable: do_mlp as in xp_latent_pass_ex (1 = xp_jacobi_pass).
 * d_W2t: [V,R], the readout weight transposed, as in xp_jacobi_pass. */
XP_API xp_status xp_jacobi_pass_ex(int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache,
                                   const xp_bf16* d_E, const xp_bf16* d_W_lat, const float* d_L,
                                   const xp_bf16* d_Wg, const xp_bf16* d_Wu, const xp_bf16* d_Wd,
                                   const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base, int64_t N,
                                   int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int32_t do_mlp,
                                   int32_t* d_changed, void* d_workspace, size_t workspace_bytes,
                                   xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_jacobi_fixpoint -- Jacobi passes to the fixpoint, without a host
 * round trip: up to max_passes passes of xp_jacobi_pass on blk in place,
 * stopping after the first pass that changes no slot of blk (that pass is
 * counted).  Each pass reads the blk the previous one wrote
 * (_xpress_add_argmax_reduce_to_blk_kernel docstring).
 *
 * On a stream that is not being captured, all max_passes passes are
 * enqueued at once (4 launches each, plus two small memsets); the kernels of
 * a pass enqueued after the fixpoint find the workspace's convergence flag
 * set and exit at their first instruction.  On a stream that is being
 * captured into a CUDA graph, the call adds the two memsets and one
 * conditional while node whose body is one pass (captured on a private
 * stream); the readout's last CTA sets the node's condition, so each launch
 * of the graph runs exactly the passes needed.  Both forms give the same
 * blk, *d_passes and *d_changed.
 * d_W2t: [V,R], the readout weight transposed, as in xp_jacobi_pass.
 * d_passes (device int32, required) receives the number of passes that ran;
 * d_changed (nullable, device int32) is incremented by the slots each pass
 * changed.  max_passes in [1, 1024].  Other arguments, constraints and the
 * workspace (xp_jacobi_workspace_size) as for xp_jacobi_pass.
 * ---------------------------------------------------------------------- */
XP_API xp_status xp_jacobi_fixpoint(int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache,
                                    const xp_bf16* d_E, const xp_bf16* d_W_lat, const float* d_L,
                                    const xp_bf16* d_Wg, const xp_bf16* d_Wu, const xp_bf16* d_Wd,
                                    const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base, int64_t N,
                                    int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int32_t max_passes,
                                    int32_t* d_passes, int32_t* d_changed, void* d_workspace,
                                    size_t workspace_bytes, xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_selftest_wait_timeout -- failure-detection self-test.  Enqueues one
 * small kernel that runs the library's bounded mbarrier wait on a barrier
 * nothing arrives on, with a limit of limit_us microseconds (1 .. 2,000,000)
 * instead of the kernels' 2 s.  The wait gives up, the kernel sets
 * XP_DEVERR_TIMEOUT in the workspace header and returns: xp_read_error()
 * then reports the bit, and the context stays usable.  No copy is in flight
 * and no memory besides the header is touched.  d_workspace: any workspace
 * of at least 256 bytes (256-byte aligned).
 * ---------------------------------------------------------------------- */
XP_API xp_status xp_selftest_wait_timeout(void* d_workspace, size_t workspace_bytes, uint32_t limit_us,
                                          xp_stream_t stream);

/* ------------------------------------------------------------------------
 * xp_read_error -- copy the workspace's device-side error bits (XP_DEVERR_*)
 * to *host_bits and clear them.  Synchronises `stream`; do not call it while
 * the stream is being captured into a CUDA graph.
 * ---------------------------------------------------------------------- */
XP_API xp_status xp_read_error(void* d_workspace, xp_stream_t stream, uint32_t* host_bits);

#ifdef __cplusplus
}
#endif
#endif /* XPRESS_H */
