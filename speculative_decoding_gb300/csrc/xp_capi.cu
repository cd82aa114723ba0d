// xp_capi.cu -- the extern "C" entry points of libxpress.so: argument
// validation (before any launch), workspace checks, and dispatch to the
// launchers.  See include/xpress.h for the contract of each call.
#include <stdint.h>

#include <atomic>

#include "xp_common.cuh"
#include "xp_internal.h"

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned256(const void* p) { return ((uintptr_t)p & 255u) == 0; }

// The kernels are compiled for sm_103a only; refuse other devices up front
// rather than failing at launch.
xp_status check_device() {
  static std::atomic<int> cached[64];  // 0 unknown, 1 ok, 2 unsupported (any thread may fill it)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return XP_ERR_LAUNCH;
  if (dev < 0 || dev >= 64) return XP_ERR_UNSUPPORTED;
  int c = cached[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return XP_ERR_LAUNCH;
    c = (major == 10 && minor == 3) ? 1 : 2;
    cached[dev].store(c, std::memory_order_relaxed);
  }
  return c == 1 ? XP_OK : XP_ERR_UNSUPPORTED;
}

}  // namespace

extern "C" {

const char* xp_status_string(xp_status s) {
  switch (s) {
    case XP_OK: return "XP_OK";
    case XP_ERR_NULL: return "XP_ERR_NULL: a required pointer is NULL";
    case XP_ERR_SHAPE: return "XP_ERR_SHAPE: inconsistent or out-of-range sizes";
    case XP_ERR_ALIGN: return "XP_ERR_ALIGN: pointer or leading dimension misaligned";
    case XP_ERR_WORKSPACE: return "XP_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case XP_ERR_LAUNCH: return "XP_ERR_LAUNCH: a CUDA launch or driver call failed";
    case XP_ERR_UNSUPPORTED: return "XP_ERR_UNSUPPORTED: the current device is not sm_103 (GB300)";
    default: return "unknown xp_status";
  }
}

int32_t xp_version(void) { return 100; }

size_t xp_add_argmax_workspace_size(int64_t rows, int64_t V) {
  (void)V;
  if (rows < 0) return 0;
  return xp::argmax_ws_bytes(rows);
}

xp_status xp_add_argmax(const xp_bf16* d_base, int64_t ld_base, const xp_bf16* d_bias, int64_t ld_bias,
                        int64_t rows, int64_t V, int64_t* d_blk, int64_t N, int64_t B, void* d_workspace,
                        size_t workspace_bytes, xp_stream_t stream) {
  if (N < 0 || B < 2 || V < 1 || V > (int64_t(1) << 30) || rows != N * (B - 1)) return XP_ERR_SHAPE;
  if (ld_base < V || ld_bias < V) return XP_ERR_SHAPE;
  if (rows == 0) return XP_OK;
  if (!d_base || !d_bias || !d_blk || !d_workspace) return XP_ERR_NULL;
  if (!aligned16(d_base) || !aligned16(d_bias) || (ld_base & 7) || (ld_bias & 7) || ((uintptr_t)d_blk & 7))
    return XP_ERR_ALIGN;
  if (!aligned256(d_workspace) || workspace_bytes < xp::argmax_ws_bytes(rows)) return XP_ERR_WORKSPACE;
  xp_status st = check_device();
  if (st != XP_OK) return st;
  return xp::launch_add_argmax(d_base, ld_base, d_bias, ld_bias, rows, V, d_blk, B, d_workspace,
                               (cudaStream_t)stream);
}

xp_status xp_add_argmax_noalloc(const xp_bf16* d_base, int64_t ld_base, const xp_bf16* d_bias, int64_t ld_bias,
                                int64_t rows, int64_t V, int64_t* d_blk, int64_t N, int64_t B, xp_stream_t stream) {
  if (N < 0 || B < 2 || V < 1 || V > (int64_t(1) << 30) || rows != N * (B - 1)) return XP_ERR_SHAPE;
  if (ld_base < V || ld_bias < V || rows > XP_ADD_ARGMAX_NOALLOC_MAX_ROWS) return XP_ERR_SHAPE;
  if (rows == 0) return XP_OK;
  if (!d_base || !d_bias || !d_blk) return XP_ERR_NULL;
  if (!aligned16(d_base) || !aligned16(d_bias) || (ld_base & 7) || (ld_bias & 7) || ((uintptr_t)d_blk & 7))
    return XP_ERR_ALIGN;
  xp_status st = check_device();
  if (st != XP_OK) return st;
  return xp::launch_add_argmax_noalloc(d_base, ld_base, d_bias, ld_bias, rows, V, d_blk, B, (cudaStream_t)stream);
}

size_t xp_readout_workspace_size(int64_t rows, int64_t V) {
  (void)V;
  if (rows < 0) return 0;
  return xp::argmax_ws_bytes(rows);
}

xp_status xp_readout_argmax(const xp_bf16* d_lat, const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base,
                            int64_t rows, int64_t V, int64_t R, int64_t* d_blk, int64_t N, int64_t B,
                            int32_t* d_changed, void* d_workspace, size_t workspace_bytes, xp_stream_t stream) {
  if (N < 0 || B < 2 || V < 1 || V > (int64_t(1) << 30) || rows != N * (B - 1)) return XP_ERR_SHAPE;
  if (R < 8 || R > 512 || ld_base < V || rows > (int64_t(1) << 24)) return XP_ERR_SHAPE;
  if (rows == 0) return XP_OK;
  if (!d_lat || !d_W2t || !d_base || !d_blk || !d_workspace) return XP_ERR_NULL;
  if (!aligned16(d_lat) || !aligned16(d_W2t) || !aligned16(d_base) || (ld_base & 7) || (R & 7) ||
      ((uintptr_t)d_blk & 7) || ((uintptr_t)d_changed & 3))
    return XP_ERR_ALIGN;
  if (!aligned256(d_workspace) || workspace_bytes < xp::argmax_ws_bytes(rows)) return XP_ERR_WORKSPACE;
  xp_status st = check_device();
  if (st != XP_OK) return st;
  return xp::launch_readout_argmax(d_lat, d_W2t, d_base, ld_base, rows, V, R, d_blk, B, d_changed, d_workspace,
                                   (cudaStream_t)stream);
}

}  // extern "C"

namespace {

// Shape and alignment checks shared by the latent stage and the full pass.
xp_status check_latent_args(const int64_t* blk, const int64_t* am1, const xp_bf16* hcache, const xp_bf16* E,
                            const xp_bf16* W_lat, const float* L, const xp_bf16* Wg, const xp_bf16* Wu,
                            const xp_bf16* Wd, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H) {
  if (N < 0 || B < 2 || B > 16 || V < 1 || V > (int64_t(1) << 30)) return XP_ERR_SHAPE;
  if (D < 8 || D > (int64_t(1) << 20) || R < 16 || R > 512 || H < 64 || H > (int64_t(1) << 16)) return XP_ERR_SHAPE;
  if (N * B > (int64_t(1) << 22)) return XP_ERR_SHAPE;
  if (N == 0) return XP_OK;
  if (!blk || !am1 || !hcache || !E || !W_lat || !L || !Wg || !Wu || !Wd) return XP_ERR_NULL;
  if ((D & 7) || (R & 15) || (H & 63)) return XP_ERR_ALIGN;
  if (!aligned16(hcache) || !aligned16(E) || !aligned16(W_lat) || !aligned16(Wg) || !aligned16(Wu) ||
      !aligned16(Wd) || !aligned16(L) || ((uintptr_t)blk & 7) || ((uintptr_t)am1 & 7))
    return XP_ERR_ALIGN;
  return XP_OK;
}

// xp_jacobi_fixpoint on a stream that is being captured: one conditional
// while node whose body is one pass (the latent stage, then the readout in
// fixpoint mode, which sets the node's handle), so the graph runs exactly the
// passes the fixpoint needs.  The handle starts at 1 on every launch of the
// graph; the counters the body reads were zeroed on `s` before this call.
// The body is captured on a private stream in relaxed mode (the caller's
// capture may be global).
xp_status fixpoint_while_node(int64_t* blk, const int64_t* am1, const xp_bf16* hcache, const xp_bf16* E,
                              const xp_bf16* W_lat, const float* L, const xp_bf16* Wg, const xp_bf16* Wu,
                              const xp_bf16* Wd, uint16_t* lat, const xp_bf16* W2t, const xp_bf16* base,
                              int64_t ld_base, int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H,
                              int32_t max_passes, int32_t* passes, int32_t* changed, void* ws, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaGraph_t graph = nullptr;
  const cudaGraphNode_t* deps = nullptr;
  const cudaGraphEdgeData* edges = nullptr;
  size_t ndeps = 0;
  if (cudaStreamGetCaptureInfo(s, &cs, nullptr, &graph, &deps, &edges, &ndeps) != cudaSuccess ||
      cs != cudaStreamCaptureStatusActive)
    return XP_ERR_LAUNCH;
  cudaGraphConditionalHandle handle;
  if (cudaGraphConditionalHandleCreate(&handle, graph, 1, cudaGraphCondAssignDefault) != cudaSuccess)
    return XP_ERR_LAUNCH;
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = handle;
  np.conditional.type = cudaGraphCondTypeWhile;
  np.conditional.size = 1;
  cudaGraphNode_t node;
  if (cudaGraphAddNode(&node, graph, deps, edges, ndeps, &np) != cudaSuccess) return XP_ERR_LAUNCH;
  if (cudaStreamUpdateCaptureDependencies(s, &node, nullptr, 1, cudaStreamSetCaptureDependencies) != cudaSuccess)
    return XP_ERR_LAUNCH;
  cudaGraph_t body = np.conditional.phGraph_out[0];

  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) return XP_ERR_LAUNCH;
  xp_status st = XP_OK;
  cudaStream_t bs = nullptr;
  if (cudaStreamCreateWithFlags(&bs, cudaStreamNonBlocking) != cudaSuccess) {
    st = XP_ERR_LAUNCH;
  } else {
    if (cudaStreamBeginCaptureToGraph(bs, body, nullptr, nullptr, 0, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
      st = XP_ERR_LAUNCH;
    } else {
      st = xp::launch_latent(blk, am1, hcache, E, W_lat, L, Wg, Wu, Wd, lat, N, B, V, D, R, H, ws, bs);
      if (st == XP_OK)
        st = xp::launch_readout_argmax(lat, W2t, base, ld_base, N * (B - 1), V, R, blk, B, changed, ws, bs, nullptr,
                                       passes, (unsigned long long)handle, max_passes);
      cudaGraph_t out = nullptr;
      if (cudaStreamEndCapture(bs, &out) != cudaSuccess && st == XP_OK) st = XP_ERR_LAUNCH;
    }
    (void)cudaStreamDestroy(bs);
  }
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess && st == XP_OK) st = XP_ERR_LAUNCH;
  if (st != XP_OK) (void)cudaGetLastError();
  return st;
}

}  // namespace

extern "C" {

xp_status xp_topc_argmax(const xp_bf16* d_base_c, const xp_bf16* d_bias_c, const int64_t* d_cand, int64_t rows,
                         int64_t C, int64_t* d_blk, int64_t N, int64_t B, xp_stream_t stream) {
  if (N < 0 || B < 2 || C < 1 || C > (int64_t(1) << 30) || rows != N * (B - 1)) return XP_ERR_SHAPE;
  if (rows == 0) return XP_OK;
  if (!d_base_c || !d_bias_c || !d_cand || !d_blk) return XP_ERR_NULL;
  if (((uintptr_t)d_base_c & 1) || ((uintptr_t)d_bias_c & 1) || ((uintptr_t)d_cand & 7) || ((uintptr_t)d_blk & 7))
    return XP_ERR_ALIGN;
  xp_status st = check_device();
  if (st != XP_OK) return st;
  return xp::launch_topc_argmax(d_base_c, d_bias_c, d_cand, rows, C, d_blk, B, (cudaStream_t)stream);
}

size_t xp_latent_workspace_size(int64_t N, int64_t B, int64_t D, int64_t R, int64_t H) {
  if (N < 0 || B < 2 || D < 0 || R < 0 || H < 0) return 0;
  return xp::latent_ws_layout(N, B, D, R, H).total_latent;
}

xp_status xp_latent_pass(const int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache, const xp_bf16* d_E,
                         const xp_bf16* d_W_lat, const float* d_L, const xp_bf16* d_Wg, const xp_bf16* d_Wu,
                         const xp_bf16* d_Wd, xp_bf16* d_lat_out, int64_t N, int64_t B, int64_t V, int64_t D,
                         int64_t R, int64_t H, void* d_workspace, size_t workspace_bytes, xp_stream_t stream) {
  return xp_latent_pass_ex(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, d_lat_out, N, B, V, D, R, H,
                           1, d_workspace, workspace_bytes, stream);
}

xp_status xp_latent_pass_ex(const int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache,
                            const xp_bf16* d_E, const xp_bf16* d_W_lat, const float* d_L, const xp_bf16* d_Wg,
                            const xp_bf16* d_Wu, const xp_bf16* d_Wd, xp_bf16* d_lat_out, int64_t N, int64_t B,
                            int64_t V, int64_t D, int64_t R, int64_t H, int32_t do_mlp, void* d_workspace,
                            size_t workspace_bytes, xp_stream_t stream) {
  if (do_mlp != 0 && do_mlp != 1) return XP_ERR_SHAPE;
  xp_status st = check_latent_args(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, N, B, V, D, R, H);
  if (st != XP_OK || N == 0) return st;
  if (!d_lat_out || !d_workspace) return XP_ERR_NULL;
  if (!aligned16(d_lat_out)) return XP_ERR_ALIGN;
  if (!aligned256(d_workspace) || workspace_bytes < xp::latent_ws_layout(N, B, D, R, H).total_latent)
    return XP_ERR_WORKSPACE;
  st = check_device();
  if (st != XP_OK) return st;
  return xp::launch_latent(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, d_lat_out, N, B, V, D, R, H,
                           d_workspace, (cudaStream_t)stream, nullptr, do_mlp != 0);
}

size_t xp_jacobi_workspace_size(int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H) {
  (void)V;
  if (N < 0 || B < 2 || D < 0 || R < 0 || H < 0) return 0;
  return xp::latent_ws_layout(N, B, D, R, H).total_pass;
}

xp_status xp_jacobi_pass(int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache, const xp_bf16* d_E,
                         const xp_bf16* d_W_lat, const float* d_L, const xp_bf16* d_Wg, const xp_bf16* d_Wu,
                         const xp_bf16* d_Wd, const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base, int64_t N,
                         int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int32_t* d_changed,
                         void* d_workspace, size_t workspace_bytes, xp_stream_t stream) {
  return xp_jacobi_pass_ex(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, d_W2t, d_base, ld_base, N, B,
                           V, D, R, H, 1, d_changed, d_workspace, workspace_bytes, stream);
}

xp_status xp_jacobi_pass_ex(int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache, const xp_bf16* d_E,
                            const xp_bf16* d_W_lat, const float* d_L, const xp_bf16* d_Wg, const xp_bf16* d_Wu,
                            const xp_bf16* d_Wd, const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base,
                            int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int32_t do_mlp,
                            int32_t* d_changed, void* d_workspace, size_t workspace_bytes, xp_stream_t stream) {
  if (do_mlp != 0 && do_mlp != 1) return XP_ERR_SHAPE;
  xp_status st = check_latent_args(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, N, B, V, D, R, H);
  if (st != XP_OK || N == 0) return st;
  if (ld_base < V) return XP_ERR_SHAPE;
  if (!d_W2t || !d_base || !d_workspace) return XP_ERR_NULL;
  if (!aligned16(d_W2t) || !aligned16(d_base) || (ld_base & 7) || ((uintptr_t)d_changed & 3)) return XP_ERR_ALIGN;
  const xp::LatentWsLayout lay = xp::latent_ws_layout(N, B, D, R, H);
  if (!aligned256(d_workspace) || workspace_bytes < lay.total_pass) return XP_ERR_WORKSPACE;
  st = check_device();
  if (st != XP_OK) return st;
  uint16_t* lat = reinterpret_cast<uint16_t*>(static_cast<char*>(d_workspace) + lay.lat);
  st = xp::launch_latent(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, lat, N, B, V, D, R, H,
                         d_workspace, (cudaStream_t)stream, nullptr, do_mlp != 0);
  if (st != XP_OK) return st;
  return xp::launch_readout_argmax(lat, d_W2t, d_base, ld_base, N * (B - 1), V, R, d_blk, B, d_changed, d_workspace,
                                   (cudaStream_t)stream);
}

xp_status xp_jacobi_fixpoint(int64_t* d_blk, const int64_t* d_am1, const xp_bf16* d_hcache, const xp_bf16* d_E,
                             const xp_bf16* d_W_lat, const float* d_L, const xp_bf16* d_Wg, const xp_bf16* d_Wu,
                             const xp_bf16* d_Wd, const xp_bf16* d_W2t, const xp_bf16* d_base, int64_t ld_base,
                             int64_t N, int64_t B, int64_t V, int64_t D, int64_t R, int64_t H, int32_t max_passes,
                             int32_t* d_passes, int32_t* d_changed, void* d_workspace, size_t workspace_bytes,
                             xp_stream_t stream) {
  xp_status st = check_latent_args(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, N, B, V, D, R, H);
  if (st != XP_OK) return st;
  if (ld_base < V || max_passes < 1 || max_passes > 1024) return XP_ERR_SHAPE;
  if (!d_W2t || !d_base || !d_workspace || !d_passes) return XP_ERR_NULL;
  if (!aligned16(d_W2t) || !aligned16(d_base) || (ld_base & 7) || ((uintptr_t)d_changed & 3) ||
      ((uintptr_t)d_passes & 3))
    return XP_ERR_ALIGN;
  const xp::LatentWsLayout lay = xp::latent_ws_layout(N, B, D, R, H);
  if (!aligned256(d_workspace) || workspace_bytes < lay.total_pass) return XP_ERR_WORKSPACE;
  st = check_device();
  if (st != XP_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  xp::WsHeader* hdr = static_cast<xp::WsHeader*>(d_workspace);
  // converged = 0, passes = 0 (adjacent fields); then N == 0 runs no pass
  if (cudaMemsetAsync(&hdr->converged, 0, 2 * sizeof(unsigned int), s) != cudaSuccess ||
      cudaMemsetAsync(d_passes, 0, sizeof(int32_t), s) != cudaSuccess)
    return XP_ERR_LAUNCH;
  if (N == 0) return XP_OK;
  uint16_t* lat = reinterpret_cast<uint16_t*>(static_cast<char*>(d_workspace) + lay.lat);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return XP_ERR_LAUNCH;
  if (cs == cudaStreamCaptureStatusActive)
    return fixpoint_while_node(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, lat, d_W2t, d_base,
                               ld_base, N, B, V, D, R, H, max_passes, d_passes, d_changed, d_workspace, s);
  const uint32_t* skip = &hdr->converged;
  for (int32_t k = 0; k < max_passes; ++k) {
    st = xp::launch_latent(d_blk, d_am1, d_hcache, d_E, d_W_lat, d_L, d_Wg, d_Wu, d_Wd, lat, N, B, V, D, R, H,
                           d_workspace, s, skip);
    if (st != XP_OK) return st;
    st = xp::launch_readout_argmax(lat, d_W2t, d_base, ld_base, N * (B - 1), V, R, d_blk, B, d_changed, d_workspace,
                                   s, skip, d_passes);
    if (st != XP_OK) return st;
  }
  return XP_OK;
}

xp_status xp_selftest_wait_timeout(void* d_workspace, size_t workspace_bytes, uint32_t limit_us,
                                   xp_stream_t stream) {
  if (!d_workspace) return XP_ERR_NULL;
  if (!aligned256(d_workspace) || workspace_bytes < sizeof(xp::WsHeader)) return XP_ERR_WORKSPACE;
  if (limit_us < 1 || limit_us > 2000000u) return XP_ERR_SHAPE;
  xp_status st = check_device();
  if (st != XP_OK) return st;
  return xp::launch_wait_timeout_probe(d_workspace, 1000ull * limit_us, (cudaStream_t)stream);
}

xp_status xp_read_error(void* d_workspace, xp_stream_t stream, uint32_t* host_bits) {
  if (!d_workspace || !host_bits) return XP_ERR_NULL;
  if (!aligned256(d_workspace)) return XP_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned int bits = 0;
  if (cudaMemcpyAsync(&bits, d_workspace, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return XP_ERR_LAUNCH;
  if (cudaMemsetAsync(d_workspace, 0, sizeof(bits), s) != cudaSuccess) return XP_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return XP_ERR_LAUNCH;
  *host_bits = bits;
  return XP_OK;
}

}  // extern "C"
