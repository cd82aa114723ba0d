// xp_selftest.cu -- the failure-detection self-test: one bounded mbarrier
// wait that runs out.
//
// Every wait in the kernels is bounded: when its wall-clock limit passes, the
// kernel sets XP_DEVERR_TIMEOUT in the workspace header and returns instead
// of hanging.  This kernel runs that same wait (mbar_wait_for) on a barrier
// nothing arrives on, with a short limit and no copy in flight, so a test can
// check on the GPU that the wait gives up, the error bit reaches the host,
// and the context stays usable.
#include "xp_common.cuh"
#include "xp_internal.h"
#include "xp_ptx.cuh"

namespace xp {

__global__ void wait_timeout_probe_kernel(WsHeader* hdr, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  // phase 0 never completes: nothing arrives on the barrier
  if (!mbar_wait_for(&bar, 0, limit_ns)) flag_error(hdr, XP_DEVERR_TIMEOUT);
}

xp_status launch_wait_timeout_probe(void* ws, unsigned long long limit_ns, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(static_cast<WsHeader*>(ws), limit_ns);
  return cudaGetLastError() == cudaSuccess ? XP_OK : XP_ERR_LAUNCH;
}

}  // namespace xp
