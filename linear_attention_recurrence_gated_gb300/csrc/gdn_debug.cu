// Self-test of the bounded waits and the status word (include/gdn_debug.h):
// one CTA waits on mbarriers that nothing completes, so the waits must give
// up and report instead of hanging.  No copy or tensor-memory allocation is
// in flight, so the CTA leaves cleanly.
#include "gdn_debug.h"
#include "gdn_tc_common.cuh"

namespace gdn {
namespace {

__global__ void __launch_bounds__(64) gdn_debug_wait_kernel(DeviceStatus *status) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars[0]), 1);
    ptx::mbar_init(ptx::smem_u32(&bars[1]), 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (lane == 0) {
    // whichever warp's limit passes first records the timeout and raises the
    // flag; the other leaves on seeing the flag (or at its own limit)
    const uint32_t bar = ptx::smem_u32(&bars[warp]);
    tc::role_wait_slow(bar, 0u, &abort_flag, status, 7, 3, 100u + warp);
  }
  __syncthreads();
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_debug_wait_timeout(void *workspace, size_t workspace_bytes,
                                             void *stream) {
  if (!workspace || workspace_bytes < gdn::kStatusBytes) return GDN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return GDN_ERR_INVALID_ARG;
  gdn::gdn_debug_wait_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(
      static_cast<gdn::DeviceStatus *>(workspace));
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
