// Self-test of the bounded pipeline wait that every kernel of the library uses.
//
// Each pipeline wait of the attention, decode and gather kernels is an mbarrier try_wait loop
// with a time limit (2 s): when the limit passes, the kernel sets the timeout bit of the
// workspace status word and returns instead of hanging, and irm_device_status() reports
// IRM_ERR_DEVICE_TIMEOUT.  This entry point launches one warp that waits, through the same
// helper, on a barrier nothing ever arrives on, so tests can exercise that path on purpose:
// the wait gives up by itself, the status is set, and the context stays usable.
#include <cuda_runtime.h>
#include <cstdint>

#include "irm_common.cuh"

namespace irm {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) mbar_init(smem_u32(&bar), 1);
  __syncthreads();
  // no thread ever arrives: every lane's bounded wait must give up after its time limit
  const bool ok = mbar_wait(smem_u32(&bar), 0, nullptr);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) set_status(status, kDevErrTimeout);
}

}  // namespace
}  // namespace irm

extern "C" irm_status irm_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                                cudaStream_t stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < IRM_WORKSPACE_HEADER)
    return IRM_ERR_WORKSPACE;
  irm::wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(static_cast<int*>(workspace));
  return cudaGetLastError() == cudaSuccess ? IRM_OK : IRM_ERR_CUDA;
}
