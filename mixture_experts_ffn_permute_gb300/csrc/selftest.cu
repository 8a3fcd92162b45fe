// Self-test of the bounded waits every kernel of the library uses: one CTA
// waits on an mbarrier that nothing ever arrives on, through the same
// mbar_wait, so the wait runs out after the given limit, records
// MOE_ERR_DEVICE_TIMEOUT in the workspace status word and the kernel returns
// normally -- the device context stays usable.  No fault, trap or endless
// loop is involved.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_ffn.h"
#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint32_t* status, uint64_t limit_ns) {
  pdl_enter();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // nothing arrives: phase 0 never completes
    fence_mbarrier_init();
    mbar_wait(&bar, 0, status, limit_ns);
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_selftest_wait_timeout(void* ws, uint64_t limit_ns, void* stream) {
  if (!ws || limit_ns == 0 || limit_ns > moe::kWaitLimitNs) return MOE_ERR_INVALID_ARG;
  // the status word is the workspace's first field
  return moe::launch_kernel(moe::wait_timeout_kernel, dim3(1), dim3(32), 0,
                            static_cast<cudaStream_t>(stream), 1, static_cast<uint32_t*>(ws),
                            limit_ns) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
