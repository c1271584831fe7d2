// selftest.cu -- a check of the device-side timeout path (ssm_selftest_wait).
//
// One CTA initialises an mbarrier for one arrival and waits for its first phase
// with the library's bounded wait, here with the caller's time limit.  Without an
// arrival the wait gives up at the limit and the kernel records
// SSM_ERR_DEVICE_TIMEOUT in the workspace status words, exactly as a scan kernel
// whose TMA copies never completed would; with `arrive` set the same thread arrives
// first and the wait succeeds.  The kernel always returns: no trap, no fault.
#include "ssm_host.cuh"

namespace ssm {

constexpr unsigned int kSelftestWhere = 0xFFFFu;

__global__ void __launch_bounds__(32) selftest_wait_kernel(DeviceStatus* st,
                                                           unsigned long long limit_ns,
                                                           int arrive) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (arrive) mbar_arrive_expect_tx(&bar, 0);
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) record_timeout(st, kSelftestWhere);
  }
}

}  // namespace ssm

extern "C" {

ssm_status ssm_selftest_wait(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                             int arrive, ssm_stream_t stream) {
  using namespace ssm_host;
  if (!workspace || workspace_bytes < sizeof(ssm::DeviceStatus) || !aligned(workspace, 16))
    return SSM_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return SSM_ERR_INVALID_ARG;
  ssm::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<ssm::DeviceStatus*>(workspace), static_cast<unsigned long long>(limit_ns),
      arrive ? 1 : 0);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return SSM_OK;
}

}  // extern "C"
