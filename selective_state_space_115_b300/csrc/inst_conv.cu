// inst_conv.cu -- launches of the causal depthwise conv1d kernels (full sequence
// and decode step).
#include "ssm_host.cuh"

namespace ssm_host {

template <typename IO, bool VEC>
static ssm_status conv_fwd(const ssm::ConvParams& p0, cudaStream_t s) {
  constexpr int TB = 16 / static_cast<int>(sizeof(IO));
  constexpr int64_t kRowsPerLaunch = 65535;
  ssm::ConvParams p = p0;
  const unsigned gx = static_cast<unsigned>(((p.seqlen + TB - 1) / TB + 127) / 128);
  for (int64_t r0 = 0; r0 < p0.rows; r0 += kRowsPerLaunch) {
    p.row0 = r0;
    const int64_t n = (p0.rows - r0 < kRowsPerLaunch) ? p0.rows - r0 : kRowsPerLaunch;
    ssm::conv1d_fwd_kernel<IO, VEC><<<dim3(gx, static_cast<unsigned>(n)), 128, 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "conv1d_fwd launch");
  }
  return SSM_OK;
}

ssm_status launch_conv1d_fwd(bool bf16, const ssm::ConvParams& p, bool vec, cudaStream_t s) {
  if (bf16) return vec ? conv_fwd<uint16_t, true>(p, s) : conv_fwd<uint16_t, false>(p, s);
  return vec ? conv_fwd<float, true>(p, s) : conv_fwd<float, false>(p, s);
}

ssm_status launch_conv1d_update(bool bf16, const ssm::ConvParams& p, cudaStream_t s) {
  const int64_t grid = (p.rows + 255) / 256;
  if (grid > INT32_MAX) return SSM_ERR_INVALID_ARG;
  if (bf16)
    ssm::conv1d_update_kernel<uint16_t><<<static_cast<unsigned>(grid), 256, 0, s>>>(p);
  else
    ssm::conv1d_update_kernel<float><<<static_cast<unsigned>(grid), 256, 0, s>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "conv1d_update launch");
  return SSM_OK;
}

}  // namespace ssm_host
