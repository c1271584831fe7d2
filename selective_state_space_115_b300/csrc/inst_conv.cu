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

template <typename IO, int W>
static ssm_status conv_fwd_vec(const ssm::ConvParams& p0, cudaStream_t s) {
  constexpr int TB = 16 / static_cast<int>(sizeof(IO));
  // launches of whole rows with fewer than 2^31 vectors each (32-bit indexing)
  const int64_t vpr = p0.seqlen / TB;
  const int64_t rows_per_launch = (int64_t(INT32_MAX) - 128 * 4) / vpr;
  if (rows_per_launch < 1) return SSM_ERR_INVALID_ARG;
  ssm::ConvParams p = p0;
  p.div_vpr = ssm::FastDivU32::make(static_cast<uint32_t>(vpr));
  p.div_dim = ssm::FastDivU32::make(static_cast<uint32_t>(p0.dim));
  for (int64_t r0 = 0; r0 < p0.rows; r0 += rows_per_launch) {
    const int64_t n = (p0.rows - r0 < rows_per_launch) ? p0.rows - r0 : rows_per_launch;
    p.row0 = r0;
    p.rows = n;
    p.nvec = static_cast<uint32_t>(n * vpr);
    p.row0_mod = static_cast<uint32_t>(r0 % p0.dim);
    const int64_t grid = (static_cast<int64_t>(p.nvec) + 128 * 4 - 1) / (128 * 4);
    // programmatic stream serialisation: this launch overlaps the previous kernel's
    // last wave; the kernel waits for it before reading x
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, ssm::conv1d_fwd_vec_kernel<IO, W>, p);
    if (e != cudaSuccess) return cuda_fail(e, "conv1d_fwd launch");
  }
  return SSM_OK;
}

template <typename IO>
static ssm_status conv_fwd_vec_w(const ssm::ConvParams& p, cudaStream_t s) {
  switch (p.width) {
    case 1: return conv_fwd_vec<IO, 1>(p, s);
    case 2: return conv_fwd_vec<IO, 2>(p, s);
    case 3: return conv_fwd_vec<IO, 3>(p, s);
    case 4: return conv_fwd_vec<IO, 4>(p, s);
    case 5: return conv_fwd_vec<IO, 5>(p, s);
    case 6: return conv_fwd_vec<IO, 6>(p, s);
    case 7: return conv_fwd_vec<IO, 7>(p, s);
    case 8: return conv_fwd_vec<IO, 8>(p, s);
    default: return SSM_ERR_UNSUPPORTED;
  }
}

ssm_status launch_conv1d_fwd(bool bf16, const ssm::ConvParams& p, bool vec, cudaStream_t s) {
  if (bf16) return vec ? conv_fwd_vec_w<uint16_t>(p, s) : conv_fwd<uint16_t, false>(p, s);
  return vec ? conv_fwd_vec_w<float>(p, s) : conv_fwd<float, false>(p, s);
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
