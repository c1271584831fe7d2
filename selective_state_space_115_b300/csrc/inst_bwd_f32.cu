// inst_bwd_f32.cu -- scan-gradient kernels for fp32 io.
#include "inst_bwd.cuh"

namespace ssm_host {
template ssm_status launch_scan_bwd<float>(const ssm::BwdParams&, int, bool, bool, bool, void*,
                                           void*, float*, float*, float*, cudaStream_t);
}  // namespace ssm_host
