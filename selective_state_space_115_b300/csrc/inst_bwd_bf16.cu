// inst_bwd_bf16.cu -- scan-gradient kernels for bf16 io.
#include "inst_bwd.cuh"

namespace ssm_host {
template ssm_status launch_scan_bwd<uint16_t>(const ssm::BwdParams&, int, bool, bool, bool, void*,
                                              void*, float*, float*, float*, cudaStream_t);
}  // namespace ssm_host
