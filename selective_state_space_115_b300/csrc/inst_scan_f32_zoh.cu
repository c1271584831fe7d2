// inst_scan_f32_zoh.cu -- instantiates the scan dispatchers for f32 io with the
// zero-order-hold input term (one translation unit per type so the kernels compile in
// parallel).
#include "ssm_launch.cuh"

namespace ssm_host {
template ssm_status dispatch_scan_n<float, 4, false>(const ScanCall&, ssm_algo, void*, cudaStream_t,
                                                  const SegPlan&, const MixPlan&);
template ssm_status dispatch_scan_n<float, 8, false>(const ScanCall&, ssm_algo, void*, cudaStream_t,
                                                  const SegPlan&, const MixPlan&);
template ssm_status dispatch_scan_n<float, 16, false>(const ScanCall&, ssm_algo, void*, cudaStream_t,
                                                   const SegPlan&, const MixPlan&);
}  // namespace ssm_host
