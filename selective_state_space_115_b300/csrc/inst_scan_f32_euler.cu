// inst_scan_f32_euler.cu -- instantiates the scan dispatchers for f32 io with the
// Euler input term (one translation unit per type so the kernels compile in
// parallel).
#include "ssm_launch.cuh"

namespace ssm_host {
template ssm_status dispatch_scan_n<float, 4, true>(const ScanCall&, ssm_algo, void*, cudaStream_t,
                                                  const SegPlan&, const MixPlan&);
template ssm_status dispatch_scan_n<float, 8, true>(const ScanCall&, ssm_algo, void*, cudaStream_t,
                                                  const SegPlan&, const MixPlan&);
template ssm_status dispatch_scan_n<float, 16, true>(const ScanCall&, ssm_algo, void*, cudaStream_t,
                                                   const SegPlan&, const MixPlan&);
}  // namespace ssm_host
