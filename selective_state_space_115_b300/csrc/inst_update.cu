// inst_update.cu -- instantiates the decode state-update dispatchers (every io
// type, dstate and input term).
#include "ssm_launch.cuh"

namespace ssm_host {
#define SSM_INST_UPDATE(T, N, E) \
  template ssm_status dispatch_update_n<T, N, E>(const ssm::UpdateParams&, bool, cudaStream_t);
SSM_INST_UPDATE(uint16_t, 4, false)
SSM_INST_UPDATE(uint16_t, 8, false)
SSM_INST_UPDATE(uint16_t, 16, false)
SSM_INST_UPDATE(uint16_t, 4, true)
SSM_INST_UPDATE(uint16_t, 8, true)
SSM_INST_UPDATE(uint16_t, 16, true)
SSM_INST_UPDATE(float, 4, false)
SSM_INST_UPDATE(float, 8, false)
SSM_INST_UPDATE(float, 16, false)
SSM_INST_UPDATE(float, 4, true)
SSM_INST_UPDATE(float, 8, true)
SSM_INST_UPDATE(float, 16, true)
#undef SSM_INST_UPDATE
}  // namespace ssm_host
