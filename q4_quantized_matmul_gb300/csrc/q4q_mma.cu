// q4q_mma.cu -- tensor-core path for ne11 >= 8 (placeholder until the tcgen05 kernel lands).
#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {

unsigned int mma_take_device_status() { return 0; }
bool mma_supported(int64_t, int64_t, int64_t, const DeviceInfo&) { return false; }
size_t mma_workspace_bytes(int64_t, int64_t) { return 0; }
q4q_status mma_mul_mat(const void*, int64_t, int64_t, const float*, int64_t, float*, void*, size_t,
                       cudaStream_t, const DeviceInfo&) { return Q4Q_ERR_ARG; }
q4q_status mma_debug_isums(const void*, const void*, int64_t, int64_t, int64_t, int32_t*, cudaStream_t,
                           const DeviceInfo&) { return Q4Q_ERR_ARG; }

}  // namespace q4q
