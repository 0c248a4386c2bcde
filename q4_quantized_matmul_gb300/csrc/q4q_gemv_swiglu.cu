// q4q_gemv_swiglu.cu -- the Llama MLP's gate and up projections with the SwiGLU
// epilogue in one GEMV launch, for 1..7 tokens ("llama.cpp 深度解读" §4, Step I:
// up = ffn_up x, gate = ffn_gate x, cur = silu(gate) * up, SiLU(x) = x * sigmoid(x)).
//
// Both weight matrices have the same shape and share the activations, so one
// kernel streams a unit's rows of both into the same shared-memory stage, forms
// both dot products from one copy of the quantized activations, and writes only
// silu(gate) * up: the two projections' outputs never go through HBM.
#include "q4q_gemv.cuh"

namespace q4q {

unsigned int gemv_swiglu_take_device_status() { return take_gemv_status_word(); }

bool gemv_swiglu_supported(const void* gate, const void* up, int64_t ne00, int64_t ne01, const float* src1,
                           int64_t ne11, const DeviceInfo& info) {
    GemvPlan plan;
    return aligned(gate, 16) && aligned(up, 16) && aligned(src1, 16) &&
           plan_gemv(ne00, ne01, ne11, info, &plan, Q4_0_BYTES, 2);
}

q4q_status gemv_mul_mat_swiglu(const void* gate, const void* up, int64_t ne00, int64_t ne01, const float* src1,
                               int64_t ne11, float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl) {
    GemvPlan plan;
    if (!plan_gemv(ne00, ne01, ne11, info, &plan, Q4_0_BYTES, 2)) return Q4Q_ERR_SHAPE;
    const GemvArgs a{static_cast<const uint8_t*>(gate), static_cast<const uint8_t*>(up), src1, dst, nullptr,
                     Q4Q_ACT_NONE, GemvGroup{}};
    return launch_gemv<WQ4_0, M_DUAL>(plan, ne11, a, stream, info.device, pdl);
}

}  // namespace q4q
