// q4q_gemv_epi.cu -- the Q4_0 GEMV for 1..7 tokens with the bias / activation
// epilogue in its output write: a projection followed by its bias and GELU, as
// the GPT-2 graph of the "ggml GPT-2 117M inference walkthrough" runs them (§3.2,
// §3.5: ggml_add(ggml_repeat(b, cur), cur), then GELU after the MLP's first
// projection).  A separate instantiation, so that the plain kernel of q4q_gemv.cu
// carries no epilogue code.
#include "q4q_gemv.cuh"

namespace q4q {

unsigned int gemv_epi_take_device_status() { return take_gemv_status_word(); }

q4q_status gemv_mul_mat_epi(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                            float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl, const float* bias,
                            int act) {
    GemvPlan plan;
    if (!plan_gemv(ne00, ne01, ne11, info, &plan)) return Q4Q_ERR_SHAPE;
    const GemvArgs a{static_cast<const uint8_t*>(src0), nullptr, src1, dst, bias, act, GemvGroup{}};
    return launch_gemv<WQ4_0, M_EPI>(plan, ne11, a, stream, info.device, pdl);
}

}  // namespace q4q
