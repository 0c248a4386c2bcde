// q4q_gemv_group.cu -- several Q4_0 projections of one input in one GEMV launch,
// for 1..7 tokens: the q, k and v projections of a layer (the separate wq / wk /
// wv weights that llm_build_mul_mat_qkv takes when a model has no fused wqkv,
// "llama.cpp 深度解读" §3.2 of the Gemma3 graph page; the fused wqkv is the
// same thing with the rows concatenated in one tensor).
//
// One plan covers the rows of all matrices; units never straddle two matrices,
// so each unit is still one contiguous byte range of one weight tensor.  The
// activations are quantized once per CTA for all of them, and each launch gap
// between the projections disappears.
#include "q4q_gemv.cuh"

namespace q4q {
namespace {

bool plan_gemv_group(int n, const int64_t* ne01, int64_t ne00, int64_t ne11, const DeviceInfo& info,
                     GemvPlan* plan, GemvGroup* grp) {
    if (n < 1 || n > GROUP_MAX) return false;
    int64_t total = 0;
    for (int m = 0; m < n; ++m) {
        if (ne01[m] <= 0) return false;
        total += ne01[m];
    }
    if (total >= (1ll << 31) || !plan_gemv(ne00, total, ne11, info, plan)) return false;
    const int64_t G = plan->p.G;
    int64_t units = 0;
    *grp = GemvGroup{};
    grp->n = n;
    for (int m = 0; m < n; ++m) {
        grp->unit0[m] = (int)units;
        grp->rows[m] = (int)ne01[m];
        units += (ne01[m] + G - 1) / G;
    }
    for (int m = n; m <= GROUP_MAX; ++m) grp->unit0[m] = (int)units;
    plan->p.n_units = (int)units;
    plan->grid = (int)std::min<int64_t>(units, plan->grid_cap);
    return true;
}

}  // namespace

unsigned int gemv_group_take_device_status() { return take_gemv_status_word(); }

bool gemv_group_supported(int n, const void* const* src0, const int64_t* ne01, int64_t ne00, const float* src1,
                          int64_t ne11, const DeviceInfo& info) {
    for (int m = 0; m < n; ++m)
        if (!aligned(src0[m], 16)) return false;
    GemvPlan plan;
    GemvGroup grp;
    return aligned(src1, 16) && plan_gemv_group(n, ne01, ne00, ne11, info, &plan, &grp);
}

q4q_status gemv_mul_mat_group(int n, const void* const* src0, const int64_t* ne01, int64_t ne00, const float* src1,
                              int64_t ne11, float* const* dst, cudaStream_t stream, const DeviceInfo& info,
                              bool pdl) {
    GemvPlan plan;
    GemvArgs a{nullptr, nullptr, src1, nullptr, nullptr, Q4Q_ACT_NONE, GemvGroup{}};
    if (!plan_gemv_group(n, ne01, ne00, ne11, info, &plan, &a.grp)) return Q4Q_ERR_SHAPE;
    for (int m = 0; m < n; ++m) {
        a.grp.w[m] = static_cast<const uint8_t*>(src0[m]);
        a.grp.dst[m] = dst[m];
    }
    return launch_gemv<WQ4_0, M_GROUP>(plan, ne11, a, stream, info.device, pdl);
}

}  // namespace q4q
