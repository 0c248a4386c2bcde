// q4q_debug.cu -- test entry points that need no kernel of the hot path:
//  * the failure path of the bounded waits, driven on its own: one wait on an
//    mbarrier phase that nothing completes, with the same helper every kernel
//    uses, gives up after the caller's limit and records Q4Q_ERR_TIMEOUT;
//  * host-only views of the launch planning (the GEMV plan, the GEMM's split-K).
#include "q4q_gemv.cuh"

namespace q4q {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
        if (!mbar_wait_bounded(smem_u32(&bar), 0, limit_ns)) record_error(&g_gemv_status, DEV_TIMEOUT);
    }
}

}  // namespace

unsigned int debug_take_device_status() { return take_gemv_status_word(); }

q4q_status launch_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return launch_status();
}

q4q_status debug_gemv_plan(int64_t ne00, int64_t ne01, int64_t ne11, int block_bytes, int mats, int sm_count,
                           int smem_optin, int64_t* out) {
    DeviceInfo info{};
    info.sm_count = sm_count;
    info.max_smem_optin = smem_optin;
    info.cc_major = 10;
    GemvPlan plan;
    if (!plan_gemv(ne00, ne01, ne11, info, &plan, block_bytes, mats)) return Q4Q_ERR_SHAPE;
    const GemvParams& p = plan.p;
    const int64_t v[Q4Q_DEBUG_GEMV_PLAN_FIELDS] = {p.G, p.S, p.stage_bytes, (int64_t)plan.smem, plan.grid, plan.cl,
                                                   plan.lpr, plan.ppl_reg, p.n_units, p.act_off, p.stage_off,
                                                   p.half_off, p.row_bytes, p.dy_off, p.sy_off};
    for (int i = 0; i < Q4Q_DEBUG_GEMV_PLAN_FIELDS; ++i) out[i] = v[i];
    return Q4Q_OK;
}

int debug_mma_splits(int64_t ne00, int64_t ne01, int64_t ne11, int sm_count) {
    DeviceInfo info{};
    info.sm_count = sm_count;
    return mma_desired_splits(ne00, ne01, ne11, info);
}

}  // namespace q4q
