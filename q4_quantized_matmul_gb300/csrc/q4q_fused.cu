// q4q_fused.cu -- the operations next to the quantized matmul on the pages'
// decode graphs, and the Q8_0-weight matmul:
//  * bias add and GELU after a projection (the GPT-2 graph of the "ggml GPT-2
//    117M inference walkthrough", §3.2 and §3.5: ggml_add(ggml_repeat(b, cur),
//    cur), then GELU on the MLP's first projection) -- "matmul + bias +
//    activation", the fusion "llama.cpp 深度解读" §4 names as a graph benefit;
//  * the Llama MLP's SwiGLU, silu(ffn_gate x) * (ffn_up x) (same page, §4 Step I);
//  * ggml_mul_mat with Q8_0 weights (the Q8_0 type of that page's §2 table);
//  * several projections of one input (q, k, v) in one launch.
// For 1..7 tokens the epilogues run inside the GEMV (q4q_gemv*.cu); other paths
// run the matmul and then one elementwise kernel over its output.
#include <algorithm>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

constexpr int EW_THREADS = 256;

// y[t][r] = act(y[t][r] + bias[r]) in place (bias may be null).
__global__ void __launch_bounds__(EW_THREADS)
bias_act_kernel(float* __restrict__ y, const float* __restrict__ bias, int act, int64_t ne01, int64_t total) {
    for (int64_t i = blockIdx.x * (int64_t)EW_THREADS + threadIdx.x; i < total; i += (int64_t)gridDim.x * EW_THREADS) {
        float v = y[i];
        if (bias) v = __fadd_rn(v, __ldg(bias + i % ne01));
        if (act == Q4Q_ACT_GELU) v = gelu_f32(v);
        y[i] = v;
    }
}

// y[i] = silu(gate[i]) * y[i], with y holding the up projection.
__global__ void __launch_bounds__(EW_THREADS)
swiglu_kernel(const float* __restrict__ gate, float* __restrict__ y, int64_t total) {
    for (int64_t i = blockIdx.x * (int64_t)EW_THREADS + threadIdx.x; i < total; i += (int64_t)gridDim.x * EW_THREADS)
        y[i] = swiglu_f32(__ldg(gate + i), y[i]);
}

int ew_grid(int64_t total, const DeviceInfo& info) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((total + EW_THREADS - 1) / EW_THREADS, (int64_t)info.sm_count * 8));
}

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace
}  // namespace q4q

using namespace q4q;

extern "C" q4q_status q4q_mul_mat_bias_act(const void* src0, int64_t ne00, int64_t ne01,
                                           const float* src1, int64_t ne10, int64_t ne11,
                                           const float* bias, int act, float* dst,
                                           void* workspace, size_t workspace_bytes,
                                           unsigned int flags, q4q_stream_t stream_) {
    if (flags & ~Q4Q_MUL_MAT_PDL) return Q4Q_ERR_ARG;
    if (act != Q4Q_ACT_NONE && act != Q4Q_ACT_GELU) return Q4Q_ERR_ARG;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne10, ne11);
    if (st != Q4Q_OK) return st;
    if (ne01 == 0 || ne11 == 0) return Q4Q_OK;
    if (!src0 || !src1 || !dst) return Q4Q_ERR_NULL;
    if (!aligned(src0, 2) || !aligned(src1, 4) || !aligned(dst, 4) || (bias && !aligned(bias, 4)))
        return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (ne11 < 8 && gemv_supported(src0, ne00, ne01, src1, ne11, info))
        return gemv_mul_mat_epi(src0, ne00, ne01, src1, ne11, dst, stream, info, (flags & Q4Q_MUL_MAT_PDL) != 0,
                                bias, act);
    st = q4q_mul_mat_ex(src0, ne00, ne01, src1, ne10, ne11, dst, workspace, workspace_bytes, 0u, stream_);
    if (st != Q4Q_OK || (!bias && act == Q4Q_ACT_NONE)) return st;
    const int64_t total = ne01 * ne11;
    bias_act_kernel<<<ew_grid(total, info), EW_THREADS, 0, stream>>>(dst, bias, act, ne01, total);
    return launch_status();
}

extern "C" q4q_status q4q_mul_mat_swiglu_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes) {
    if (!bytes) return Q4Q_ERR_NULL;
    size_t mm = 0;
    q4q_status st = q4q_mul_mat_workspace_size(ne00, ne01, ne11, &mm);
    if (st != Q4Q_OK) return st;
    *bytes = round256(mm) + (size_t)ne01 * (size_t)ne11 * sizeof(float);
    return Q4Q_OK;
}

extern "C" q4q_status q4q_mul_mat_swiglu(const void* gate, const void* up, int64_t ne00, int64_t ne01,
                                         const float* src1, int64_t ne10, int64_t ne11, float* dst,
                                         void* workspace, size_t workspace_bytes, unsigned int flags,
                                         q4q_stream_t stream_) {
    if (flags & ~Q4Q_MUL_MAT_PDL) return Q4Q_ERR_ARG;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne10, ne11);
    if (st != Q4Q_OK) return st;
    if (ne01 == 0 || ne11 == 0) return Q4Q_OK;
    if (!gate || !up || !src1 || !dst) return Q4Q_ERR_NULL;
    if (!aligned(gate, 2) || !aligned(up, 2) || !aligned(src1, 4) || !aligned(dst, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (ne11 < 8 && gemv_swiglu_supported(gate, up, ne00, ne01, src1, ne11, info))
        return gemv_mul_mat_swiglu(gate, up, ne00, ne01, src1, ne11, dst, stream, info,
                                   (flags & Q4Q_MUL_MAT_PDL) != 0);
    // two matmuls (gate into the workspace, up into dst), then the elementwise SwiGLU
    size_t mm = 0, need = 0;
    if ((st = q4q_mul_mat_workspace_size(ne00, ne01, ne11, &mm)) != Q4Q_OK) return st;
    if ((st = q4q_mul_mat_swiglu_workspace_size(ne00, ne01, ne11, &need)) != Q4Q_OK) return st;
    if (workspace_bytes < need) return Q4Q_ERR_WORKSPACE;
    if (!workspace) return Q4Q_ERR_NULL;
    if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
    float* g = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + round256(mm));
    if ((st = q4q_mul_mat_ex(gate, ne00, ne01, src1, ne10, ne11, g, workspace, mm, 0u, stream_)) != Q4Q_OK) return st;
    if ((st = q4q_mul_mat_ex(up, ne00, ne01, src1, ne10, ne11, dst, workspace, mm, 0u, stream_)) != Q4Q_OK) return st;
    const int64_t total = ne01 * ne11;
    swiglu_kernel<<<ew_grid(total, info), EW_THREADS, 0, stream>>>(g, dst, total);
    return launch_status();
}

extern "C" q4q_status q4q_mul_mat_q8_0_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes) {
    if (!bytes) return Q4Q_ERR_NULL;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    size_t need = generic_workspace_bytes(ne00, ne11);
    if (ne11 >= 8) {
        DeviceInfo info;
        if ((st = current_device_info(&info)) != Q4Q_OK) return st;
        if (mma_supported(ne00, ne01, ne11, info)) need = std::max(need, mma_workspace_bytes_split(ne00, ne01, ne11, info));
    }
    *bytes = need;
    return Q4Q_OK;
}

extern "C" q4q_status q4q_mul_mat_q8_0(const void* src0, int64_t ne00, int64_t ne01,
                                       const float* src1, int64_t ne10, int64_t ne11,
                                       float* dst, void* workspace, size_t workspace_bytes,
                                       unsigned int flags, q4q_stream_t stream_) {
    if (flags & ~Q4Q_MUL_MAT_PDL) return Q4Q_ERR_ARG;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne10, ne11);
    if (st != Q4Q_OK) return st;
    if (ne01 == 0 || ne11 == 0) return Q4Q_OK;
    if (!src0 || !src1 || !dst) return Q4Q_ERR_NULL;
    if (!aligned(src0, 2) || !aligned(src1, 4) || !aligned(dst, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    const bool pdl = (flags & Q4Q_MUL_MAT_PDL) != 0;
    if (ne11 >= 8 && mma_supported(ne00, ne01, ne11, info) && aligned(src0, 16) && aligned(src1, 16)) {
        // the tensor-core GEMM with the Q8_0 dequantizer
        if (workspace_bytes < mma_workspace_bytes(ne00, ne11)) return Q4Q_ERR_WORKSPACE;
        if (!workspace) return Q4Q_ERR_NULL;
        if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
        return mma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info, true);
    }
    if (gemv_w8_supported(src0, ne00, ne01, src1, std::min<int64_t>(ne11, 7), info)) {
        // 1..7 tokens per launch; a batch the GEMM does not take runs in chunks of 7
        // tokens, each streaming the weights again
        for (int64_t t0 = 0; t0 < ne11; t0 += 7) {
            const int64_t nt = std::min<int64_t>(7, ne11 - t0);
            st = gemv_mul_mat_w8(src0, ne00, ne01, src1 + t0 * ne00, nt, dst + t0 * ne01, stream, info,
                                 pdl && t0 == 0);
            if (st != Q4Q_OK) return st;
        }
        return Q4Q_OK;
    }
    return generic_mul_mat_w8(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info);
}

extern "C" q4q_status q4q_debug_block_isums_q8_0(const void* src0_q8_0, const void* src1_q8_0, int64_t ne00,
                                                 int64_t ne01, int64_t ne11, int path, int32_t* out,
                                                 void* workspace, size_t workspace_bytes, q4q_stream_t stream_) {
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    if (path != 0 && path != 1) return Q4Q_ERR_ARG;
    if (ne01 == 0 || ne11 == 0) return Q4Q_OK;
    if (!src0_q8_0 || !src1_q8_0 || !out) return Q4Q_ERR_NULL;
    if (!aligned(src0_q8_0, 2) || !aligned(src1_q8_0, 2) || !aligned(out, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    if (path == 0) return gemv_w8_debug_isums(src0_q8_0, src1_q8_0, ne00, ne01, ne11, out, (cudaStream_t)stream_, info);
    return mma_debug_isums(src0_q8_0, src1_q8_0, ne00, ne01, ne11, out, workspace, workspace_bytes,
                           (cudaStream_t)stream_, info, true);
}

extern "C" q4q_status q4q_mul_mat_group_workspace_size(int n, const int64_t* ne01, int64_t ne00, int64_t ne11,
                                                       size_t* bytes) {
    if (!bytes || !ne01) return Q4Q_ERR_NULL;
    if (n < 1 || n > Q4Q_GROUP_MAX) return Q4Q_ERR_ARG;
    size_t need = 0;
    for (int m = 0; m < n; ++m) {
        size_t b = 0;
        q4q_status st = q4q_mul_mat_workspace_size(ne00, ne01[m], ne11, &b);
        if (st != Q4Q_OK) return st;
        need = std::max(need, b);
    }
    *bytes = need;
    return Q4Q_OK;
}

extern "C" q4q_status q4q_mul_mat_group(int n, const void* const* src0, const int64_t* ne01, int64_t ne00,
                                        const float* src1, int64_t ne10, int64_t ne11, float* const* dst,
                                        void* workspace, size_t workspace_bytes, unsigned int flags,
                                        q4q_stream_t stream_) {
    if (flags & ~Q4Q_MUL_MAT_PDL) return Q4Q_ERR_ARG;
    if (n < 1 || n > Q4Q_GROUP_MAX) return Q4Q_ERR_ARG;
    if (!src0 || !ne01 || !dst) return Q4Q_ERR_NULL;
    q4q_status st;
    // the non-empty matrices, in order
    const void* w[Q4Q_GROUP_MAX];
    int64_t rows[Q4Q_GROUP_MAX];
    float* out[Q4Q_GROUP_MAX];
    int k = 0;
    for (int m = 0; m < n; ++m) {
        if ((st = check_mul_mat_shapes(ne00, ne01[m], ne10, ne11)) != Q4Q_OK) return st;
        if (ne01[m] == 0 || ne11 == 0) continue;
        if (!src0[m] || !dst[m]) return Q4Q_ERR_NULL;
        if (!aligned(src0[m], 2) || !aligned(dst[m], 4)) return Q4Q_ERR_ALIGN;
        w[k] = src0[m];
        rows[k] = ne01[m];
        out[k] = dst[m];
        ++k;
    }
    if (k == 0) return Q4Q_OK;
    if (!src1) return Q4Q_ERR_NULL;
    if (!aligned(src1, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (ne11 < 8 && gemv_group_supported(k, w, rows, ne00, src1, ne11, info))
        return gemv_mul_mat_group(k, w, rows, ne00, src1, ne11, out, stream, info, (flags & Q4Q_MUL_MAT_PDL) != 0);
    for (int m = 0; m < k; ++m)
        if ((st = q4q_mul_mat_ex(w[m], ne00, rows[m], src1, ne10, ne11, out[m], workspace, workspace_bytes, flags,
                                 stream_)) != Q4Q_OK)
            return st;
    return Q4Q_OK;
}
