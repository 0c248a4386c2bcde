// q4q_api.cu -- host side of the C ABI: argument checks, path choice, status.
//
// ggml_mul_mat(Q4_0 src0 [ne00, ne01], F32 src1 [ne10, ne11]) -> F32 [ne01, ne11]
// ("llama.cpp 深度解读" §3 "量化矩阵乘法 — 核心算子").  Paths:
//   ne11 = 1, or 2..3 on matrices of at most 2^24 weights (prefer_gemv)
//                                                          -> fused GEMV (q4q_gemv.cu)
//   2 <= ne11 <= 32, ne00 % 256 == 0, 16-byte aligned src0/src1, and a workspace
//   of at least q4q_mul_mat_workspace_size's minimum        -> warp-MMA kernel (q4q_rmma.cu)
//   ne11 < 8, ne00 % 256 == 0, 16-byte aligned src0/src1  -> fused GEMV (q4q_gemv.cu)
//   ne11 >= 8 and the tensor-core GEMM accepts the shape    -> q4q_mma.cu
//   anything else                                           -> generic two-kernel path
#include <mutex>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {

namespace {
constexpr int MAX_DEVICES = 64;
std::mutex g_info_mutex;
DeviceInfo g_info[MAX_DEVICES];
bool g_info_valid[MAX_DEVICES] = {};
}  // namespace

q4q_status current_device_info(DeviceInfo* info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return Q4Q_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES) return Q4Q_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_info_mutex);
    if (!g_info_valid[dev]) {
        DeviceInfo d{};
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return Q4Q_ERR_CUDA;
        g_info[dev] = d;
        g_info_valid[dev] = true;
    }
    *info = g_info[dev];
    return Q4Q_OK;
}

q4q_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? Q4Q_OK : Q4Q_ERR_CUDA;
}

q4q_status check_mul_mat_shapes(int64_t ne00, int64_t ne01, int64_t ne10, int64_t ne11) {
    if (ne00 <= 0 || ne00 % QK != 0 || ne00 >= (1 << 20)) return Q4Q_ERR_SHAPE;
    if (ne10 != ne00) return Q4Q_ERR_SHAPE;
    if (ne01 < 0 || ne01 >= (1ll << 31) || ne11 < 0 || ne11 >= (1 << 20)) return Q4Q_ERR_SHAPE;
    return Q4Q_OK;
}

namespace {

// Token counts the warp-MMA kernel takes (timed against the GEMV below and the
// tensor-core GEMM above on the Llama-3-8B projection set).
constexpr int64_t RMMA_MIN_TOKENS = 2;
constexpr int64_t RMMA_MAX_TOKENS = 32;

// Below 8 tokens the GEMV, which needs no activation kernel and no split-K, beats the
// warp-MMA kernel's fixed cost on small matrices at 2 or 3 tokens, and nowhere else
// (chains of 8 calls with PDL in CUDA graphs, us per call, GEMV / warp-MMA:
// 4096 x 1024 at 2 / 3 / 4 / 5 / 7 tokens 3.8 / 4.6 / 5.9 / 6.0 / 8.2 against 5.7;
// 4096 x 4096 5.4 / 5.9 / 8.0 / 9.0 / 12.3 against 7.0; 4096 x 14336 at 2 tokens 12.1
// against 11.9; 14336 x 4096 14.0 against 13.4; 4096 x 128256 63.6 against 52.1).
bool prefer_gemv(int64_t ne00, int64_t ne01, int64_t ne11) {
    return ne11 < 2 || (ne11 <= 3 && ne00 * ne01 <= (1ll << 24));
}

bool use_rmma(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11, const DeviceInfo& info) {
    return ne11 >= RMMA_MIN_TOKENS && ne11 <= RMMA_MAX_TOKENS && rmma_supported(ne00, ne01, ne11, info) &&
           aligned(src0, 16) && aligned(src1, 16);
}

q4q_status workspace_bytes_of(int64_t ne00, int64_t ne01, int64_t ne11, bool with_splits, size_t* bytes) {
    if (!bytes) return Q4Q_ERR_NULL;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    size_t need = generic_workspace_bytes(ne00, ne11);
    // the device is looked at only for shapes a device-specific kernel could take
    if (ne11 >= 8 || (ne11 >= RMMA_MIN_TOKENS && ne00 % 256 == 0)) {
        DeviceInfo info;
        if ((st = current_device_info(&info)) != Q4Q_OK) return st;
        if (ne11 <= RMMA_MAX_TOKENS && !(ne11 < 8 && prefer_gemv(ne00, ne01, ne11)) &&
            rmma_supported(ne00, ne01, ne11, info))
            need = std::max(need, with_splits ? rmma_workspace_bytes(ne00, ne01, ne11, info)
                                              : rmma_min_workspace_bytes(ne00, ne01, ne11));
        if (ne11 >= 8 && mma_supported(ne00, ne01, ne11, info))
            need = std::max(need, with_splits ? mma_workspace_bytes_split(ne00, ne01, ne11, info)
                                              : mma_workspace_bytes(ne00, ne11));
    }
    *bytes = need;
    return Q4Q_OK;
}

}  // namespace

q4q_status mul_mat_min_workspace_bytes(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes) {
    return workspace_bytes_of(ne00, ne01, ne11, false, bytes);
}

}  // namespace q4q

using namespace q4q;

extern "C" q4q_status q4q_mul_mat_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes) {
    return workspace_bytes_of(ne00, ne01, ne11, true, bytes);
}

extern "C" q4q_status q4q_mul_mat(const void* src0, int64_t ne00, int64_t ne01,
                                  const float* src1, int64_t ne10, int64_t ne11,
                                  float* dst, void* workspace, size_t workspace_bytes,
                                  q4q_stream_t stream_) {
    return q4q_mul_mat_ex(src0, ne00, ne01, src1, ne10, ne11, dst, workspace, workspace_bytes, 0u, stream_);
}

extern "C" q4q_status q4q_mul_mat_ex(const void* src0, int64_t ne00, int64_t ne01,
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
    const bool gemv_ok = ne11 < 8 && gemv_supported(src0, ne00, ne01, src1, ne11, info);
    if (gemv_ok && prefer_gemv(ne00, ne01, ne11))
        return gemv_mul_mat(src0, ne00, ne01, src1, ne11, dst, stream, info, pdl);
    if (use_rmma(src0, ne00, ne01, src1, ne11, info) && workspace && aligned(workspace, 256) &&
        workspace_bytes >= rmma_min_workspace_bytes(ne00, ne01, ne11))
        return rmma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info, pdl);
    if (gemv_ok) return gemv_mul_mat(src0, ne00, ne01, src1, ne11, dst, stream, info, pdl);
    if (ne11 >= 8 && mma_supported(ne00, ne01, ne11, info) && aligned(src0, 16) && aligned(src1, 16)) {
        if (workspace_bytes < mma_workspace_bytes(ne00, ne11)) return Q4Q_ERR_WORKSPACE;
        if (!workspace) return Q4Q_ERR_NULL;
        if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
        return mma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info);
    }
    return generic_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info);
}

extern "C" q4q_status q4q_debug_workspace_size(int64_t ne00, int64_t ne11, int path, size_t* bytes) {
    if (!bytes) return Q4Q_ERR_NULL;
    if (ne00 <= 0 || ne00 % QK != 0 || ne00 >= (1 << 20) || ne11 < 0 || ne11 >= (1 << 20)) return Q4Q_ERR_SHAPE;
    if (path != 0 && path != 1) return Q4Q_ERR_ARG;
    *bytes = path == 0 ? 0 : mma_workspace_bytes(ne00, ne11);
    return Q4Q_OK;
}

extern "C" q4q_status q4q_debug_block_isums(const void* src0, const void* src1_q8_0,
                                            int64_t ne00, int64_t ne01, int64_t ne11, int path,
                                            int32_t* out, void* workspace, size_t workspace_bytes,
                                            q4q_stream_t stream_) {
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    if (path != 0 && path != 1) return Q4Q_ERR_ARG;
    if (ne01 == 0 || ne11 == 0) return Q4Q_OK;
    if (!src0 || !src1_q8_0 || !out) return Q4Q_ERR_NULL;
    if (!aligned(src0, 2) || !aligned(src1_q8_0, 2) || !aligned(out, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (path == 0) return gemv_debug_isums(src0, src1_q8_0, ne00, ne01, ne11, out, stream, info);
    return mma_debug_isums(src0, src1_q8_0, ne00, ne01, ne11, out, workspace, workspace_bytes, stream, info);
}

extern "C" q4q_status q4q_debug_gemv_plan(int64_t ne00, int64_t ne01, int64_t ne11, int weight_block_bytes,
                                          int mats, int sm_count, int smem_optin, int64_t* out) {
    if (!out) return Q4Q_ERR_NULL;
    if (weight_block_bytes != Q4Q_BLOCK_Q4_0_BYTES && weight_block_bytes != Q4Q_BLOCK_Q8_0_BYTES) return Q4Q_ERR_ARG;
    if (mats != 1 && mats != 2) return Q4Q_ERR_ARG;
    if (sm_count <= 0 || smem_optin <= 0) return Q4Q_ERR_ARG;
    return debug_gemv_plan(ne00, ne01, ne11, weight_block_bytes, mats, sm_count, smem_optin, out);
}

extern "C" q4q_status q4q_debug_mma_splits(int64_t ne00, int64_t ne01, int64_t ne11, int sm_count, int* splits) {
    if (!splits) return Q4Q_ERR_NULL;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    if (sm_count <= 0 || ne00 % 256 != 0 || ne11 < 8 || ne01 == 0) return Q4Q_ERR_ARG;
    *splits = debug_mma_splits(ne00, ne01, ne11, sm_count);
    return Q4Q_OK;
}

extern "C" q4q_status q4q_debug_wait_timeout(uint64_t limit_ns, q4q_stream_t stream) {
    if (limit_ns == 0 || limit_ns > WAIT_LIMIT_NS) return Q4Q_ERR_ARG;
    return launch_wait_timeout(limit_ns, (cudaStream_t)stream);
}

extern "C" q4q_status q4q_debug_mul_mat_timeout(const void* src0, int64_t ne00, int64_t ne01, const float* src1,
                                                int64_t ne11, float* dst, void* workspace, size_t workspace_bytes,
                                                int path, uint64_t limit_ns, q4q_stream_t stream_) {
    if (path < 0 || path > 3) return Q4Q_ERR_ARG;
    if (limit_ns == 0 || limit_ns > WAIT_LIMIT_NS) return Q4Q_ERR_ARG;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    if (ne01 == 0 || ne11 == 0) return Q4Q_ERR_SHAPE;
    if (!src0 || !src1 || !dst) return Q4Q_ERR_NULL;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    const KernelDebug dbg{limit_ns, 1};
    if (path == 0) {
        if (ne11 >= 8 || !gemv_supported(src0, ne00, ne01, src1, ne11, info)) return Q4Q_ERR_SHAPE;
        return gemv_mul_mat(src0, ne00, ne01, src1, ne11, dst, stream, info, false, &dbg);
    }
    if (path == 2) {
        // a two-link chain of this matrix on the same input (link 1 rewrites dst)
        if (ne11 != 1) return Q4Q_ERR_SHAPE;
        const q4q_chain_link links[2] = {{src0, ne00, ne01, src1, dst}, {src0, ne00, ne01, src1, dst}};
        if ((st = chain_check(links, 2)) != Q4Q_OK) return st;
        if (workspace_bytes < chain_workspace_bytes(2)) return Q4Q_ERR_WORKSPACE;
        if (!workspace) return Q4Q_ERR_NULL;
        if (!aligned(workspace, 4)) return Q4Q_ERR_ALIGN;
        return chain_launch(links, 2, workspace, stream, info, &dbg);
    }
    if (path == 3) {
        if (!rmma_supported(ne00, ne01, ne11, info) || !aligned(src0, 16) || !aligned(src1, 16))
            return Q4Q_ERR_SHAPE;
        if (workspace_bytes < rmma_min_workspace_bytes(ne00, ne01, ne11)) return Q4Q_ERR_WORKSPACE;
        if (!workspace) return Q4Q_ERR_NULL;
        if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
        return rmma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info, false,
                            &dbg);
    }
    if (ne11 < 8 || !mma_supported(ne00, ne01, ne11, info) || !aligned(src0, 16) || !aligned(src1, 16))
        return Q4Q_ERR_SHAPE;
    if (workspace_bytes < mma_workspace_bytes(ne00, ne11)) return Q4Q_ERR_WORKSPACE;
    if (!workspace) return Q4Q_ERR_NULL;
    if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
    return mma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info, false, &dbg);
}

extern "C" q4q_status q4q_debug_mul_mat_path(const void* src0, int64_t ne00, int64_t ne01, const float* src1,
                                             int64_t ne11, float* dst, void* workspace, size_t workspace_bytes,
                                             int path, q4q_stream_t stream_) {
    if (path != 0 && path != 1 && path != 3) return Q4Q_ERR_ARG;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    if (ne01 == 0 || ne11 == 0) return Q4Q_ERR_SHAPE;
    if (!src0 || !src1 || !dst) return Q4Q_ERR_NULL;
    if (!aligned(src0, 16) || !aligned(src1, 16) || !aligned(dst, 4)) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    cudaStream_t stream = (cudaStream_t)stream_;
    if (path == 0) {
        if (ne11 >= 8 || !gemv_supported(src0, ne00, ne01, src1, ne11, info)) return Q4Q_ERR_SHAPE;
        return gemv_mul_mat(src0, ne00, ne01, src1, ne11, dst, stream, info, false);
    }
    const bool ok = path == 1 ? (ne11 >= 8 && mma_supported(ne00, ne01, ne11, info))
                              : rmma_supported(ne00, ne01, ne11, info);
    if (!ok) return Q4Q_ERR_SHAPE;
    if (workspace_bytes < (path == 1 ? mma_workspace_bytes(ne00, ne11) : rmma_min_workspace_bytes(ne00, ne01, ne11)))
        return Q4Q_ERR_WORKSPACE;
    if (!workspace) return Q4Q_ERR_NULL;
    if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
    if (path == 1) return mma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info);
    return rmma_mul_mat(src0, ne00, ne01, src1, ne11, dst, workspace, workspace_bytes, stream, info);
}

extern "C" q4q_status q4q_debug_mul_mat_path_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, int path,
                                                            size_t* bytes) {
    if (!bytes) return Q4Q_ERR_NULL;
    if (path != 0 && path != 1 && path != 3) return Q4Q_ERR_ARG;
    q4q_status st = check_mul_mat_shapes(ne00, ne01, ne00, ne11);
    if (st != Q4Q_OK) return st;
    if (path == 0) {
        *bytes = 0;
        return Q4Q_OK;
    }
    DeviceInfo info;
    if ((st = current_device_info(&info)) != Q4Q_OK) return st;
    *bytes = path == 1 ? mma_workspace_bytes_split(ne00, ne01, ne11, info) : rmma_workspace_bytes(ne00, ne01, ne11, info);
    return Q4Q_OK;
}

extern "C" q4q_status q4q_device_status(q4q_status* status) {
    if (!status) return Q4Q_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return Q4Q_ERR_CUDA;
    // every translation unit that records device errors has its own word: read
    // and clear all of them, report the first one set
    const unsigned int words[] = {gemv_take_device_status(), mma_take_device_status(),
                                  gemv_swiglu_take_device_status(), gemv_w8_take_device_status(),
                                  gemv_group_take_device_status(), gemv_epi_take_device_status(),
                                  rows_take_device_status(), debug_take_device_status(),
                                  chain_take_device_status(), rmma_take_device_status()};
    unsigned int first = 0;
    for (unsigned int w : words)
        if (!first) first = w;
    *status = (q4q_status)first;
    return Q4Q_OK;
}

extern "C" const char* q4q_status_string(q4q_status s) {
    switch (s) {
        case Q4Q_OK: return "ok";
        case Q4Q_ERR_NULL: return "null pointer";
        case Q4Q_ERR_SHAPE: return "invalid shape";
        case Q4Q_ERR_ALIGN: return "misaligned pointer";
        case Q4Q_ERR_WORKSPACE: return "workspace too small";
        case Q4Q_ERR_CUDA: return "CUDA error";
        case Q4Q_ERR_TIMEOUT: return "device wait timed out";
        case Q4Q_ERR_ARG: return "invalid argument";
    }
    return "unknown status";
}

extern "C" int q4q_version(void) { return (1 << 16) | 1; }
