// q4q_internal.h -- host-side helpers shared by the translation units of libq4q.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/q4q.h"

namespace q4q {

struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;    // bytes of dynamic shared memory a CTA may opt into
    int cc_major, cc_minor;
};

// Cached properties of the current device (queried once per device).
q4q_status current_device_info(DeviceInfo* info);

// Map the result of the last launch to a status (consumes cudaGetLastError).
q4q_status launch_status();

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Test-only knobs of one matmul launch (q4q_debug_mul_mat_timeout); the normal
// path passes none, which means every wait is bounded by WAIT_LIMIT_NS and no
// hand-off is left out.
struct KernelDebug {
    uint64_t limit_ns;   // bound of every wait of the launch
    int fault;           // 1: the first CTA leaves out one hand-off (its first stage)
};

// device status words of the translation units that wait on async copies
unsigned int gemv_take_device_status();
unsigned int mma_take_device_status();

// tensor-core path (q4q_mma.cu)
bool mma_supported(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info);
// the least workspace the tensor-core path runs in (no split-K), and the size that
// also holds the partial sums of the split-K it would pick for the shape
size_t mma_workspace_bytes(int64_t ne00, int64_t ne11);
size_t mma_workspace_bytes_split(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info);
// q8_weights: src0 holds Q8_0 blocks instead of Q4_0 ones
q4q_status mma_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                       float* dst, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                       const DeviceInfo& info, bool q8_weights = false, const KernelDebug* dbg = nullptr);
q4q_status mma_debug_isums(const void* src0, const void* src1_q8_0, int64_t ne00, int64_t ne01,
                           int64_t ne11, int32_t* out, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream, const DeviceInfo& info, bool q8_weights = false);

// GEMV path (q4q_gemv.cu)
bool gemv_supported(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                    const DeviceInfo& info);
q4q_status gemv_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                        float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl,
                        const KernelDebug* dbg = nullptr);

// the same GEMV with the bias / activation epilogue (q4q_gemv_epi.cu)
unsigned int gemv_epi_take_device_status();
q4q_status gemv_mul_mat_epi(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                            float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl, const float* bias,
                            int act);
size_t generic_workspace_bytes(int64_t ne00, int64_t ne11);
q4q_status generic_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                           float* dst, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           const DeviceInfo& info);
q4q_status gemv_debug_isums(const void* src0, const void* src1_q8_0, int64_t ne00, int64_t ne01,
                            int64_t ne11, int32_t* out, cudaStream_t stream, const DeviceInfo& info);

// dual-weight GEMV with the SwiGLU epilogue (q4q_gemv_swiglu.cu)
unsigned int gemv_swiglu_take_device_status();
bool gemv_swiglu_supported(const void* gate, const void* up, int64_t ne00, int64_t ne01, const float* src1,
                           int64_t ne11, const DeviceInfo& info);
q4q_status gemv_mul_mat_swiglu(const void* gate, const void* up, int64_t ne00, int64_t ne01, const float* src1,
                               int64_t ne11, float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl);

// Q8_0 weights (q4q_gemv_w8.cu)
unsigned int gemv_w8_take_device_status();
bool gemv_w8_supported(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                       const DeviceInfo& info);
q4q_status gemv_mul_mat_w8(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                           float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl);
q4q_status generic_mul_mat_w8(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                              float* dst, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                              const DeviceInfo& info);
q4q_status gemv_w8_debug_isums(const void* src0, const void* src1_q8_0, int64_t ne00, int64_t ne01, int64_t ne11,
                               int32_t* out, cudaStream_t stream, const DeviceInfo& info);

// several projections of one input in one launch (q4q_gemv_group.cu)
unsigned int gemv_group_take_device_status();
bool gemv_group_supported(int n, const void* const* src0, const int64_t* ne01, int64_t ne00, const float* src1,
                          int64_t ne11, const DeviceInfo& info);
q4q_status gemv_mul_mat_group(int n, const void* const* src0, const int64_t* ne01, int64_t ne00, const float* src1,
                              int64_t ne11, float* const* dst, cudaStream_t stream, const DeviceInfo& info,
                              bool pdl);

// A 2-D tiled tensor map (no swizzle, out-of-range elements read as zero), encoded by
// the driver entry point q4q_mma.cu looks up; false if it is missing or rejects the
// arguments.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1);

// few-token path: warp-level MMA on registers (q4q_rmma.cu)
unsigned int rmma_take_device_status();
bool rmma_supported(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info);
size_t rmma_min_workspace_bytes(int64_t ne00, int64_t ne01, int64_t ne11);
size_t rmma_workspace_bytes(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info);
// pdl: the activation kernel is launched with programmatic dependent launch behind
// the work before it on the stream (the caller's Q4Q_MUL_MAT_PDL)
q4q_status rmma_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11, float* dst,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream, const DeviceInfo& info,
                        bool pdl = false, const KernelDebug* dbg = nullptr);

// the GEMM's split-K count for a shape (q4q_mma.cu)
int mma_desired_splits(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info);

// test entry points (q4q_debug.cu): host-only views of the launch planning, and
// the bounded-wait failure path on its own (with its own device status word)
q4q_status debug_gemv_plan(int64_t ne00, int64_t ne01, int64_t ne11, int block_bytes, int mats, int sm_count,
                           int smem_optin, int64_t* out);
int debug_mma_splits(int64_t ne00, int64_t ne01, int64_t ne11, int sm_count);
q4q_status launch_wait_timeout(uint64_t limit_ns, cudaStream_t stream);
unsigned int debug_take_device_status();

// row gather (q4q_rows.cu)
unsigned int rows_take_device_status();

// chains of dependent one-token projections in one launch (q4q_chain.cu)
unsigned int chain_take_device_status();
size_t chain_workspace_bytes(int n);
q4q_status chain_check(const q4q_chain_link* links, int n);
q4q_status chain_launch(const q4q_chain_link* links, int n, void* workspace, cudaStream_t stream,
                        const DeviceInfo& info, const KernelDebug* dbg);

// Shape rules shared by every matmul entry point (q4q_api.cu).
q4q_status check_mul_mat_shapes(int64_t ne00, int64_t ne01, int64_t ne10, int64_t ne11);
// The least workspace q4q_mul_mat runs in for this shape (the tensor-core path then
// uses fewer K splits than q4q_mul_mat_workspace_size makes room for).
q4q_status mul_mat_min_workspace_bytes(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes);

// quantizers (q4q_quant.cu), also used by the GEMM / generic paths
q4q_status launch_quantize(bool q4, const float* src, void* dst, int64_t ncols, int64_t nrows,
                           cudaStream_t stream, const DeviceInfo& info);

}  // namespace q4q
