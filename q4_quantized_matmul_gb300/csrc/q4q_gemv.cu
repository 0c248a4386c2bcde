// q4q_gemv.cu -- Q4_0 x Q8_0 matrix-vector product for 1..7 tokens (decode):
// the Q4_0 instantiations of the GEMV kernels of q4q_gemv.cuh, plus the generic
// path (any ne00 % 32 == 0, any alignment, any ne11) and the debug block sums of
// the GEMV's block-dot routine.
//
// ggml_mul_mat(Q4_0 src0 [ne00, ne01], F32 src1 [ne00, ne11]) as "llama.cpp
// 深度解读" §3 "量化矩阵乘法 — 核心算子" states it: src1 rows are quantized to
// Q8_0, and every output is sum_b fp32(d_w * d_x) * isum_b with isum_b the exact
// integer dot of one 32-element block (nibble - 8 times int8).
#include "q4q_gemv.cuh"

namespace q4q {
namespace {

// ------------------------------------------------------------ generic path --
// Any ne00 % 32 == 0, any ne11, src0 2-byte aligned: activations are first
// quantized to public Q8_0 blocks in the workspace, then one warp per output
// row reads blocks with 16-bit loads and forms the exact integer block sums.
__global__ void __launch_bounds__(PLAIN_THREADS)
generic_q4_0_q8_0_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ yq,
                         float* __restrict__ dst, int nb, int ne01, int ne11) {
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * PLAIN_THREADS) >> 5;
    for (int row = (blockIdx.x * PLAIN_THREADS + threadIdx.x) >> 5; row < ne01; row += warps) {
        const uint8_t* wr = w + (int64_t)row * nb * Q4_0_BYTES;
        for (int t = 0; t < ne11; ++t) {
            const uint8_t* yr = yq + (int64_t)t * nb * Q8_0_BYTES;
            float acc = 0.0f;
            for (int b = lane; b < nb; b += 32) {
                const uint16_t* wb = reinterpret_cast<const uint16_t*>(wr + b * Q4_0_BYTES);
                const uint16_t* yb = reinterpret_cast<const uint16_t*>(yr + b * Q8_0_BYTES);
                const float dw = fp16_to_f32(wb[0]);
                const float dx = fp16_to_f32(yb[0]);
                int isum = 0;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const uint32_t two = wb[1 + h];        // bytes 2h, 2h+1 of qs
                    const uint32_t ya = yb[1 + 2 * h];     // int8 elements 4h, 4h+1
                    const uint32_t yc = yb[2 + 2 * h];     // int8 elements 4h+2, 4h+3
                    const int n0 = (int)(two & 0xF) - 8, n1 = (int)((two >> 4) & 0xF) - 8;
                    const int n2 = (int)((two >> 8) & 0xF) - 8, n3 = (int)((two >> 12) & 0xF) - 8;
                    isum += n0 * (int)(int8_t)(ya & 0xff) + n1 * (int)(int8_t)(ya >> 8)
                          + n2 * (int)(int8_t)(yc & 0xff) + n3 * (int)(int8_t)(yc >> 8);
                }
                acc = fmaf(dw * dx, (float)isum, acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) dst[(int64_t)t * ne01 + row] = acc;
        }
    }
}

// ------------------------------------------------------------- debug path 0 --
// One thread per (token, row, block pair): the GEMV's unpack_pair / block_dot
// routines on words assembled with 16-bit loads (any 2-byte-aligned input).
__global__ void __launch_bounds__(PLAIN_THREADS)
debug_isums_gemv_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ yq,
                        int32_t* __restrict__ out, int nb, int ne01, int ne11) {
    const int np = nb / 2;
    const int64_t total = (int64_t)ne11 * ne01 * np;
    for (int64_t g = blockIdx.x * (int64_t)PLAIN_THREADS + threadIdx.x; g < total; g += (int64_t)gridDim.x * PLAIN_THREADS) {
        const int pr = (int)(g % np);
        const int64_t tr = g / np;
        const int row = (int)(tr % ne01);
        const int t = (int)(tr / ne01);
        const uint16_t* wh = reinterpret_cast<const uint16_t*>(w + ((int64_t)row * nb + 2 * pr) * Q4_0_BYTES);
        uint32_t wv[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) wv[i] = (uint32_t)wh[2 * i] | ((uint32_t)wh[2 * i + 1] << 16);
        const PairWeights pw = unpack_pair(wv);
        int isum[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint8_t* yb = yq + ((int64_t)t * nb + 2 * pr + h) * Q8_0_BYTES + 2;
            uint32_t e[4], o[4];
            int sq = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                e[i] = 0; o[i] = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int8_t qe = (int8_t)yb[8 * i + 2 * c], qo = (int8_t)yb[8 * i + 2 * c + 1];
                    sq += qe + qo;
                    e[i] |= (uint32_t)(uint8_t)qe << (8 * c);
                    o[i] |= (uint32_t)(uint8_t)qo << (8 * c);
                }
            }
            const uint4 ye = make_uint4(e[0], e[1], e[2], e[3]);
            const uint4 yo = make_uint4(o[0], o[1], o[2], o[3]);
            isum[h] = block_dot(h == 0 ? pw.qa : pw.qb, ye, yo) - 8 * sq;
        }
        int32_t* o = out + ((int64_t)t * ne01 + row) * nb + 2 * pr;
        o[0] = isum[0];
        o[1] = isum[1];
    }
}

}  // namespace

unsigned int gemv_take_device_status() { return take_gemv_status_word(); }

bool gemv_supported(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                    const DeviceInfo& info) {
    GemvPlan plan;
    return aligned(src0, 16) && aligned(src1, 16) && plan_gemv(ne00, ne01, ne11, info, &plan);
}

q4q_status gemv_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                        float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl, const KernelDebug* dbg) {
    GemvPlan plan;
    if (!plan_gemv(ne00, ne01, ne11, info, &plan)) return Q4Q_ERR_SHAPE;
    if (dbg) {
        plan.p.limit_ns = dbg->limit_ns;
        plan.p.fault = dbg->fault;
    }
    const GemvArgs a{static_cast<const uint8_t*>(src0), nullptr, src1, dst, nullptr, Q4Q_ACT_NONE, GemvGroup{}};
    return launch_gemv<WQ4_0, M_SINGLE>(plan, ne11, a, stream, info.device, pdl);
}

size_t generic_workspace_bytes(int64_t ne00, int64_t ne11) {
    return (size_t)(ne00 / QK) * (size_t)ne11 * Q8_0_BYTES;
}

q4q_status generic_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                           float* dst, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           const DeviceInfo& info) {
    if (workspace_bytes < generic_workspace_bytes(ne00, ne11)) return Q4Q_ERR_WORKSPACE;
    if (!workspace) return Q4Q_ERR_NULL;
    if (!aligned(workspace, 2)) return Q4Q_ERR_ALIGN;
    q4q_status st = launch_quantize(false, src1, workspace, ne00, ne11, stream, info);
    if (st != Q4Q_OK) return st;
    const int64_t warps_needed = ne01;
    const int grid = (int)std::min<int64_t>((warps_needed + 7) / 8, (int64_t)info.sm_count * 8);
    generic_q4_0_q8_0_kernel<<<grid, PLAIN_THREADS, 0, stream>>>(static_cast<const uint8_t*>(src0),
                                                           static_cast<const uint8_t*>(workspace), dst,
                                                           (int)(ne00 / QK), (int)ne01, (int)ne11);
    return launch_status();
}

q4q_status gemv_debug_isums(const void* src0, const void* src1_q8_0, int64_t ne00, int64_t ne01,
                            int64_t ne11, int32_t* out, cudaStream_t stream, const DeviceInfo& info) {
    if (ne00 % 64 != 0) return Q4Q_ERR_SHAPE;
    const int nb = (int)(ne00 / QK);
    const int64_t total = ne11 * ne01 * (nb / 2);
    if (total == 0) return Q4Q_OK;
    const int grid = (int)std::min<int64_t>((total + PLAIN_THREADS - 1) / PLAIN_THREADS, (int64_t)info.sm_count * 8);
    debug_isums_gemv_kernel<<<grid, PLAIN_THREADS, 0, stream>>>(static_cast<const uint8_t*>(src0),
                                                          static_cast<const uint8_t*>(src1_q8_0), out, nb,
                                                          (int)ne01, (int)ne11);
    return launch_status();
}

}  // namespace q4q
