// q4q_rows.cu -- ggml_get_rows on a quantized table: the embedding lookup at the
// start of the Llama graph in "llama.cpp 深度解读" §4 (ggml_get_rows(tok_embeddings,
// inp_tokens)), with the token-embedding tensor stored as Q4_0 (the GGUF tensor
// info example of §1) or Q8_0.  Output row i is the decode of table row ids[i]
// (§2: (nibble - 8) * d, resp. q * d), which is exact in fp32.
//
// HBM-bound and write-dominated (4 bytes out per 0.5625 or 1.0625 bytes in): one
// thread decodes 8 consecutive elements (a quarter of a block) and writes them as
// two 16-byte streaming stores, so a warp writes 1 KB of one output row at once.
#include <algorithm>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

__device__ unsigned int g_rows_status = 0;

constexpr int ROWS_THREADS = 256;

template <bool Q4>
__global__ void __launch_bounds__(ROWS_THREADS)
get_rows_kernel(const uint8_t* __restrict__ table, int64_t nrows, int nb, const int32_t* __restrict__ ids,
                int64_t n, float* __restrict__ dst) {
    constexpr int BB = Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    const int per_row = nb * 4;                     // items (8 elements) per output row
    const int64_t total = n * per_row;
    const int64_t row_bytes = (int64_t)nb * BB;
    for (int64_t g = blockIdx.x * (int64_t)ROWS_THREADS + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * ROWS_THREADS) {
        const int64_t i = g / per_row;
        const int c = (int)(g - i * per_row);
        const int b = c >> 2, qtr = c & 3;
        const int64_t id = ids ? (int64_t)__ldg(ids + i) : i;
        float v[8];
        if (id < 0 || id >= nrows) {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.0f;
            if (c == 0) record_error(&g_rows_status, Q4Q_ERR_ARG);
        } else {
            const uint16_t* blk = reinterpret_cast<const uint16_t*>(table + id * row_bytes + (int64_t)b * BB);
            const float d = fp16_to_f32(__ldg(blk));
            if constexpr (Q4) {
                // elements 8q .. 8q+7 are qs bytes 4q .. 4q+3: low nibble first
                const uint32_t wv = (uint32_t)__ldg(blk + 1 + 2 * qtr) | ((uint32_t)__ldg(blk + 2 + 2 * qtr) << 16);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __fmul_rn((float)((int)((wv >> (4 * e)) & 0xFu) - 8), d);
            } else {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const uint32_t two = __ldg(blk + 1 + 4 * qtr + h);   // elements 8q + 2h, 8q + 2h + 1
                    v[2 * h] = __fmul_rn((float)(int8_t)(two & 0xffu), d);
                    v[2 * h + 1] = __fmul_rn((float)(int8_t)(two >> 8), d);
                }
            }
        }
        float4* o = reinterpret_cast<float4*>(dst + i * (int64_t)nb * QK + c * 8);
        __stcs(o, make_float4(v[0], v[1], v[2], v[3]));
        __stcs(o + 1, make_float4(v[4], v[5], v[6], v[7]));
    }
}

q4q_status get_rows(bool q4, const void* src0, int64_t ne00, int64_t ne01, const int32_t* ids, int64_t n_ids,
                    float* dst, cudaStream_t stream) {
    if (ne00 <= 0 || ne00 % QK != 0 || ne00 >= (1 << 20) || ne01 < 0 || ne01 >= (1ll << 31) || n_ids < 0 ||
        n_ids >= (1ll << 31))
        return Q4Q_ERR_SHAPE;
    if (!ids && n_ids > ne01) return Q4Q_ERR_SHAPE;
    if (n_ids == 0) return Q4Q_OK;
    if (!src0 || !dst) return Q4Q_ERR_NULL;
    if (!aligned(src0, 2) || !aligned(dst, 16) || (ids && !aligned(ids, 4))) return Q4Q_ERR_ALIGN;
    DeviceInfo info;
    q4q_status st = current_device_info(&info);
    if (st != Q4Q_OK) return st;
    const int64_t items = n_ids * (ne00 / 8);
    const int grid = (int)std::min<int64_t>((items + ROWS_THREADS - 1) / ROWS_THREADS, (int64_t)info.sm_count * 16);
    const int nb = (int)(ne00 / QK);
    if (q4)
        get_rows_kernel<true><<<grid, ROWS_THREADS, 0, stream>>>(static_cast<const uint8_t*>(src0), ne01, nb, ids,
                                                                 n_ids, dst);
    else
        get_rows_kernel<false><<<grid, ROWS_THREADS, 0, stream>>>(static_cast<const uint8_t*>(src0), ne01, nb, ids,
                                                                  n_ids, dst);
    return launch_status();
}

}  // namespace

unsigned int rows_take_device_status() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_rows_status, sizeof(v)) != cudaSuccess) return Q4Q_ERR_CUDA;
    if (v) cudaMemcpyToSymbol(g_rows_status, &z, sizeof(z));
    return v;
}

}  // namespace q4q

extern "C" q4q_status q4q_get_rows_q4_0(const void* src0, int64_t ne00, int64_t ne01, const int32_t* ids,
                                        int64_t n_ids, float* dst, q4q_stream_t stream) {
    return q4q::get_rows(true, src0, ne00, ne01, ids, n_ids, dst, (cudaStream_t)stream);
}

extern "C" q4q_status q4q_get_rows_q8_0(const void* src0, int64_t ne00, int64_t ne01, const int32_t* ids,
                                        int64_t n_ids, float* dst, q4q_stream_t stream) {
    return q4q::get_rows(false, src0, ne00, ne01, ids, n_ids, dst, (cudaStream_t)stream);
}
