// q4q_quant.cu -- Q4_0 and Q8_0 block quantizers (device, sm_103a).
//
// Q4_0: "llama.cpp 深度解读" §2 "量化数据结构 — Q4_0 格式详解" (encode steps 1-4,
// block { fp16 d; uint8 qs[16]; }).  Q8_0: the activation format of §3
// "量化矩阵乘法 — 核心算子" (fp16 d + 32 int8; scale amax/127).
//
// Both are HBM-bound: 4 bytes read per element, 0.5625 (Q4_0) or 1.0625 (Q8_0)
// bytes written.  Four consecutive lanes own one 32-element block (8 elements,
// two 16-byte loads each), the block amax is a 2-step xor shuffle, and the
// 18/34-byte blocks of 64 consecutive blocks are assembled in shared memory so
// that the output leaves as 16-byte stores (64 * 18 = 72 * 16, 64 * 34 = 136 * 16).
#include <algorithm>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

constexpr int CHUNK = 64;        // blocks per CTA iteration (256 threads x 8 elements)
constexpr int THREADS = 256;

template <bool IS_Q4>
__global__ void __launch_bounds__(THREADS)
quantize_fast_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int64_t nblocks) {
    constexpr int BB = IS_Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    __shared__ __align__(16) uint8_t stage[CHUNK * BB];
    const int tid = threadIdx.x;
    const int bl = tid >> 2;       // block within the chunk
    const int part = tid & 3;      // which 8 elements of the block
    const int64_t nchunks = (nblocks + CHUNK - 1) / CHUNK;

    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x) {
        const int64_t gb = c * CHUNK + bl;
        float v[8];
        if (gb < nblocks) {
            const float4* p = reinterpret_cast<const float4*>(src + gb * QK + part * 8);
            float4 a = __ldcs(p), b = __ldcs(p + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        amax = warp_max4(amax);
        uint8_t* sb = stage + bl * BB;
        if (IS_Q4) {
            const float d = scale_q4(amax);
            const uint32_t w = pack_q4_word(v, d);
            uint16_t* q = reinterpret_cast<uint16_t*>(sb + 2 + 4 * part);
            q[0] = (uint16_t)(w & 0xffffu);
            q[1] = (uint16_t)(w >> 16);
            if (part == 0) *reinterpret_cast<uint16_t*>(sb) = fp16_bits(d);
        } else {
            const float d = scale_q8(amax);
            int qv[8];
            quant8(v, d, -127.0f, 127.0f, qv);
            uint16_t* q = reinterpret_cast<uint16_t*>(sb + 2 + 8 * part);
#pragma unroll
            for (int e = 0; e < 8; e += 2)
                q[e >> 1] = (uint16_t)((uint32_t)(qv[e] & 0xff) | ((uint32_t)(qv[e + 1] & 0xff) << 8));
            if (part == 0) *reinterpret_cast<uint16_t*>(sb) = fp16_bits(d);
        }
        __syncthreads();
        const int64_t left = nblocks - c * CHUNK;
        const int bytes = (int)((left < CHUNK ? left : CHUNK) * BB);
        uint8_t* out = dst + c * (int64_t)(CHUNK * BB);
        const int nvec = bytes >> 4;
        for (int i = tid; i < nvec; i += THREADS)
            reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(stage)[i];
        for (int i = (nvec << 4) + tid; i < bytes; i += THREADS) out[i] = stage[i];
        __syncthreads();
    }
}

// Any alignment (src 4-byte aligned): one thread per block; the blocks of a
// CTA are assembled in shared memory and leave as consecutive byte stores.
template <bool IS_Q4>
__global__ void __launch_bounds__(THREADS)
quantize_generic_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int64_t nblocks) {
    constexpr int BB = IS_Q4 ? Q4_0_BYTES : Q8_0_BYTES;
    __shared__ __align__(16) uint8_t stage[THREADS * BB];
    for (int64_t g0 = (int64_t)blockIdx.x * THREADS; g0 < nblocks; g0 += (int64_t)gridDim.x * THREADS) {
        const int64_t gb = g0 + threadIdx.x;
        uint8_t* o = stage + threadIdx.x * BB;
        if (gb < nblocks) {
            const float* x = src + gb * QK;
            float amax = 0.0f;
            for (int k = 0; k < QK; ++k) amax = fmaxf(amax, fabsf(x[k]));
            const float d = __fdiv_rn(amax, IS_Q4 ? 8.0f : 127.0f);
            *reinterpret_cast<uint16_t*>(o) = fp16_bits(d);     // o is 2-byte aligned (BB is even)
            if (IS_Q4) {
                for (int j = 0; j < QK / 2; ++j) {
                    const int lo = quant_one(x[2 * j], d, -8.0f, 7.0f) + 8;
                    const int hi = quant_one(x[2 * j + 1], d, -8.0f, 7.0f) + 8;
                    o[2 + j] = (uint8_t)(lo | (hi << 4));
                }
            } else {
                for (int k = 0; k < QK; ++k) o[2 + k] = (uint8_t)(quant_one(x[k], d, -127.0f, 127.0f) & 0xff);
            }
        }
        __syncthreads();
        const int64_t left = nblocks - g0;
        const int bytes = (int)((left < THREADS ? left : THREADS) * BB);
        uint8_t* out = dst + g0 * BB;
        for (int i = threadIdx.x; i < bytes; i += THREADS) out[i] = stage[i];
        __syncthreads();
    }
}

q4q_status validate(const float* src, const void* dst, int64_t ncols, int64_t nrows) {
    if (ncols <= 0 || ncols % QK != 0 || nrows < 0) return Q4Q_ERR_SHAPE;
    if (nrows > 0 && ncols > ((int64_t)1 << 40) / nrows) return Q4Q_ERR_SHAPE;
    if (nrows == 0) return Q4Q_OK;
    if (!src || !dst) return Q4Q_ERR_NULL;
    if (!aligned(src, 4)) return Q4Q_ERR_ALIGN;
    return Q4Q_OK;
}

}  // namespace

q4q_status launch_quantize(bool q4, const float* src, void* dst, int64_t ncols, int64_t nrows,
                           cudaStream_t stream, const DeviceInfo& info) {
    const int64_t nblocks = ncols / QK * nrows;
    if (nblocks == 0) return Q4Q_OK;
    uint8_t* out = static_cast<uint8_t*>(dst);
    if (aligned(src, 16) && aligned(dst, 16)) {
        const int64_t nchunks = (nblocks + CHUNK - 1) / CHUNK;
        const int grid = (int)std::min<int64_t>(nchunks, (int64_t)info.sm_count * 8);
        if (q4) quantize_fast_kernel<true><<<grid, THREADS, 0, stream>>>(src, out, nblocks);
        else    quantize_fast_kernel<false><<<grid, THREADS, 0, stream>>>(src, out, nblocks);
    } else {
        const int grid = (int)std::min<int64_t>((nblocks + THREADS - 1) / THREADS, (int64_t)info.sm_count * 4);
        if (q4) quantize_generic_kernel<true><<<grid, THREADS, 0, stream>>>(src, out, nblocks);
        else    quantize_generic_kernel<false><<<grid, THREADS, 0, stream>>>(src, out, nblocks);
    }
    return launch_status();
}

}  // namespace q4q

extern "C" q4q_status q4q_quantize_q4_0(const float* src, void* dst, int64_t ncols, int64_t nrows,
                                        q4q_stream_t stream) {
    q4q_status st = q4q::validate(src, dst, ncols, nrows);
    if (st != Q4Q_OK || nrows == 0) return st;
    q4q::DeviceInfo info;
    if ((st = q4q::current_device_info(&info)) != Q4Q_OK) return st;
    return q4q::launch_quantize(true, src, dst, ncols, nrows, (cudaStream_t)stream, info);
}

extern "C" q4q_status q4q_quantize_q8_0(const float* src, void* dst, int64_t ncols, int64_t nrows,
                                        q4q_stream_t stream) {
    q4q_status st = q4q::validate(src, dst, ncols, nrows);
    if (st != Q4Q_OK || nrows == 0) return st;
    q4q::DeviceInfo info;
    if ((st = q4q::current_device_info(&info)) != Q4Q_OK) return st;
    return q4q::launch_quantize(false, src, dst, ncols, nrows, (cudaStream_t)stream, info);
}
