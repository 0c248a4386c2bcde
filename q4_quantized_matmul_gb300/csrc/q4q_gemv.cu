// q4q_gemv.cu -- Q4_0 x Q8_0 matrix-vector product for 1..7 tokens (decode).
//
// Computes ggml_mul_mat(Q4_0 src0 [ne00, ne01], F32 src1 [ne00, ne11]) as
// "llama.cpp 深度解读" §3 "量化矩阵乘法 — 核心算子" states it: src1 rows are
// quantized to Q8_0, and every output is sum_b fp32(d_w * d_x) * isum_b with
// isum_b the exact integer dot of one 32-element block (nibble - 8 times int8).
//
// Design (HBM-bound: every weight byte is read exactly once):
//  * One persistent CTA per SM slot streams "units" of G consecutive weight rows
//    (rows are contiguous, so a unit is one contiguous byte range) into a ring of
//    S shared-memory stages with 1-D TMA bulk copies (cp.async.bulk), completion
//    tracked by mbarriers.  Requires ne00 % 256 == 0 so rows are 16-byte multiples.
//  * Before the first stage is consumed, the CTA quantizes the activations itself
//    (the per-row Q8_0 step of the same page) into shared memory, in a layout
//    made for the dot: per pair of blocks four 16-byte quads {even elements of
//    block a, odd of a, even of b, odd of b}, plus per block the widened fp16
//    scale and 8 * sum(q).  This runs while the first weight stages are in flight.
//  * LPR lanes own one row; lane s owns block pairs s, s+LPR, ...  A pair of
//    18-byte blocks is 36 bytes = 9 aligned words, so lanes reading consecutive
//    pairs hit 9-word strides: conflict-free shared-memory loads.
//  * Nibbles: byte j holds element 2j (low) and 2j+1 (high) (§2), so the low
//    nibbles of a qs word pair with the even activations and the high nibbles
//    with the odd ones: isum = dp4a(lo, even) + dp4a(hi, odd) - 8 * sum(q).
#include <algorithm>
#include <atomic>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

__device__ unsigned int g_gemv_status = 0;

constexpr int THREADS = 288;            // 8 consumer warps + 1 producer warp
constexpr int CONSUMERS = 256;
constexpr int MAX_STAGES = 8;
constexpr int PLAIN_THREADS = 256;      // generic and debug kernels

struct GemvParams {
    int ne00, nb, np, ne01, row_bytes;
    int G;             // rows per unit
    int n_units;
    int S;             // stages in the ring
    int stage_bytes;   // bytes per stage (multiple of 128)
    int act_off;       // smem offset of the activation quads
    int dy_off, sy_off, stage_off;
};

// Integer dot of one pair of Q4_0 blocks (9 aligned words, block a at byte 0,
// block b at byte 18) against Q8_0 activations in the even/odd quad layout.
struct PairWeights {
    float da, db;
    uint32_t qa[4], qb[4];
};

__device__ __forceinline__ PairWeights unpack_pair(const uint32_t (&w)[9]) {
    PairWeights p;
    p.da = fp16_to_f32(w[0]);
    p.db = fp16_to_f32(w[4] >> 16);
    // block a's 16 nibble bytes start at byte 2 of word 0
#pragma unroll
    for (int i = 0; i < 4; ++i) p.qa[i] = __byte_perm(w[i], w[i + 1], 0x5432);
#pragma unroll
    for (int i = 0; i < 4; ++i) p.qb[i] = w[5 + i];
    return p;
}

__device__ __forceinline__ int block_dot(const uint32_t (&q)[4], const uint4& ye, const uint4& yo) {
    int s = 0;
    s = __dp4a((int)(q[0] & 0x0F0F0F0Fu), (int)ye.x, s);
    s = __dp4a((int)((q[0] >> 4) & 0x0F0F0F0Fu), (int)yo.x, s);
    s = __dp4a((int)(q[1] & 0x0F0F0F0Fu), (int)ye.y, s);
    s = __dp4a((int)((q[1] >> 4) & 0x0F0F0F0Fu), (int)yo.y, s);
    s = __dp4a((int)(q[2] & 0x0F0F0F0Fu), (int)ye.z, s);
    s = __dp4a((int)((q[2] >> 4) & 0x0F0F0F0Fu), (int)yo.z, s);
    s = __dp4a((int)(q[3] & 0x0F0F0F0Fu), (int)ye.w, s);
    s = __dp4a((int)((q[3] >> 4) & 0x0F0F0F0Fu), (int)yo.w, s);
    return s;
}

// Quantize 8 consecutive activations (elements 8i..8i+7 of one block) to Q8_0
// and split them into the even word (elements 8i, 8i+2, 8i+4, 8i+6) and the odd
// word (8i+1, ...).  Returns sum of the 8 codes.  All 32 lanes must call it.
__device__ __forceinline__ int quant_q8_split(const float (&v)[8], float d, uint32_t& ye, uint32_t& yo) {
    int s = 0;
    ye = 0; yo = 0;
    int qv[8];
    quant8(v, d, -127.0f, 127.0f, qv);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int q = qv[e];
        s += q;
        const uint32_t b = (uint32_t)(q & 0xff);
        if (e & 1) yo |= b << (8 * (e >> 1));
        else       ye |= b << (8 * (e >> 1));
    }
    return s;
}

// Activations of one block pair in the quad layout (+ scales and 8 * sum(q)).
struct PairActs {
    uint4 ea, oa, eb, ob;
    float2 d;
    int2 s8;
};

__device__ __forceinline__ PairActs load_pair_acts(const uint4* quads, const float* dy, const int* sy8, int np,
                                                   int nb, int t, int pr) {
    PairActs a;
    const uint4* qp = quads + (t * 4) * np + pr;
    a.ea = qp[0];
    a.oa = qp[np];
    a.eb = qp[2 * np];
    a.ob = qp[3 * np];
    a.d = reinterpret_cast<const float2*>(dy + t * nb)[pr];
    a.s8 = reinterpret_cast<const int2*>(sy8 + t * nb)[pr];
    return a;
}

__device__ __forceinline__ float pair_dot(const uint8_t* rowp, int pr, const PairActs& a, float acc) {
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowp + 36 * pr);
    uint32_t wv[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) wv[i] = wp[i];
    const PairWeights pw = unpack_pair(wv);
    const int ia = block_dot(pw.qa, a.ea, a.oa) - a.s8.x;
    const int ib = block_dot(pw.qb, a.eb, a.ob) - a.s8.y;
    acc = fmaf(pw.da * a.d.x, (float)ia, acc);
    acc = fmaf(pw.db * a.d.y, (float)ib, acc);
    return acc;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS) : "memory");
}

// T tokens; LPR lanes per row; PPL > 0: the lane's PPL block pairs of activations
// are held in registers for the whole kernel (T == 1), PPL == 0: read from shared
// memory for every row.
template <int T, int LPR, int PPL>
__global__ void __launch_bounds__(THREADS, (PPL > 0 && PPL <= 3) ? 2 : 1)
gemv_q4_0_kernel(const uint8_t* __restrict__ w, const float* __restrict__ x, float* __restrict__ dst,
                 const GemvParams p) {
    static_assert(PPL == 0 || T == 1, "register-resident activations are for one token");
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);              // full[0..7], empty[8..15]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 128);
    uint4* quads = reinterpret_cast<uint4*>(smem + p.act_off);
    float* dy = reinterpret_cast<float*>(smem + p.dy_off);
    int* sy8 = reinterpret_cast<int*>(smem + p.sy_off);
    uint8_t* stages = smem + p.stage_off;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grid = gridDim.x;
    const uint32_t full0 = smem_u32(&bars[0]), empty0 = smem_u32(&bars[MAX_STAGES]);

    if (tid == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, CONSUMERS / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // the next kernel on the stream may start its own set-up now; it still waits
    // for this grid to finish before it touches memory this grid writes
    pdl_trigger();

    if (warp == CONSUMERS / 32) {
        // ---------------- producer: stream weight units through the ring
        if (lane == 0) {
            int k = 0;
            for (int u = blockIdx.x; u < p.n_units; u += grid, ++k) {
                const int s = k % p.S;
                if (k >= p.S) {
                    const uint32_t bar = empty0 + 8 * s, par = ((k / p.S) + 1) & 1;
                    bool ok = mbar_try_wait(bar, par);
                    if (!ok) {
                        const uint64_t t0 = global_timer_ns();
                        while (!ok && !*abort_flag && global_timer_ns() - t0 < WAIT_LIMIT_NS)
                            ok = mbar_try_wait_sleep(bar, par, SLEEP_HINT_NS);
                    }
                    if (!ok) {
                        if (!*abort_flag) record_error(&g_gemv_status, DEV_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                }
                const int r0 = u * p.G;
                const int nr = min(p.G, p.ne01 - r0);
                const uint32_t bytes = (uint32_t)nr * (uint32_t)p.row_bytes;
                mbar_arrive_expect_tx(full0 + 8 * s, bytes);
                bulk_g2s(smem_u32(stages + (size_t)s * p.stage_bytes), w + (int64_t)r0 * p.row_bytes, bytes,
                         full0 + 8 * s);
            }
            if (*abort_flag) {
                // let the copies still in flight land before the CTA exits
                for (int k2 = max(0, k - p.S); k2 < k; ++k2)
                    mbar_wait_bounded(full0 + 8 * (k2 % p.S), (uint32_t)((k2 / p.S) & 1), WAIT_LIMIT_NS);
            }
        }
        return;
    }

    // ---------------- consumers: activations first (they may come from the previous kernel)
    pdl_wait();
    {
        // Each thread owns 8 consecutive activations of one block per item; the
        // loads of U items are issued together so that their L2 latencies overlap.
        constexpr int U = 4;
        const int per_tok = p.nb * 4;
        const int total = T * per_tok;               // a multiple of 32: warps stay uniform
        for (int m0 = 0; m0 < total; m0 += CONSUMERS * U) {
            float4 va[U], vb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int m = m0 + u * CONSUMERS + tid;
                if (m < total) {
                    const int t = m / per_tok, rem = m - t * per_tok;
                    const float4* src =
                        reinterpret_cast<const float4*>(x + (int64_t)t * p.ne00 + (rem >> 2) * QK + (rem & 3) * 8);
                    va[u] = __ldg(src);
                    vb[u] = __ldg(src + 1);
                } else {
                    va[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    vb[u] = va[u];
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int m = m0 + u * CONSUMERS + tid;
                if (m0 + u * CONSUMERS >= total) break;    // uniform across the CTA
                const bool ok = m < total;
                const int t = ok ? m / per_tok : 0;
                const int rem = m - t * per_tok;
                const int b = rem >> 2, i = rem & 3;
                const float v[8] = {va[u].x, va[u].y, va[u].z, va[u].w, vb[u].x, vb[u].y, vb[u].z, vb[u].w};
                float amax = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
                amax = warp_max4(amax);
                const float d = scale_q8(amax);
                uint32_t ye, yo;
                int sq = quant_q8_split(v, d, ye, yo);
                sq = warp_sum4(sq);
                if (ok) {
                    const int qi = (t * 4 + (b & 1) * 2) * p.np + (b >> 1);
                    reinterpret_cast<uint32_t*>(&quads[qi])[i] = ye;
                    reinterpret_cast<uint32_t*>(&quads[qi + p.np])[i] = yo;
                    if (i == 0) {
                        dy[t * p.nb + b] = fp16_to_f32(fp16_bits(d));
                        sy8[t * p.nb + b] = 8 * sq;
                    }
                }
            }
        }
    }
    consumer_sync();

    constexpr int RP = CONSUMERS / LPR;     // rows processed side by side
    const int rr = tid / LPR, sl = tid % LPR;
    const int passes = (p.G + RP - 1) / RP;
    PairActs areg[PPL > 0 ? PPL : 1];
    if (PPL > 0) {
#pragma unroll
        for (int kk = 0; kk < (PPL > 0 ? PPL : 1); ++kk)
            areg[kk] = load_pair_acts(quads, dy, sy8, p.np, p.nb, 0, sl + kk * LPR);
    }
    const int ppl = p.np / LPR;

    int k = 0;
    for (int u = blockIdx.x; u < p.n_units; u += grid, ++k) {
        const int s = k % p.S;
        {
            const uint32_t bar = full0 + 8 * s, par = (uint32_t)((k / p.S) & 1);
            int ok = 1;
            if (lane == 0) {
                bool got = mbar_try_wait(bar, par);
                if (!got) {
                    const uint64_t t0 = global_timer_ns();
                    while (!got && !*abort_flag && global_timer_ns() - t0 < WAIT_LIMIT_NS)
                        got = mbar_try_wait_sleep(bar, par, SLEEP_HINT_NS);
                }
                if (!got) {
                    if (!*abort_flag) record_error(&g_gemv_status, DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                ok = got ? 1 : 0;
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            mbar_try_wait(bar, par);       // per-lane acquire of the completed phase
        }
        const uint8_t* stage = stages + (size_t)s * p.stage_bytes;
        const int r0 = u * p.G;
        const int nr = min(p.G, p.ne01 - r0);
        for (int pass = 0; pass < passes; ++pass) {
            const int j = rr + pass * RP;
            const bool valid = j < nr;
            float acc[T];
#pragma unroll
            for (int t = 0; t < T; ++t) acc[t] = 0.0f;
            if (valid) {
                const uint8_t* rowp = stage + (size_t)j * p.row_bytes;
                if (PPL > 0) {
#pragma unroll
                    for (int kk = 0; kk < (PPL > 0 ? PPL : 1); ++kk)
                        acc[0] = pair_dot(rowp, sl + kk * LPR, areg[kk], acc[0]);
                } else {
                    for (int kk = 0; kk < ppl; ++kk) {
                        const int pr = sl + kk * LPR;
#pragma unroll
                        for (int t = 0; t < T; ++t)
                            acc[t] = pair_dot(rowp, pr, load_pair_acts(quads, dy, sy8, p.np, p.nb, t, pr), acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < T; ++t) {
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1)
                    acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
            }
            if (valid && sl == 0) {
#pragma unroll
                for (int t = 0; t < T; ++t) dst[(int64_t)t * p.ne01 + r0 + j] = acc[t];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
}

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

struct GemvPlan {
    GemvParams p;
    int lpr;
    int ppl_reg;       // > 0: activations in registers
    int grid;
    size_t smem;
};

bool plan_gemv(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info, GemvPlan* plan) {
    if (ne11 < 1 || ne11 > 7 || ne00 % 256 != 0 || ne00 > (1 << 20) || ne01 <= 0 || ne01 >= (1ll << 31))
        return false;
    GemvParams& p = plan->p;
    p.ne00 = (int)ne00;
    p.nb = (int)(ne00 / QK);
    p.np = p.nb / 2;
    p.ne01 = (int)ne01;
    p.row_bytes = p.nb * Q4_0_BYTES;
    int lpr = 4;
    for (int c : {32, 16, 8}) if (p.np % c == 0) { lpr = c; break; }
    const int ppl = p.np / lpr;
    plan->ppl_reg = (ne11 == 1 && ppl <= 8) ? ppl : 0;
    const int RP = CONSUMERS / lpr;
    const int64_t act = ne11 * ((int64_t)p.np * 64 + (int64_t)p.nb * 8);
    const int64_t head = 256;  // mbarriers + abort flag
    const int64_t act_bytes = (act + 127) / 128 * 128;
    const int64_t limit = std::min<int64_t>(info.max_smem_optin, 227 * 1024) - 1024;
    const int64_t sms = info.sm_count;
    const int64_t wbytes = ne01 * (int64_t)p.row_bytes;
    const bool two_per_sm = plan->ppl_reg == 0 || plan->ppl_reg <= 3;
    int64_t G, S, stage;
    bool small = false;
    if (two_per_sm && wbytes <= 96 * 1024 * sms) {
        // Small matrix: one CTA per SM holds every unit it owns in flight from the
        // start (about two units each), and leaves room on the SM for the next
        // kernel's CTA, which can then prefetch its own weights under PDL.
        G = std::max<int64_t>(1, (ne01 + 2 * sms - 1) / (2 * sms));
        const int64_t units = (ne01 + G - 1) / G;
        S = std::min<int64_t>(MAX_STAGES, (units + sms - 1) / sms);
        stage = ((G * p.row_bytes) + 127) / 128 * 128;
        small = head + act_bytes + S * stage <= std::min<int64_t>(limit, 110 * 1024);
    }
    if (!small) {
        // rows per unit: aim at ~32 KB stages, but keep >= 2 units per SM when the matrix allows
        const int64_t rp_bytes = (int64_t)RP * p.row_bytes;
        G = RP * std::max<int64_t>(1, (32768 + rp_bytes / 2) / rp_bytes);
        while (G > 8 && (ne01 + G - 1) / G < 2 * sms) G = std::max<int64_t>(8, G / 2);
        G = std::min<int64_t>(G, ne01);
        stage = ((G * p.row_bytes) + 127) / 128 * 128;
        S = 0;
        if (two_per_sm) S = (std::min<int64_t>(limit, 110 * 1024) - head - act_bytes) / stage;
        if (S < 3) S = (limit - head - act_bytes) / stage;
        if (S < 2) return false;
        S = std::min<int64_t>(S, MAX_STAGES);
    }
    p.G = (int)G;
    p.n_units = (int)((ne01 + G - 1) / G);
    p.S = (int)S;
    p.stage_bytes = (int)stage;
    p.act_off = (int)head;
    p.dy_off = (int)(head + ne11 * (int64_t)p.np * 64);
    p.sy_off = (int)(p.dy_off + ne11 * (int64_t)p.nb * 4);
    p.stage_off = (int)(head + act_bytes);
    plan->smem = (size_t)(head + act_bytes + S * stage);
    plan->lpr = lpr;
    const int per_sm = (!small && plan->smem <= 113 * 1024 && two_per_sm) ? 2 : 1;
    plan->grid = (int)std::min<int64_t>(p.n_units, sms * per_sm);
    return true;
}

template <int T, int LPR, int PPL>
q4q_status launch_gemv_t(const GemvPlan& plan, const uint8_t* w, const float* x, float* dst, cudaStream_t stream,
                         int device, bool pdl) {
    // the opt-in shared-memory size is raised once per device and kernel
    static std::atomic<int> configured[64];
    auto kern = gemv_q4_0_kernel<T, LPR, PPL>;
    if (device < 0 || device >= 64) return Q4Q_ERR_CUDA;
    if ((int)plan.smem > configured[device].load()) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem) != cudaSuccess)
            return Q4Q_ERR_CUDA;
        configured[device].store((int)plan.smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, w, x, dst, plan.p) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4Q_ERR_CUDA;
    }
    return launch_status();
}

template <int T, int LPR>
q4q_status launch_gemv_ppl(const GemvPlan& plan, const uint8_t* w, const float* x, float* dst, cudaStream_t stream,
                           int device, bool pdl) {
    if (T == 1) {
        switch (plan.ppl_reg) {
            case 1: return launch_gemv_t<T, LPR, (T == 1 ? 1 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 2: return launch_gemv_t<T, LPR, (T == 1 ? 2 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 3: return launch_gemv_t<T, LPR, (T == 1 ? 3 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 4: return launch_gemv_t<T, LPR, (T == 1 ? 4 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 5: return launch_gemv_t<T, LPR, (T == 1 ? 5 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 6: return launch_gemv_t<T, LPR, (T == 1 ? 6 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 7: return launch_gemv_t<T, LPR, (T == 1 ? 7 : 0)>(plan, w, x, dst, stream, device, pdl);
            case 8: return launch_gemv_t<T, LPR, (T == 1 ? 8 : 0)>(plan, w, x, dst, stream, device, pdl);
            default: break;
        }
    }
    return launch_gemv_t<T, LPR, 0>(plan, w, x, dst, stream, device, pdl);
}

template <int T>
q4q_status launch_gemv_lpr(const GemvPlan& plan, const uint8_t* w, const float* x, float* dst, cudaStream_t stream,
                           int device, bool pdl) {
    switch (plan.lpr) {
        case 32: return launch_gemv_ppl<T, 32>(plan, w, x, dst, stream, device, pdl);
        case 16: return launch_gemv_ppl<T, 16>(plan, w, x, dst, stream, device, pdl);
        case 8:  return launch_gemv_ppl<T, 8>(plan, w, x, dst, stream, device, pdl);
        default: return launch_gemv_ppl<T, 4>(plan, w, x, dst, stream, device, pdl);
    }
}

}  // namespace

unsigned int gemv_take_device_status() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(v)) != cudaSuccess) return Q4Q_ERR_CUDA;
    if (v) cudaMemcpyToSymbol(g_gemv_status, &z, sizeof(z));
    return v;
}

bool gemv_supported(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                    const DeviceInfo& info) {
    GemvPlan plan;
    return aligned(src0, 16) && aligned(src1, 16) && plan_gemv(ne00, ne01, ne11, info, &plan);
}

q4q_status gemv_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11,
                        float* dst, cudaStream_t stream, const DeviceInfo& info, bool pdl) {
    GemvPlan plan;
    if (!plan_gemv(ne00, ne01, ne11, info, &plan)) return Q4Q_ERR_SHAPE;
    const uint8_t* w = static_cast<const uint8_t*>(src0);
    switch (ne11) {
        case 1: return launch_gemv_lpr<1>(plan, w, src1, dst, stream, info.device, pdl);
        case 2: return launch_gemv_lpr<2>(plan, w, src1, dst, stream, info.device, pdl);
        case 3: return launch_gemv_lpr<3>(plan, w, src1, dst, stream, info.device, pdl);
        case 4: return launch_gemv_lpr<4>(plan, w, src1, dst, stream, info.device, pdl);
        case 5: return launch_gemv_lpr<5>(plan, w, src1, dst, stream, info.device, pdl);
        case 6: return launch_gemv_lpr<6>(plan, w, src1, dst, stream, info.device, pdl);
        default: return launch_gemv_lpr<7>(plan, w, src1, dst, stream, info.device, pdl);
    }
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
