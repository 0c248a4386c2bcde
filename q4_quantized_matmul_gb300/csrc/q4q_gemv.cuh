// q4q_gemv.cuh -- the GEMV kernels for 1..7 tokens (decode), shared by the
// translation units that instantiate them: Q4_0 weights (q4q_gemv.cu), Q4_0
// gate/up pairs with the SwiGLU epilogue (q4q_gemv_swiglu.cu) and Q8_0 weights
// (q4q_gemv_w8.cu).  Each unit gets its own copy of everything below, including
// its own device status word.
//
// Computes ggml_mul_mat(Q src0 [ne00, ne01], F32 src1 [ne00, ne11]) as
// "llama.cpp 深度解读" §3 "量化矩阵乘法 — 核心算子" states it: src1 rows are
// quantized to Q8_0, and every output is sum_b fp32(d_w * d_x) * isum_b with
// isum_b the exact integer dot of one 32-element block (nibble - 8 times int8
// for Q4_0 weights, int8 times int8 for Q8_0 weights).
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
//    18-byte blocks is 36 bytes = 9 aligned words (Q8_0: 68 bytes = 17 words), so
//    lanes reading consecutive pairs hit odd word strides: conflict-free
//    shared-memory loads.
//  * Nibbles: byte j holds element 2j (low) and 2j+1 (high) (§2), so the low
//    nibbles of a qs word pair with the even activations and the high nibbles
//    with the odd ones: isum = dp4a(lo, even) + dp4a(hi, odd) - 8 * sum(q).
#pragma once

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {


__device__ unsigned int g_gemv_status = 0;

constexpr int THREADS = 288;            // 8 consumer warps + 1 producer warp
constexpr int CONSUMERS = 256;
constexpr int MAX_STAGES = 8;
constexpr int PLAIN_THREADS = 256;      // generic and debug kernels
constexpr int WQ4_0 = 0;                 // weight block types
constexpr int WQ8_0 = 1;
constexpr int M_SINGLE = 0;              // kernel modes: one matrix,
constexpr int M_DUAL = 1;                //   two matrices, SwiGLU of the pair,
constexpr int M_GROUP = 2;               //   up to GROUP_MAX matrices with one input,
constexpr int M_EPI = 3;                 //   one matrix with the bias / activation epilogue
constexpr int GROUP_MAX = Q4Q_GROUP_MAX;

// Group mode: matrix m owns the units [unit0[m], unit0[m+1]) (unit0[n] = all units).
struct GemvGroup {
    int n;
    int unit0[GROUP_MAX + 1];
    int rows[GROUP_MAX];
    const uint8_t* w[GROUP_MAX];
    float* dst[GROUP_MAX];
};
constexpr int64_t CLUSTER_MIN_X = 8192;  // activations (elements) from which CTA pairs share the quantization

struct GemvParams {
    int ne00, nb, np, ne01, row_bytes;
    int G;             // rows per unit
    int n_units;
    int S;             // stages in the ring
    int stage_bytes;   // bytes per stage (multiple of 128)
    int act_off;       // smem offset of the activation quads
    int dy_off, sy_off, stage_off;
    int half_off;      // dual-weight ring: offset of the second matrix's rows in a stage
    int act;           // Q4Q_ACT_* applied to every output (after the bias)
    const float* bias; // [ne01] added to every output row, or null
    GemvGroup grp;     // group mode only
    uint64_t limit_ns; // bound of every wait (WAIT_LIMIT_NS unless a test asks for less)
    int fault;         // test only: 1 = CTA 0 leaves out its first unit's copies
};

// The rows a unit covers: its matrix's weights, output and row count, and its
// first row there.  Group mode picks the matrix with static indices only (a
// dynamic index into the parameter struct would copy it to local memory).
struct UnitRows {
    const uint8_t* w;
    float* dst;
    int rows, r0;
};

template <int MODE>
__device__ __forceinline__ UnitRows unit_rows(const GemvParams& p, const uint8_t* w, float* dst, int u) {
    UnitRows r{w, dst, p.ne01, u * p.G};
    if constexpr (MODE == M_GROUP) {
        r.w = p.grp.w[0];
        r.dst = p.grp.dst[0];
        r.rows = p.grp.rows[0];
        int base = 0;
#pragma unroll
        for (int q = 1; q < GROUP_MAX; ++q) {
            if (q < p.grp.n && u >= p.grp.unit0[q]) {
                r.w = p.grp.w[q];
                r.dst = p.grp.dst[q];
                r.rows = p.grp.rows[q];
                base = p.grp.unit0[q];
            }
        }
        r.r0 = (u - base) * p.G;
    }
    return r;
}

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

// Item m of the activations (token t, m = t * 4 nb + 4 b + i) covers elements
// 8i..8i+7 of block b; thread tid owns items m0 + u * CONSUMERS + tid.
template <int T>
__device__ __forceinline__ int act_item(int m, int per_tok, int& rem) {
    int t = 0;
    rem = m;
#pragma unroll
    for (int tt = 1; tt < T; ++tt)
        if (rem >= per_tok) { rem -= per_tok; ++t; }
    return t;
}

// Where the quantized activations go: the shared-memory base address of each of
// the CL CTAs of the cluster (CL == 1: this CTA only) and the offsets of the
// quad, scale and 8 * sum(q) arrays, which are the same in every CTA.
template <int CL>
struct ActDst {
    uint32_t base[CL];
    uint32_t q, d, s;
};

template <int CL>
__device__ __forceinline__ void act_put(const uint32_t (&base)[CL], uint32_t off, uint32_t v) {
    if constexpr (CL == 1) {
        st_shared_u32(base[0] + off, v);
    } else {
#pragma unroll
        for (int r = 0; r < CL; ++r) st_cluster_u32(base[r] + off, v);
    }
}

// Quantize items C0 .. C0 + C - 1 (C <= 4) of the NI loaded ones to Q8_0 and
// store them in the quad layout; each step runs across the C items so that the
// latencies of the shuffles, reciprocals and the warp vote overlap.  The codes
// of an item are split into the even word (elements 8i, 8i+2, 8i+4, 8i+6) and
// the odd word (8i+1, ...).  Chunks of at most 4 keep the codes of only 4 items
// live next to the loaded values.  Item u of this thread is m0 + u * CONSUMERS +
// tid; items at or past `end` are not stored.
template <int T, int NI, int C0, int CL>
__device__ __forceinline__ void quantize_chunk(const float (&v)[NI][8], int nb, int np, int m0, int end,
                                               const ActDst<CL>& dst, int tid) {
    constexpr int C = (NI - C0) < 4 ? (NI - C0) : 4;
    const int per_tok = nb * 4;
    float w[C][8], d[C];
#pragma unroll
    for (int u = 0; u < C; ++u) {
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            w[u][e] = v[C0 + u][e];
            amax = fmaxf(amax, fabsf(w[u][e]));
        }
        d[u] = amax;
    }
#pragma unroll
    for (int u = 0; u < C; ++u) d[u] = fmaxf(d[u], __shfl_xor_sync(0xffffffffu, d[u], 1));
#pragma unroll
    for (int u = 0; u < C; ++u) d[u] = scale_q8(fmaxf(d[u], __shfl_xor_sync(0xffffffffu, d[u], 2)));
    int q[C][8];
    quant8n<C, true>(w, d, -127.0f, 127.0f, q);
    uint32_t ye[C], yo[C];
    int sq[C];
#pragma unroll
    for (int u = 0; u < C; ++u) {
        // low bytes of the codes: even elements into ye, odd into yo
        const uint32_t e01 = __byte_perm((uint32_t)q[u][0], (uint32_t)q[u][2], 0x0040);
        const uint32_t e23 = __byte_perm((uint32_t)q[u][4], (uint32_t)q[u][6], 0x0040);
        const uint32_t o01 = __byte_perm((uint32_t)q[u][1], (uint32_t)q[u][3], 0x0040);
        const uint32_t o23 = __byte_perm((uint32_t)q[u][5], (uint32_t)q[u][7], 0x0040);
        ye[u] = d[u] == 0.0f ? 0u : __byte_perm(e01, e23, 0x5410);
        yo[u] = d[u] == 0.0f ? 0u : __byte_perm(o01, o23, 0x5410);
        sq[u] = __dp4a((int)ye[u], 0x01010101, __dp4a((int)yo[u], 0x01010101, 0));
    }
#pragma unroll
    for (int u = 0; u < C; ++u) sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], 1);
#pragma unroll
    for (int u = 0; u < C; ++u) sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], 2);
#pragma unroll
    for (int u = 0; u < C; ++u) {
        const int m = m0 + (C0 + u) * CONSUMERS + tid;
        if (m < end) {
            int rem;
            const int t = act_item<T>(m, per_tok, rem);
            const int b = rem >> 2, i = rem & 3;
            const uint32_t qoff = (uint32_t)(((t * 4 + (b & 1) * 2) * np + (b >> 1)) * 16 + i * 4);
            act_put<CL>(dst.base, dst.q + qoff, ye[u]);
            act_put<CL>(dst.base, dst.q + qoff + (uint32_t)np * 16u, yo[u]);
            if (i == 0) {
                const uint32_t soff = (uint32_t)(t * nb + b) * 4u;
                act_put<CL>(dst.base, dst.d + soff, __float_as_uint(fp16_to_f32(fp16_bits(d[u]))));
                act_put<CL>(dst.base, dst.s + soff, (uint32_t)(8 * sq[u]));
            }
        }
    }
    if constexpr (C0 + C < NI) quantize_chunk<T, NI, C0 + C, CL>(v, nb, np, m0, end, dst, tid);
}

// Quantize NI items per thread of the activations (items m0 + u * CONSUMERS +
// tid below `end`) to Q8_0 into shared memory.  Every load is issued before any
// arithmetic, so their latencies overlap.  m0 is a multiple of 4, so the four
// lanes of a block stay in one aligned group; all 32 lanes of every consumer
// warp must call it.  COHERENT: the activations may have been written earlier by
// the same kernel (another CTA), so they are read from L2 (ld.global.cg) rather
// than through the read-only path.
template <int T, int NI, int CL, bool COHERENT = false>
__device__ __forceinline__ void quantize_acts(const float* __restrict__ x, int ne00, int nb, int np, int m0,
                                              int end, const ActDst<CL>& dst, int tid) {
    const int per_tok = nb * 4;
    float v[NI][8];
#pragma unroll
    for (int u = 0; u < NI; ++u) {
        const int m = m0 + u * CONSUMERS + tid;
        if (m < end) {
            int rem;
            const int t = act_item<T>(m, per_tok, rem);
            const float4* src = reinterpret_cast<const float4*>(x + (int64_t)t * ne00 + (rem >> 2) * QK + (rem & 3) * 8);
            const float4 lo = COHERENT ? __ldcg(src) : __ldg(src), hi = COHERENT ? __ldcg(src + 1) : __ldg(src + 1);
            v[u][0] = lo.x; v[u][1] = lo.y; v[u][2] = lo.z; v[u][3] = lo.w;
            v[u][4] = hi.x; v[u][5] = hi.y; v[u][6] = hi.z; v[u][7] = hi.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[u][e] = 0.0f;
        }
    }
    quantize_chunk<T, NI, 0, CL>(v, nb, np, m0, end, dst, tid);
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

// Integer dot of one pair of Q8_0 weight blocks (17 aligned words, block a at
// byte 0, block b at byte 34): the codes are in element order, so the even and
// odd elements of each group of 8 are gathered with byte permutes to meet the
// activations' even/odd words; signed x signed dp4a, no offset.
struct PairWeights8 {
    float da, db;
    uint32_t qa[8], qb[8];
};

__device__ __forceinline__ PairWeights8 unpack_pair8(const uint32_t (&w)[17]) {
    PairWeights8 p;
    p.da = fp16_to_f32(w[0]);
    p.db = fp16_to_f32(w[8] >> 16);
    // block a's 32 code bytes start at byte 2 of word 0, block b's at word 9
#pragma unroll
    for (int i = 0; i < 8; ++i) p.qa[i] = __byte_perm(w[i], w[i + 1], 0x5432);
#pragma unroll
    for (int i = 0; i < 8; ++i) p.qb[i] = w[9 + i];
    return p;
}

__device__ __forceinline__ int block_dot8(const uint32_t (&q)[8], const uint4& ye, const uint4& yo) {
    int s = 0;
    s = __dp4a((int)__byte_perm(q[0], q[1], 0x6420), (int)ye.x, s);
    s = __dp4a((int)__byte_perm(q[0], q[1], 0x7531), (int)yo.x, s);
    s = __dp4a((int)__byte_perm(q[2], q[3], 0x6420), (int)ye.y, s);
    s = __dp4a((int)__byte_perm(q[2], q[3], 0x7531), (int)yo.y, s);
    s = __dp4a((int)__byte_perm(q[4], q[5], 0x6420), (int)ye.z, s);
    s = __dp4a((int)__byte_perm(q[4], q[5], 0x7531), (int)yo.z, s);
    s = __dp4a((int)__byte_perm(q[6], q[7], 0x6420), (int)ye.w, s);
    s = __dp4a((int)__byte_perm(q[6], q[7], 0x7531), (int)yo.w, s);
    return s;
}

// acc += sum over the pair's two blocks of fp32(d_w * d_x) * isum.  WT selects the
// weight block type: WQ4_0 (18-byte blocks, nibble - 8) or WQ8_0 (34-byte blocks).
template <int WT>
__device__ __forceinline__ float pair_dot(const uint8_t* rowp, int pr, const PairActs& a, float acc) {
    if constexpr (WT == WQ4_0) {
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowp + 36 * pr);
        uint32_t wv[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) wv[i] = wp[i];
        const PairWeights pw = unpack_pair(wv);
        const int ia = block_dot(pw.qa, a.ea, a.oa) - a.s8.x;
        const int ib = block_dot(pw.qb, a.eb, a.ob) - a.s8.y;
        acc = fmaf(pw.da * a.d.x, (float)ia, acc);
        acc = fmaf(pw.db * a.d.y, (float)ib, acc);
    } else {
        const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowp + 68 * pr);
        uint32_t wv[17];
#pragma unroll
        for (int i = 0; i < 17; ++i) wv[i] = wp[i];
        const PairWeights8 pw = unpack_pair8(wv);
        const int ia = block_dot8(pw.qa, a.ea, a.oa);
        const int ib = block_dot8(pw.qb, a.eb, a.ob);
        acc = fmaf(pw.da * a.d.x, (float)ia, acc);
        acc = fmaf(pw.db * a.d.y, (float)ib, acc);
    }
    return acc;
}

// What the write of one output applies: the bias of its row (loaded ahead by the
// caller), then the activation.
__device__ __forceinline__ float output_epilogue(float v, bool has_bias, float bias, int act) {
    if (has_bias) v = __fadd_rn(v, bias);
    if (act == Q4Q_ACT_GELU) v = gelu_f32(v);
    return v;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(CONSUMERS) : "memory");
}

// The body of every GEMV kernel.  WT: weight block type.  T tokens; LPR lanes per
// row; PPL > 0: the lane's PPL block pairs of activations are held in registers
// for the whole kernel (T == 1), PPL == 0: read from shared memory for every row.
// CL > 1: the grid is made of clusters of CL CTAs that split the activation
// quantization: each quantizes 1/CL of the blocks and writes the result into the
// shared memory of every CTA of its cluster, so each SM loads only 1/CL of the
// fp32 activations from L2.  DUAL: two weight matrices of the same shape (w and
// w2) are streamed side by side, each unit's rows of both in one stage, and every
// output is silu(w x) * (w2 x) (the SwiGLU of the Llama MLP).  EPI: every output
// is the bias / activation epilogue of p applied to w x (the plain kernel carries
// no epilogue code at all).  GROUP: the units
// run over up to GROUP_MAX matrices of rows that share the activations (the q, k
// and v projections of one input), each written to its own output.
template <int WT, int T, int LPR, int PPL, int CL, int MODE>
__device__ __forceinline__ void gemv_body(const uint8_t* __restrict__ w, const uint8_t* __restrict__ w2,
                                          const float* __restrict__ x, float* __restrict__ dst,
                                          const GemvParams& p) {
    static_assert(PPL == 0 || T == 1, "register-resident activations are for one token");
    constexpr bool DUAL = MODE == M_DUAL;
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
    if constexpr (CL > 1) {
        // first cluster barrier phase: every CTA of the cluster has started, so
        // its shared memory may be written by its peers from here on
        cluster_arrive();
        cluster_wait();
    }
    // the next kernel on the stream may start its own set-up now; it still waits
    // for this grid to finish before it touches memory this grid writes
    pdl_trigger();

    if (warp == CONSUMERS / 32) {
        // ---------------- producer: stream weight units through the ring
        if (lane == 0) {
            // second phase: the producer publishes nothing, it arrives at once (the
            // other lanes of this warp have exited and are not waited for)
            if constexpr (CL > 1) cluster_arrive();
            int k = 0;
            for (int u = blockIdx.x; u < p.n_units; u += grid, ++k) {
                const int s = k % p.S;
                if (k >= p.S) {
                    const uint32_t bar = empty0 + 8 * s, par = ((k / p.S) + 1) & 1;
                    const bool ok = mbar_wait_until(bar, par, abort_flag, p.limit_ns);
                    if (!ok) {
                        if (!*abort_flag) record_error(&g_gemv_status, DEV_TIMEOUT);
                        *abort_flag = 1;
                        break;
                    }
                }
                // test only: CTA 0 leaves out its first unit (no expected bytes, no copy), so
                // that stage never completes and the consumers' bounded waits run out
                if (p.fault && k == 0 && blockIdx.x == 0) continue;
                const UnitRows ur = unit_rows<MODE>(p, w, dst, u);
                const int r0 = ur.r0;
                const int nr = min(p.G, ur.rows - r0);
                const uint32_t bytes = (uint32_t)nr * (uint32_t)p.row_bytes;
                mbar_arrive_expect_tx(full0 + 8 * s, DUAL ? 2 * bytes : bytes);
                bulk_g2s(smem_u32(stages + (size_t)s * p.stage_bytes), ur.w + (int64_t)r0 * p.row_bytes, bytes,
                         full0 + 8 * s);
                if constexpr (DUAL)
                    bulk_g2s(smem_u32(stages + (size_t)s * p.stage_bytes + p.half_off),
                             w2 + (int64_t)r0 * p.row_bytes, bytes, full0 + 8 * s);
            }
            // let every copy issued land before the CTA can exit: consumers that gave up
            // no longer wait for them (the unit a test leaves out never lands)
            for (int k2 = max(0, k - p.S); k2 < k; ++k2)
                if (!(p.fault && k2 == 0 && blockIdx.x == 0))
                    mbar_wait_bounded(full0 + 8 * (k2 % p.S), (uint32_t)((k2 / p.S) & 1), p.limit_ns);
        }
        return;
    }

    // ---------------- consumers: activations first (they may come from the previous kernel)
    constexpr int RP = CONSUMERS / LPR;     // rows processed side by side
    const int rr = tid / LPR, sl = tid % LPR;
    // epilogue: the biases of the first two units' first rows are loaded before the
    // wait for the previous kernel, like the weights (resident model parameters), so
    // that small matrices, whose weights are in shared memory by then, do not wait
    // for them after the dot
    float bias_pre0 = 0.0f, bias_pre1 = 0.0f;
    if constexpr (MODE == M_EPI) {
        if (p.bias && sl == 0) {
            const int u0 = blockIdx.x, u1 = blockIdx.x + grid;
            if (u0 < p.n_units) {
                const UnitRows a = unit_rows<MODE>(p, w, dst, u0);
                if (rr < min(p.G, a.rows - a.r0)) bias_pre0 = __ldg(p.bias + a.r0 + rr);
            }
            if (u1 < p.n_units) {
                const UnitRows b = unit_rows<MODE>(p, w, dst, u1);
                if (rr < min(p.G, b.rows - b.r0)) bias_pre1 = __ldg(p.bias + b.r0 + rr);
            }
        }
    }
    pdl_wait();
    {
        // this CTA's share: blocks [f0, f1) of the T * nb blocks (token-major)
        const int nbt = T * p.nb;
        const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
        const int f0 = (int)(((int64_t)rank * nbt) / CL), f1 = (int)(((int64_t)(rank + 1) * nbt) / CL);
        ActDst<CL> ad;
        const uint32_t sbase = smem_u32(smem);
#pragma unroll
        for (int r = 0; r < CL; ++r) ad.base[r] = CL > 1 ? mapa_shared(sbase, (uint32_t)r) : sbase;
        ad.q = (uint32_t)p.act_off;
        ad.d = (uint32_t)p.dy_off;
        ad.s = (uint32_t)p.sy_off;
        if (PPL > 0) {
            // one token, nb = 2 * PPL * LPR blocks, at most ceil(nb / CL) of them
            // here (4 items each): all in one batch
            constexpr int NBMAX = (2 * (PPL > 0 ? PPL : 1) * LPR + CL - 1) / CL;
            constexpr int NI = (4 * NBMAX + CONSUMERS - 1) / CONSUMERS;
            quantize_acts<T, NI, CL>(x, p.ne00, p.nb, p.np, 4 * f0, 4 * f1, ad, tid);
        } else {
            constexpr int U = 3;
            for (int m0 = 4 * f0; m0 < 4 * f1; m0 += CONSUMERS * U)
                quantize_acts<T, U, CL>(x, p.ne00, p.nb, p.np, m0, 4 * f1, ad, tid);
        }
    }
    if constexpr (CL > 1) {
        // second phase: every CTA's share is in every CTA's shared memory
        cluster_arrive();
        cluster_wait();
    } else {
        consumer_sync();
    }

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
        const UnitRows ur = unit_rows<MODE>(p, w, dst, u);
        const int r0 = ur.r0;
        const int nr = min(p.G, ur.rows - r0);
        // epilogue: the bias of this lane group's first row (loaded ahead for the first
        // two units, else before the wait for the weights, so its latency hides behind theirs)
        float bias_cur = 0.0f;
        if constexpr (MODE == M_EPI) {
            if (k == 0) bias_cur = bias_pre0;
            else if (k == 1) bias_cur = bias_pre1;
            else if (p.bias && sl == 0 && rr < nr) bias_cur = __ldg(p.bias + r0 + rr);
        }
        {
            const uint32_t bar = full0 + 8 * s, par = (uint32_t)((k / p.S) & 1);
            int ok = 1;
            if (lane == 0) {
                const bool got = mbar_wait_until(bar, par, abort_flag, p.limit_ns);
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
        for (int pass = 0; pass < passes; ++pass) {
            const int j = rr + pass * RP;
            const bool valid = j < nr;
            float bias_next = 0.0f;      // the next pass's bias, in flight during this pass's dot
            if constexpr (MODE == M_EPI)
                if (p.bias && sl == 0 && j + RP < nr) bias_next = __ldg(p.bias + r0 + j + RP);
            float acc[T], acc2[T];
#pragma unroll
            for (int t = 0; t < T; ++t) acc[t] = acc2[t] = 0.0f;
            if (valid) {
                const uint8_t* rowp = stage + (size_t)j * p.row_bytes;
                const uint8_t* rowp2 = rowp + p.half_off;
                if (PPL > 0) {
#pragma unroll
                    for (int kk = 0; kk < (PPL > 0 ? PPL : 1); ++kk) {
                        acc[0] = pair_dot<WT>(rowp, sl + kk * LPR, areg[kk], acc[0]);
                        if constexpr (DUAL) acc2[0] = pair_dot<WT>(rowp2, sl + kk * LPR, areg[kk], acc2[0]);
                    }
                } else {
                    for (int kk = 0; kk < ppl; ++kk) {
                        const int pr = sl + kk * LPR;
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            const PairActs a = load_pair_acts(quads, dy, sy8, p.np, p.nb, t, pr);
                            acc[t] = pair_dot<WT>(rowp, pr, a, acc[t]);
                            if constexpr (DUAL) acc2[t] = pair_dot<WT>(rowp2, pr, a, acc2[t]);
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < T; ++t) {
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) {
                    acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
                    if constexpr (DUAL) acc2[t] += __shfl_xor_sync(0xffffffffu, acc2[t], off);
                }
            }
            if (valid && sl == 0) {
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    float v;
                    if constexpr (DUAL) v = swiglu_f32(acc[t], acc2[t]);
                    else if constexpr (MODE == M_EPI) v = output_epilogue(acc[t], p.bias != nullptr, bias_cur, p.act);
                    else v = acc[t];
                    ur.dst[(int64_t)t * ur.rows + r0 + j] = v;
                }
            }
            bias_cur = bias_next;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
}


// The kernels share one body and one signature (w2 is unused unless dual; the
// group kernel takes its pointers from p.grp).  With one or two register-resident
// activation pairs a lane (K <= 4096 at one token) three CTAs fit in an SM's registers
// (69 of them a thread, none spilled), so that a decode chain's next kernel can start a
// CTA beside this one's two and prefetch its weights (see plan_gemv).
constexpr int gemv_min_ctas(int ppl) { return (ppl >= 1 && ppl <= 2) ? 3 : (ppl <= 3 ? 2 : 1); }

template <int T, int LPR, int PPL, int CL>
__global__ void __launch_bounds__(THREADS, gemv_min_ctas(PPL))
gemv_q4_0_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ w2, const float* __restrict__ x,
                 float* __restrict__ dst, const GemvParams p) {
    gemv_body<WQ4_0, T, LPR, PPL, CL, M_SINGLE>(w, w2, x, dst, p);
}

template <int T, int LPR, int PPL, int CL>
__global__ void __launch_bounds__(THREADS, gemv_min_ctas(PPL))
gemv_q4_0_swiglu_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ w2, const float* __restrict__ x,
                        float* __restrict__ dst, const GemvParams p) {
    gemv_body<WQ4_0, T, LPR, PPL, CL, M_DUAL>(w, w2, x, dst, p);
}

template <int T, int LPR, int PPL, int CL>
__global__ void __launch_bounds__(THREADS, gemv_min_ctas(PPL))
gemv_q8_0_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ w2, const float* __restrict__ x,
                 float* __restrict__ dst, const GemvParams p) {
    gemv_body<WQ8_0, T, LPR, PPL, CL, M_SINGLE>(w, w2, x, dst, p);
}

template <int T, int LPR, int PPL, int CL>
__global__ void __launch_bounds__(THREADS, gemv_min_ctas(PPL))
gemv_q4_0_epi_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ w2, const float* __restrict__ x,
                     float* __restrict__ dst, const GemvParams p) {
    gemv_body<WQ4_0, T, LPR, PPL, CL, M_EPI>(w, w2, x, dst, p);
}

template <int T, int LPR, int PPL, int CL>
__global__ void __launch_bounds__(THREADS, gemv_min_ctas(PPL))
gemv_q4_0_group_kernel(const uint8_t* __restrict__ w, const uint8_t* __restrict__ w2, const float* __restrict__ x,
                       float* __restrict__ dst, const GemvParams p) {
    gemv_body<WQ4_0, T, LPR, PPL, CL, M_GROUP>(w, w2, x, dst, p);
}

using GemvKernelFn = void (*)(const uint8_t*, const uint8_t*, const float*, float*, const GemvParams);

template <int WT, int MODE, int T, int LPR, int PPL, int CL>
GemvKernelFn gemv_kernel_fn() {
    static_assert(MODE == M_SINGLE || WT == WQ4_0, "the dual, epilogue and group kernels are built for Q4_0");
    if constexpr (MODE == M_DUAL) return gemv_q4_0_swiglu_kernel<T, LPR, PPL, CL>;
    else if constexpr (MODE == M_EPI) return gemv_q4_0_epi_kernel<T, LPR, PPL, CL>;
    else if constexpr (MODE == M_GROUP) return gemv_q4_0_group_kernel<T, LPR, PPL, CL>;
    else if constexpr (WT == WQ8_0) return gemv_q8_0_kernel<T, LPR, PPL, CL>;
    else return gemv_q4_0_kernel<T, LPR, PPL, CL>;
}

// Pointers of one launch.
struct GemvArgs {
    const uint8_t* w;
    const uint8_t* w2;      // dual-weight kernel only
    const float* x;
    float* dst;
    const float* bias;      // may be null
    int act;
    GemvGroup grp;          // group kernel only
};

struct GemvPlan {
    GemvParams p;
    int lpr;
    int ppl_reg;       // > 0: activations in registers
    int grid;          // CTAs without clusters
    int grid_cap;      // CTAs the device holds at once (grid = min(units, grid_cap))
    int cl;            // cluster size to try (1 or 2)
    int sms;
    size_t smem;
};

// mats = 2: two matrices streamed side by side (dual-weight kernel); a unit's
// rows of both share one stage, so every size below counts both.
bool plan_gemv(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info, GemvPlan* plan,
               int block_bytes = Q4_0_BYTES, int mats = 1) {
    if (ne11 < 1 || ne11 > 7 || ne00 % 256 != 0 || ne00 > (1 << 20) || ne01 <= 0 || ne01 >= (1ll << 31))
        return false;
    GemvParams& p = plan->p;
    p.ne00 = (int)ne00;
    p.nb = (int)(ne00 / QK);
    p.np = p.nb / 2;
    p.ne01 = (int)ne01;
    p.row_bytes = p.nb * block_bytes;
    const int64_t urow = (int64_t)mats * p.row_bytes;   // bytes a unit stages per row
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
    const int64_t wbytes = ne01 * urow;
    const bool two_per_sm = plan->ppl_reg == 0 || plan->ppl_reg <= 3;
    int64_t G, S, stage;
    bool small = false;
    if (two_per_sm && wbytes <= 96 * 1024 * sms) {
        // Small matrix: one CTA per SM holds every unit it owns in flight from the
        // start (about two units each), and leaves room on the SM for the next
        // kernel's CTA, which can then prefetch its own weights under PDL.
        G = std::max<int64_t>(1, (ne01 + 2 * sms - 1) / (2 * sms));
        // Where one unit per CTA still fits the RP row groups, take it: the busiest CTA
        // then runs one dot pass instead of two, and under PDL the weights are in shared
        // memory already, so only that pass is on the dependency chain (Llama-3-8B k / v:
        // 7-row units, 147 of them, instead of 256 units of 4 rows).
        const int64_t g1 = (ne01 + sms - 1) / sms;
        if (g1 <= RP) G = std::max<int64_t>(1, g1);
        const int64_t units = (ne01 + G - 1) / G;
        S = std::min<int64_t>(MAX_STAGES, (units + sms - 1) / sms);
        stage = ((G * urow) + 127) / 128 * 128;
        small = head + act_bytes + S * stage <= std::min<int64_t>(limit, 110 * 1024);
    }
    if (!small) {
        // rows per unit: aim at ~16 KB stages, but keep >= 2 units per SM when the matrix
        // allows.  Small stages let two CTAs share an SM with >= 3 stages each (16
        // consumer warps): K = 4096 rows of 2304 bytes stage 8 at a time; timed on the
        // Llama-3-8B decode set, 32 KB stages (one CTA per SM, 6 stages) were 1.5% slower.
        // With one or two register-resident activation pairs a lane the ring stops at 4
        // stages (77 KB a CTA at K = 4096): two such CTAs leave room on the SM for a small
        // matrix's CTA (the next q projection of a decode chain, 68 KB), which then
        // prefetches its weights under PDL, while a third CTA of the same kernel does not
        // fit, so a freed SM never takes three of them.  Timed against 5 stages (same box,
        // Llama decode step as PDL-chained graphs): 86.8 -> 86.0 us a step, the lm_head
        // alone 50.5 -> 47.4 us.
        const int64_t rp_bytes = (int64_t)RP * urow;
        G = RP * std::max<int64_t>(1, (16384 + rp_bytes / 2) / rp_bytes);
        while (G > 8 && (ne01 + G - 1) / G < 2 * sms) G = std::max<int64_t>(8, G / 2);
        G = std::min<int64_t>(G, ne01);
        const auto stages_for = [&](int64_t g) {
            stage = ((g * urow) + 127) / 128 * 128;
            int64_t n = 0;
            if (two_per_sm) n = (std::min<int64_t>(limit, 110 * 1024) - head - act_bytes) / stage;
            if (two_per_sm && plan->ppl_reg >= 1 && plan->ppl_reg <= 2) n = std::min<int64_t>(n, 4);
            if (n < 3) n = (limit - head - act_bytes) / stage;
            return n;
        };
        S = stages_for(G);
        // Very long rows (a Q8_0 row of K = 14336 is 15 KB) or many tokens' activations
        // leave room for fewer than two stages of RP rows: stage fewer rows (the row
        // groups past G stay idle) rather than give the GEMV up.
        while (S < 2 && G > 1) {
            G = std::max<int64_t>(1, G / 2);
            S = stages_for(G);
        }
        if (S < 2) return false;
        // Balance: the persistent CTAs take units round-robin, so the busiest one streams
        // ceil(units / CTAs) units.  Among unit sizes from G/2 to G that keep the same CTAs
        // per SM, take the one that leaves it the fewest rows, if that saves at least 5%
        // (the 14336 -> 4096 down projection on 152 SMs: 512 units of 8 rows, 4 on the
        // busiest CTA, 32 rows; 586 units of 7 rows, 28 rows).
        const auto per_sm_of = [&](int64_t s, int64_t st) {
            return (two_per_sm && head + act_bytes + std::min<int64_t>(s, MAX_STAGES) * st <= 113 * 1024) ? 2 : 1;
        };
        const int64_t cap = sms * per_sm_of(S, stage);
        const auto busiest_rows = [&](int64_t g) { return ((ne01 + g - 1) / g + cap - 1) / cap * g; };
        int64_t best = G, best_rows = busiest_rows(G);
        for (int64_t g = G - 1; g >= std::max<int64_t>(1, G / 2); --g) {
            const int64_t sg = stages_for(g);
            if (sg < 2 || sms * per_sm_of(sg, stage) != cap) continue;
            if (busiest_rows(g) * 20 <= busiest_rows(G) * 19 && busiest_rows(g) < best_rows) {
                best = g;
                best_rows = busiest_rows(g);
            }
        }
        G = best;
        S = stages_for(G);
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
    p.half_off = (int)(G * p.row_bytes);
    p.act = Q4Q_ACT_NONE;
    p.bias = nullptr;
    p.grp = GemvGroup{};
    p.limit_ns = WAIT_LIMIT_NS;
    p.fault = 0;
    plan->smem = (size_t)(head + act_bytes + S * stage);
    plan->lpr = lpr;
    const int per_sm = (!small && plan->smem <= 113 * 1024 && two_per_sm) ? 2 : 1;
    plan->grid_cap = (int)(sms * per_sm);
    plan->grid = (int)std::min<int64_t>(p.n_units, sms * per_sm);
    plan->sms = (int)sms;
    // Splitting the activation quantization over a pair of CTAs pays only where
    // each SM would otherwise load tens of KB of fp32 activations: below that the
    // pair's barrier (each CTA waits for the slower one) costs more than it saves.
    // The dual-weight kernel is built without pairs.
    plan->cl = (mats == 1 && ne11 * ne00 >= CLUSTER_MIN_X) ? 2 : 1;
    return true;
}

template <int CL>
cudaLaunchConfig_t gemv_config(const GemvPlan& plan, int grid, cudaStream_t stream, bool pdl,
                               cudaLaunchAttribute (&attr)[2]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (CL > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = CL;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cfg;
}

// Raise the kernel's opt-in shared-memory size (once per device and size), and
// return how many of its CTAs fit on the device at once in clusters of CL
// (cached per device and shared-memory size; 0 if the query fails).
template <int WT, int MODE, int T, int LPR, int PPL, int CL>
int gemv_prepare(const GemvPlan& plan, int device) {
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, int> resident;
    static int configured[64] = {};
    const GemvKernelFn kern = gemv_kernel_fn<WT, MODE, T, LPR, PPL, CL>();
    std::lock_guard<std::mutex> lock(mu);
    if ((int)plan.smem > configured[device]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        configured[device] = (int)plan.smem;
    }
    const auto key = std::make_pair(device, plan.smem);
    auto it = resident.find(key);
    if (it != resident.end()) return it->second;
    int n = 0;
    if (CL == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, plan.smem) == cudaSuccess)
            n = per_sm * plan.sms;
    } else {
        cudaLaunchAttribute attr[2];
        const cudaLaunchConfig_t cfg = gemv_config<CL>(plan, CL, nullptr, false, attr);
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess) n = clusters * CL;
    }
    (void)cudaGetLastError();
    resident[key] = n;
    return n;
}

template <int WT, int MODE, int T, int LPR, int PPL, int CL>
q4q_status gemv_launch_cl(const GemvPlan& plan, int grid, const GemvArgs& a, cudaStream_t stream, bool pdl) {
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = gemv_config<CL>(plan, grid, stream, pdl, attr);
    GemvParams p = plan.p;
    p.bias = a.bias;
    p.act = a.act;
    if constexpr (MODE == M_GROUP) p.grp = a.grp;
    if (cudaLaunchKernelEx(&cfg, gemv_kernel_fn<WT, MODE, T, LPR, PPL, CL>(), a.w, a.w2, a.x, a.dst, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4Q_ERR_CUDA;
    }
    return launch_status();
}

// CTAs of a launch in clusters of cl: every unit gets a CTA where the device
// holds that many at once, rounded to whole clusters.
inline int cluster_grid(int n_units, int resident, int cl) {
    const int want = (n_units + cl - 1) / cl * cl;
    return std::min(want, resident / cl * cl);
}

template <int WT, int MODE, int T, int LPR, int PPL>
q4q_status launch_gemv_t(const GemvPlan& plan, const GemvArgs& a, cudaStream_t stream, int device, bool pdl) {
    if (device < 0 || device >= 64) return Q4Q_ERR_CUDA;
    // Clusters only where they keep (nearly) every planned CTA resident.
    const int need = plan.grid - plan.grid / 16;
    if constexpr (MODE != M_DUAL) {
        if (plan.cl >= 2) {
            const int g = cluster_grid(plan.p.n_units, gemv_prepare<WT, MODE, T, LPR, PPL, 2>(plan, device), 2);
            if (g >= 2 && g >= need) return gemv_launch_cl<WT, MODE, T, LPR, PPL, 2>(plan, g, a, stream, pdl);
        }
    }
    if (gemv_prepare<WT, MODE, T, LPR, PPL, 1>(plan, device) <= 0) return Q4Q_ERR_CUDA;
    return gemv_launch_cl<WT, MODE, T, LPR, PPL, 1>(plan, plan.grid, a, stream, pdl);
}

template <int WT, int MODE, int T, int LPR>
q4q_status launch_gemv_ppl(const GemvPlan& plan, const GemvArgs& a, cudaStream_t stream, int device, bool pdl) {
    if (T == 1) {
        switch (plan.ppl_reg) {
            case 1: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 1 : 0)>(plan, a, stream, device, pdl);
            case 2: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 2 : 0)>(plan, a, stream, device, pdl);
            case 3: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 3 : 0)>(plan, a, stream, device, pdl);
            case 4: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 4 : 0)>(plan, a, stream, device, pdl);
            case 5: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 5 : 0)>(plan, a, stream, device, pdl);
            case 6: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 6 : 0)>(plan, a, stream, device, pdl);
            case 7: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 7 : 0)>(plan, a, stream, device, pdl);
            case 8: return launch_gemv_t<WT, MODE, T, LPR, (T == 1 ? 8 : 0)>(plan, a, stream, device, pdl);
            default: break;
        }
    }
    return launch_gemv_t<WT, MODE, T, LPR, 0>(plan, a, stream, device, pdl);
}

template <int WT, int MODE, int T>
q4q_status launch_gemv_lpr(const GemvPlan& plan, const GemvArgs& a, cudaStream_t stream, int device, bool pdl) {
    switch (plan.lpr) {
        case 32: return launch_gemv_ppl<WT, MODE, T, 32>(plan, a, stream, device, pdl);
        case 16: return launch_gemv_ppl<WT, MODE, T, 16>(plan, a, stream, device, pdl);
        case 8:  return launch_gemv_ppl<WT, MODE, T, 8>(plan, a, stream, device, pdl);
        default: return launch_gemv_ppl<WT, MODE, T, 4>(plan, a, stream, device, pdl);
    }
}


// One launch of the GEMV variant <WT, MODE> for ne11 = 1..7 tokens.
template <int WT, int MODE>
q4q_status launch_gemv(const GemvPlan& plan, int64_t ne11, const GemvArgs& a, cudaStream_t stream, int device,
                       bool pdl) {
    switch (ne11) {
        case 1: return launch_gemv_lpr<WT, MODE, 1>(plan, a, stream, device, pdl);
        case 2: return launch_gemv_lpr<WT, MODE, 2>(plan, a, stream, device, pdl);
        case 3: return launch_gemv_lpr<WT, MODE, 3>(plan, a, stream, device, pdl);
        case 4: return launch_gemv_lpr<WT, MODE, 4>(plan, a, stream, device, pdl);
        case 5: return launch_gemv_lpr<WT, MODE, 5>(plan, a, stream, device, pdl);
        case 6: return launch_gemv_lpr<WT, MODE, 6>(plan, a, stream, device, pdl);
        default: return launch_gemv_lpr<WT, MODE, 7>(plan, a, stream, device, pdl);
    }
}

// Read and clear this translation unit's device status word.
inline unsigned int take_gemv_status_word() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemv_status, sizeof(v)) != cudaSuccess) return Q4Q_ERR_CUDA;
    if (v) cudaMemcpyToSymbol(g_gemv_status, &z, sizeof(z));
    return v;
}

}  // namespace
}  // namespace q4q
