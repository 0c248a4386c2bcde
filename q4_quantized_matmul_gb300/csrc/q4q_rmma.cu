// q4q_rmma.cu -- Q4_0 x Q8_0 mul_mat for a few tokens (2 <= ne11 <= 32) with warp-level MMA.
//
// The operation is the one every path of the library computes ("llama.cpp 深度解读"
// §3 "量化矩阵乘法 — 核心算子"):
//   dst[n][m] = sum_b fp32(d_w[m][b] * d_x[n][b]) * S_b[m][n],
//   S_b[m][n] = sum_{k in block b} (nibble[m][k] - 8) * q[n][k]     (exact integer).
//
// With a few tokens the work is bound by reading every weight byte once: 2 * ne11 ops
// per weight against 0.5625 bytes, a few dozen ops per byte, far below the tensor
// cores' ridge point.  What decides the speed is how few instructions turn a streamed
// byte into its share of the block dots.  On the tcgen05 path one thread issues all of
// a CTA's MMAs, and at N <= 64 each 128 x N x 16 MMA holds that thread for about 70-90
// cycles whatever N is (clock64 stamps around the issuing thread), which keeps the CTA
// well below its share of HBM bandwidth.  Here every consumer warp unpacks its own rows
// into registers and issues mma.sync.m16n8k16 on them, and the warps of a CTA, and the
// CTAs of an SM, run independently.
//
// Exact integer dots from fp16 MMA.  A nibble n masked into the low bits of an fp16
// word is the subnormal n * 2^-24 (no implicit leading one), so a 32-bit word of 8
// nibbles becomes four fp16 pairs with five bit operations: {e0,e4} and {e2,e6} as
// n * 2^-24, {e1,e5} and {e3,e7} (the high nibbles of each byte, left where they are)
// as 16 n * 2^-24.  The activation codes q (|q| <= 127) are stored as fp16 q for even
// elements and q / 16 (exact, a power-of-two scaling) for odd ones, so every product
// is n q 2^-24 exactly, and the fp32 sum of a block is D = 2^-24 sum_k n_k q_k with
// |sum| <= 32 * 15 * 127 < 2^24: exact.  (mma.sync takes fp16 subnormals as they
// are; an all-pairs check of such operands against exact dots found no difference.)
// The -8 offset of the nibbles enters as the MMA's C operand, -8 sum_k q_k * 2^-24 (the
// activation kernel supplies it per block and token), so the block's MMAs leave
// 2^-24 S_b exactly (every partial sum is an integer times 2^-24 below 1 in magnitude);
// the activation scale is stored as d_x * 2^24, and fp32(d_w * d_x * 2^24) is exactly
// fp32(d_w d_x) * 2^24 because the product of two fp16 values is never an fp32
// subnormal.  Per block and token pair that leaves one packed multiply and one packed
// FMA into the running sums.
//
// Roles and layout (persistent CTAs, two per SM; 4 consumer warps + 1 producer warp):
//  * A work item is one 128-row tile and one K split of it; CTA c takes items c,
//    c + grid, ...  The producer streams the items' 256-K stages into an S-deep ring
//    with no break between items.  The kernel is launched with programmatic dependent
//    launch behind the activation kernel: the producer starts the weight copies of
//    its first S stages, then waits for the activations.
//  * A stage holds the tile's raw Q4_0 bytes (2-D TMA box of 144 bytes x 128 rows:
//    rows are 36 words apart, so the 8 rows x 4 words a warp loads at once fall in 32
//    distinct banks), the activation codes of its 8 blocks ([block][8 NG tokens][32]
//    fp16: 64-byte token rows, conflict-free 16-byte loads) and per block and token
//    pair {2^24 d_x, 2^24 d_x', -8 sum q 2^-24, -8 sum q' 2^-24}.  The activation kernel
//    writes codes and quads in exactly that order, so each stage's share is two
//    contiguous 1-D bulk copies (three copies a stage in all).  Each 8-element group of
//    codes is stored in the order [0,4,1,5,2,6,3,7].
//  * Consumer warp w owns rows 32w .. 32w+31 (two m16 tiles).  Lane (g, t) =
//    (lane / 4, lane % 4) takes word t of each block's 16 nibble bytes for rows g,
//    g+8, g+16, g+24; the four fp16 pairs it unpacks to are exactly the A fragments
//    of two k16 MMAs against codes in the order above (the dot product does not
//    depend on the order of K).
//  * Per block the two MMAs start from the offset term; fp32(d_w d_x) * S_b is added to
//    the running sums (packed f32x2 operations).
//  * K splits: each warp writes its partial sums to the workspace, and a reduce kernel,
//    launched behind the GEMM with programmatic dependent launch, adds the splits in
//    split order (one thread per 4 outputs) and writes dst: deterministic.
// Every wait is bounded and follows the abort protocol of q4q_mma.cu (the call's abort
// word sits in the workspace and is zeroed by the activation kernel), with this file's
// own status word.  After the roles split no barrier spans more than one warp, so a
// warp that gives up never leaves another one waiting for it.
#include <algorithm>
#include <atomic>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

__device__ unsigned int g_rmma_status = 0;

constexpr int RM = 128;                    // weight rows per tile
constexpr int KST = 256;                   // K per stage: 8 blocks
constexpr int RAW_ROW = 8 * Q4_0_BYTES;    // 144 bytes of one row per stage
constexpr int RAW_BYTES = RM * RAW_ROW;    // 18432
constexpr int CWARPS = 4;                  // consumer warps, 32 rows each
constexpr int THREADS = (CWARPS + 1) * 32;
constexpr int CTAS_PER_SM = 2;
constexpr int CTRL_WORDS = 64;             // the call's control area in the workspace (word 0: abort word)
constexpr int MAX_TOKENS = 32;
constexpr int ACT_THREADS = 256;

template <int NG>
struct RCfg {
    static constexpr int NTOK = 8 * NG;             // token columns (ne11 padded to MMA n8 tiles)
    static constexpr int B_BLOCK = NTOK * 64;       // one block's activation codes: NTOK x 32 fp16
    static constexpr int B_BYTES = 8 * B_BLOCK;
    static constexpr int DS_BLOCK = NTOK / 2 * 16;  // one block's {dx, dx', m, m'} for NTOK tokens
    static constexpr int DS_BYTES = 8 * DS_BLOCK;
    static constexpr int STAGE_TX = RAW_BYTES + B_BYTES + DS_BYTES;
    static constexpr int S = NG >= 3 ? 3 : 4;       // ring depth: two CTAs fit in one SM's shared memory
    static constexpr int OFF_B = S * RAW_BYTES;     // every slot stays 128-byte aligned
    static constexpr int OFF_DS = OFF_B + S * B_BYTES;
    static constexpr int OFF_BAR = OFF_DS + S * DS_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + 2 * S * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 128;   // + alignment slack
    static constexpr int ACC = 2 * NG * 4;          // partial sums per lane
};

struct RParams {
    const uint8_t* bmat;    // activation codes, [nb][8 NG][32] fp16 (one stage = 8 blocks, contiguous)
    const uint8_t* ds;      // scale quads, [nb][4 NG][4] fp32 (one stage contiguous)
    int M, N;               // weight rows, tokens
    int nst;                // K stages (ne00 / 256)
    int tiles;              // 128-row tiles
    int whole;              // tiles 0 .. whole-1 run whole (one item each, written to dst)
    int splits;             // the other tiles run as `splits` items each (partial sums)
    int items;              // whole + (tiles - whole) * splits
    float* dst;             // [N][M]
    float* part;            // split tiles: [tile - whole][split][warp][lane][ACC] partial sums
    unsigned int* abort_word;
    uint64_t limit_ns;      // bound of every wait
    int fault;              // test only: 1 = CTA 0 leaves out the copies of its first stage
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

// d = A * B + c, m16n8k16, fp16 operands, fp32 accumulators (row-major A, column-major
// B); c is the pair (c0, c1) for both row halves of the fragment
__device__ __forceinline__ void mma_16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1, float c0, float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %10, %11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}

// d += A * B
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Nibble word (element e at bits 4e) -> the fp16 pairs {e0,e4}, {e1,e5}, {e2,e6},
// {e3,e7}: low nibbles as n * 2^-24, high nibbles as 16 n * 2^-24 (fp16 subnormals).
__device__ __forceinline__ uint4 nibbles_to_subnormals(uint32_t q) {
    const uint32_t q8 = q >> 8;
    return make_uint4(q & 0x000F000Fu, q & 0x00F000F0u, q8 & 0x000F000Fu, q8 & 0x00F000F0u);
}

// One K block for the warp's 32 rows and all token groups.  qw[r] is the lane's nibble
// word of row g + 8r, dw[r] that row's block scale; bblk / dsb are the block's
// activation codes and {2^24 dx, 2^24 dx', m, m'} quads in shared memory.  acc[mt][tg]
// holds the packed pairs (row g + 16mt, tokens 2t, 2t+1) and (row g + 16mt + 8, same
// tokens) of token group tg.
template <int NG>
__device__ __forceinline__ void block_mma(uint64_t (&acc)[2][NG][2], const uint32_t (&qw)[4], const float (&dw)[4],
                                          const uint8_t* bblk, const uint8_t* dsb, int g, int t) {
    uint4 h[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) h[r] = nibbles_to_subnormals(qw[r]);
#pragma unroll
    for (int tg = 0; tg < NG; ++tg) {
        const uint4 bv = *reinterpret_cast<const uint4*>(bblk + (8 * tg + g) * 64 + 16 * t);
        const float4 ds = *reinterpret_cast<const float4*>(dsb + (4 * tg + t) * 16);
        const uint64_t dxx = pack2(ds.x, ds.y);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            float c[4];   // 2^-24 S_b, exact
            mma_16816_c(c, h[2 * mt].x, h[2 * mt + 1].x, h[2 * mt].y, h[2 * mt + 1].y, bv.x, bv.y, ds.z, ds.w);
            mma_16816(c, h[2 * mt].z, h[2 * mt + 1].z, h[2 * mt].w, h[2 * mt + 1].w, bv.z, bv.w);
            acc[mt][tg][0] = ffma2(fmul2(pack2(dw[2 * mt], dw[2 * mt]), dxx), pack2(c[0], c[1]), acc[mt][tg][0]);
            acc[mt][tg][1] = ffma2(fmul2(pack2(dw[2 * mt + 1], dw[2 * mt + 1]), dxx), pack2(c[2], c[3]), acc[mt][tg][1]);
        }
    }
}

template <int NG>
__device__ __forceinline__ void store_outputs(const RParams& p, const float (&v)[RCfg<NG>::ACC], int row0, int t) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int tg = 0; tg < NG; ++tg)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = row0 + 16 * mt + 8 * (e >> 1);
                const int n = 8 * tg + 2 * t + (e & 1);
                if (m < p.M && n < p.N) p.dst[(size_t)n * p.M + m] = v[(mt * NG + tg) * 4 + e];
            }
}

// Work item `it`: its tile, its K stages [k0, k1), and its partial-sum slot (-1: a
// whole tile, written to dst).
struct Item {
    int tile, k0, k1, slot;
};

__device__ __forceinline__ Item item_of(const RParams& p, int it) {
    if (it < p.whole) return Item{it, 0, p.nst, -1};
    const int j = it - p.whole, z = j % p.splits;
    return Item{p.whole + j / p.splits, z * p.nst / p.splits, (z + 1) * p.nst / p.splits, j};
}

// Stage k's activation codes and scale quads: two contiguous byte ranges of the
// workspace, laid out by the activation kernel exactly as the stage slots hold them.
template <int NG>
__device__ __forceinline__ void issue_acts(const RParams& p, uint32_t sbase, int s, int k, uint32_t bar) {
    using C = RCfg<NG>;
    bulk_g2s(sbase + C::OFF_B + s * C::B_BYTES, p.bmat + (size_t)k * C::B_BYTES, C::B_BYTES, bar);
    bulk_g2s(sbase + C::OFF_DS + s * C::DS_BYTES, p.ds + (size_t)k * C::DS_BYTES, C::DS_BYTES, bar);
}

template <int NG>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
rmma_kernel(const __grid_constant__ CUtensorMap tmap_w, const RParams p) {
    using C = RCfg<NG>;
    constexpr int S = C::S;
    extern __shared__ uint8_t smem_dyn[];
    // 128-byte aligned by pointer arithmetic on the shared array (keeps the loads below in the shared space)
    uint8_t* smem = smem_dyn + ((128u - (smem_u32(smem_dyn) & 127u)) & 127u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full = sbase + C::OFF_BAR;
    const uint32_t empty = full + 8 * S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, CWARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        pdl_trigger();   // the next kernel on the stream may be scheduled (it waits for this grid itself)
    }
    __syncthreads();
    const Waiter wt{abort_flag, p.abort_word, p.limit_ns, &g_rmma_status};

    if (warp == CWARPS) {
        // ---------------- producer
        if (lane == 0) {
            const bool faulted = p.fault && blockIdx.x == 0;
            int q = 0;            // stages started by this CTA
            bool ok = true;
            bool acts_ready = false;
            int pend[S];          // K stage of each of the first S stages (-1: left out)
            for (int it = blockIdx.x; it < p.items && ok; it += gridDim.x) {
                const Item item = item_of(p, it);
                const int tile = item.tile;
                for (int k = item.k0; k < item.k1; ++k) {
                    const int s = q % S;
                    if (q >= S) {
                        if (!acts_ready) {
                            // the activations of the first S stages, once the activation kernel is done
                            pdl_wait();
                            acts_ready = true;
                            for (int i = 0; i < S; ++i)
                                if (pend[i] >= 0) issue_acts<NG>(p, sbase, i, pend[i], full + 8 * i);
                        }
                        if (!wait_or_abort(empty + 8 * s, ((q / S) + 1) & 1, wt)) {
                            ok = false;
                            break;
                        }
                    }
                    const int qi = q++;
                    if (faulted && qi == 0) {   // test only: this stage never completes
                        pend[0] = -1;
                        continue;
                    }
                    const uint32_t bar = full + 8 * s;
                    mbar_arrive_expect_tx(bar, C::STAGE_TX);
                    tma_load_2d(sbase + s * RAW_BYTES, &tmap_w, k * RAW_ROW, tile * RM, bar);
                    if (acts_ready) issue_acts<NG>(p, sbase, s, k, bar);
                    else pend[s] = k;
                }
            }
            if (!acts_ready) {   // fewer than S stages in all
                pdl_wait();
                for (int i = 0; i < min(q, S); ++i)
                    if (pend[i] >= 0) issue_acts<NG>(p, sbase, i, pend[i], full + 8 * i);
            }
            // no copy may still be writing this CTA's shared memory when it exits: the
            // last S stages started are the only ones nobody may have waited for
            for (int q2 = max(0, q - S); q2 < q; ++q2)
                if (!(faulted && q2 == 0)) mbar_wait_bounded(full + 8 * (q2 % S), (q2 / S) & 1, p.limit_ns);
        }
        return;
    }

    // ---------------- consumers
    pdl_wait();   // the split counters and dst are touched only after the activation kernel
    const int g = lane >> 2, t = lane & 3;
    int q = 0;
    for (int it = blockIdx.x; it < p.items; it += gridDim.x) {
        const Item item = item_of(p, it);
        const int tile = item.tile;
        uint64_t acc[2][NG][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int tg = 0; tg < NG; ++tg) acc[mt][tg][0] = acc[mt][tg][1] = 0ull;
        for (int k = item.k0; k < item.k1; ++k, ++q) {
            const int s = q % S;
            if (!warp_wait(full + 8 * s, (q / S) & 1, wt)) return;
            // row g of this warp's first m16 tile; rows g + 8r are 8r * 36 words further
            const uint32_t* rw =
                reinterpret_cast<const uint32_t*>(smem + s * RAW_BYTES) + (32 * warp + g) * (RAW_ROW / 4);
            const uint8_t* bsm = smem + C::OFF_B + s * C::B_BYTES;
            const uint8_t* dss = smem + C::OFF_DS + s * C::DS_BYTES;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                // blocks 2pp and 2pp+1 = the 9 words 9pp .. 9pp+8 of each row: block a's
                // scale in the low half of word 0, its nibbles in bytes 2..17, block b's
                // scale in the high half of word 4, its nibbles in words 5..8
                uint32_t qa[4], qb[4];
                float da[4], db[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const uint32_t* rp = rw + 8 * r * (RAW_ROW / 4);
                    qa[r] = __byte_perm(rp[9 * pp + t], rp[9 * pp + t + 1], 0x5432);
                    qb[r] = rp[9 * pp + 5 + t];
                    da[r] = fp16_to_f32(rp[9 * pp]);
                    db[r] = fp16_to_f32(rp[9 * pp + 4] >> 16);
                }
                block_mma<NG>(acc, qa, da, bsm + (2 * pp) * C::B_BLOCK, dss + (2 * pp) * C::DS_BLOCK, g, t);
                block_mma<NG>(acc, qb, db, bsm + (2 * pp + 1) * C::B_BLOCK, dss + (2 * pp + 1) * C::DS_BLOCK, g, t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + 8 * s);
        }
        float v[C::ACC];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int tg = 0; tg < NG; ++tg) {
                const int o = (mt * NG + tg) * 4;
                unpack2(acc[mt][tg][0], v[o + 0], v[o + 1]);
                unpack2(acc[mt][tg][1], v[o + 2], v[o + 3]);
            }
        const int row0 = tile * RM + 32 * warp + g;
        if (item.slot < 0) {
            store_outputs<NG>(p, v, row0, t);
            continue;
        }
        // split-K: this split's sums go to the workspace for the reduce kernel
        float* mine = p.part + ((size_t)item.slot * CWARPS + warp) * (32 * C::ACC) + (size_t)lane * C::ACC;
#pragma unroll
        for (int i = 0; i < C::ACC; i += 4)
            *reinterpret_cast<float4*>(mine + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
}

// dst rows of the split tiles (tile0 onwards) from their splits' partial sums, added in
// split order: one thread per 4 outputs
// (a float4 of one lane's sums).  Launched behind the GEMM with programmatic dependent
// launch; griddepcontrol.wait returns once the GEMM has finished and its writes are visible.
template <int NG>
__global__ void __launch_bounds__(256)
rmma_reduce_kernel(const float* __restrict__ part, float* __restrict__ dst, int M, int N, int tile0, int tiles,
                   int splits) {
    using C = RCfg<NG>;
    pdl_wait();
    pdl_trigger();
    constexpr int C4 = C::ACC / 4;
    const int64_t total = (int64_t)tiles * RM * C4;
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < total; i += (int64_t)gridDim.x * 256) {
        const int c4 = (int)(i % C4);
        const int64_t tl = i / C4;                       // tile * 128 + warp * 32 + lane
        const int tile = (int)(tl / RM), wl = (int)(tl % RM), warp = wl >> 5, lane = wl & 31;   // of the split tiles
        const float* src = part + ((size_t)tile * splits * CWARPS + warp) * (32 * C::ACC) + (size_t)lane * C::ACC + 4 * c4;
        float4 sum = __ldcg(reinterpret_cast<const float4*>(src));
        for (int z = 1; z < splits; ++z) {
            const float4 f = __ldcg(reinterpret_cast<const float4*>(src + (size_t)z * CWARPS * 32 * C::ACC));
            sum.x = __fadd_rn(sum.x, f.x);
            sum.y = __fadd_rn(sum.y, f.y);
            sum.z = __fadd_rn(sum.z, f.z);
            sum.w = __fadd_rn(sum.w, f.w);
        }
        // the 4 sums are acc[mt][tg] of that lane, c4 = mt * NG + tg
        const int mt = c4 / NG, tg = c4 % NG, g = lane >> 2, t = lane & 3;
        const int m0 = (tile0 + tile) * RM + 32 * warp + 16 * mt + g, n0 = 8 * tg + 2 * t;
        const float v[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = m0 + 8 * (e >> 1), n = n0 + (e & 1);
            if (m < M && n < N) dst[(size_t)n * M + m] = v[e];
        }
    }
}

// Activation operand of one call: per (token, block) the Q8_0 codes (the same
// quantization as q4q_quantize_q8_0: one 4-lane group per block, 8 values a lane) as
// fp16, odd elements divided by 16, each 8-element group in the order
// [0,4,1,5,2,6,3,7]; per block and token pair the quad {2^24 d_x, 2^24 d_x',
// -8 sum q 2^-24, -8 sum q' 2^-24}, both laid out block by block with 8 NG token
// columns (tokens from N up to 8 NG get zeros); and the call's control words zeroed
// (its abort word).
__global__ void __launch_bounds__(ACT_THREADS)
act_to_rmma_kernel(const float* __restrict__ x, __half* __restrict__ bmat, float* __restrict__ ds, int K, int N,
                   unsigned int* __restrict__ ctrl, int ctrl_words) {
    const int n8 = (N + 7) / 8 * 8;   // token columns of the layout (8 NG)
    pdl_wait();      // launched behind earlier work only with the caller's PDL flag
    pdl_trigger();   // the GEMM may start its weight copies now
    const int nb = K / QK;
    for (int i = blockIdx.x * ACT_THREADS + threadIdx.x; i < ctrl_words; i += gridDim.x * ACT_THREADS) ctrl[i] = 0u;
    const int64_t total = (int64_t)n8 * nb * 4;
    for (int64_t m0 = (int64_t)blockIdx.x * ACT_THREADS; m0 < total; m0 += (int64_t)gridDim.x * ACT_THREADS) {
        const int64_t m = m0 + threadIdx.x;
        const int64_t blk = m < total ? m >> 2 : 0;
        const int i = (int)(m & 3);
        const int n = (int)(blk / nb), b = (int)(blk % nb);
        const bool real = m < total && n < N;
        float v[8];
        if (real) {
            const float4* src = reinterpret_cast<const float4*>(x + (int64_t)n * K + b * QK + i * 8);
            const float4 a = __ldg(src), c = __ldg(src + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        amax = warp_max4(amax);
        const float d = scale_q8(amax);
        int qv[8];
        quant8(v, d, -127.0f, 127.0f, qv);          // every lane takes part (warp vote inside)
        int sq = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) sq += qv[e];
        sq = warp_sum4(sq);
        if (m < total) {   // padding tokens get zero codes
            uint32_t hw[4];
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                // positions 2pp, 2pp+1 hold elements pp and pp + 4; odd elements / 16
                const int e0 = pp, e1 = pp + 4;
                const float f0 = (e0 & 1) ? (float)qv[e0] * 0.0625f : (float)qv[e0];
                const float f1 = (e1 & 1) ? (float)qv[e1] * 0.0625f : (float)qv[e1];
                const __half2 hv = __floats2half2_rn(f0, f1);
                hw[pp] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            *reinterpret_cast<uint4*>(bmat + ((int64_t)b * n8 + n) * QK + i * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
        if (m < total && i == 0) {
            float* quad = ds + ((int64_t)b * (n8 / 2) + n / 2) * 4;
            // 2^24 d_x and -8 sum q * 2^-24, both exact power-of-two scalings
            quad[n & 1] = real ? fp16_to_f32(fp16_bits(d)) * 16777216.0f : 0.0f;
            quad[2 + (n & 1)] = real ? (float)(-8 * sq) * 0x1p-24f : 0.0f;
        }
    }
}

// ------------------------------------------------------------------ host ----

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

int ng_of(int64_t ne11) { return (int)((ne11 + 7) / 8); }

int64_t tiles_of(int64_t ne01) { return (ne01 + RM - 1) / RM; }

size_t bmat_bytes(int64_t ne00, int64_t ne11) { return round256((size_t)ne00 * 8 * ng_of(ne11) * 2); }

size_t ds_bytes(int64_t ne00, int64_t ne11) { return round256((size_t)(ne00 / QK) * 4 * ng_of(ne11) * 16); }

// Which tiles run whole and how many K splits the others take.
struct SplitPlan {
    int64_t whole;   // tiles 0 .. whole-1
    int splits;      // for tiles whole .. tiles-1
};

size_t partial_bytes(int64_t ne01, int64_t ne11, const SplitPlan& sp) {
    return sp.splits > 1 ? (size_t)sp.splits * (size_t)(tiles_of(ne01) - sp.whole) * RM * 8 * ng_of(ne11) * 4 : 0;
}

// CTAs one launch keeps resident: CTAS_PER_SM per SM, as the launch bounds and the
// shared-memory plan are made for (checked against the occupancy calculator once).
int resident_ctas(const DeviceInfo& info) { return info.sm_count * CTAS_PER_SM; }

// K splits of a shape.  A split costs its partial sums' traffic and the reduce
// kernel, so only tiles that would otherwise leave most resident CTAs idle are split:
//  * fewer tiles than a third of the resident CTAs: every tile, into the largest power
//    of two of items that still fits one wave, each split keeping at least two stages;
//  * more tiles than resident CTAs: the whole waves run whole, and the last, partial
//    wave's tiles are split so that it is about as full as the others (the 1002-tile
//    lm_head: 912 whole tiles, then 90 tiles in 3 splits each);
//  * otherwise none.
// Timed on GB300 (CUDA graphs, 1, 2, 4, 8 or 16 splits of every tile, 8 / 16 / 32
// tokens), the best counts were 4096 x 1024 (8 tiles) 8 / 8 / 8, 4096 x 4096 (32 tiles)
// 4 / 8 / 8, 14336 x 4096 (32 tiles) 8 / 8 / 8, 4096 x 14336 (112 tiles) 1 / 1 / 1 --
// what the first and third rules give, but for 4096 x 4096 at 8 tokens (8: 7.2 against
// 6.9 us) -- and the lm_head 1 / 1 / 1 among uniform splits.
SplitPlan desired_plan(int64_t ne00, int64_t ne01, const DeviceInfo& info) {
    const int64_t nst = ne00 / KST, tiles = tiles_of(ne01), grid = resident_ctas(info);
    if (tiles * 3 < grid) {
        const int64_t most = std::min<int64_t>(grid / tiles, nst / 2);
        int s = 1;
        while (2 * s <= most && s < 64) s *= 2;
        return SplitPlan{s > 1 ? 0 : tiles, s};
    }
    const int64_t rem = tiles % grid;
    if (tiles >= grid && rem > 0) {
        const int64_t s = std::min<int64_t>({grid / rem, nst / 2, 64});
        if (s >= 2) return SplitPlan{tiles - rem, (int)s};
    }
    return SplitPlan{tiles, 1};
}

template <int NG>
q4q_status launch_ng(const CUtensorMap& tw, const RParams& p, cudaStream_t stream, const DeviceInfo& info) {
    using C = RCfg<NG>;
    static std::atomic<int> configured[64];
    auto kern = rmma_kernel<NG>;
    if (info.device < 0 || info.device >= 64) return Q4Q_ERR_CUDA;
    if (!configured[info.device].load()) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return Q4Q_ERR_CUDA;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, C::SMEM) != cudaSuccess ||
            per_sm < CTAS_PER_SM)
            return Q4Q_ERR_CUDA;
        configured[info.device].store(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<int64_t>(p.items, resident_ctas(info)));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // behind the activation kernel
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tw, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return Q4Q_ERR_CUDA;
    }
    q4q_status st = launch_status();
    if (st != Q4Q_OK || p.whole == p.tiles) return st;
    // the split tiles' sums into dst, behind the GEMM
    const int64_t threads = (int64_t)(p.tiles - p.whole) * RM * (C::ACC / 4);
    cfg.gridDim = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>((threads + 255) / 256, (int64_t)info.sm_count * 4)));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    if (cudaLaunchKernelEx(&cfg, rmma_reduce_kernel<NG>, (const float*)p.part, p.dst, p.M, p.N, p.whole,
                           p.tiles - p.whole, p.splits) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return Q4Q_ERR_CUDA;
    }
    return launch_status();
}

}  // namespace

unsigned int rmma_take_device_status() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_rmma_status, sizeof(v)) != cudaSuccess) return Q4Q_ERR_CUDA;
    if (v) cudaMemcpyToSymbol(g_rmma_status, &z, sizeof(z));
    return v;
}

bool rmma_supported(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info) {
    if (info.cc_major != 10) return false;
    if (ne00 < KST || ne00 % KST != 0 || ne00 >= (1 << 20)) return false;
    if (ne01 <= 0 || ne01 >= (1ll << 31) || ne11 < 1 || ne11 > MAX_TOKENS) return false;
    return RCfg<4>::SMEM <= info.max_smem_optin;
}

// Workspace: the fp16 activation codes, the scale quads, the control area (abort
// word), then the splits' partial sums.
size_t rmma_min_workspace_bytes(int64_t ne00, int64_t ne01, int64_t ne11) {
    (void)ne01;
    return bmat_bytes(ne00, ne11) + ds_bytes(ne00, ne11) + CTRL_WORDS * 4;
}

size_t rmma_workspace_bytes(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info) {
    return rmma_min_workspace_bytes(ne00, ne01, ne11) + partial_bytes(ne01, ne11, desired_plan(ne00, ne01, info));
}

q4q_status rmma_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11, float* dst,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream, const DeviceInfo& info,
                        bool pdl, const KernelDebug* dbg) {
    const size_t base = rmma_min_workspace_bytes(ne00, ne01, ne11);
    if (workspace_bytes < base) return Q4Q_ERR_WORKSPACE;
    // as many K splits as wanted and as the workspace holds partial sums for
    SplitPlan plan = desired_plan(ne00, ne01, info);
    while (plan.splits > 1 && base + partial_bytes(ne01, ne11, plan) > workspace_bytes) --plan.splits;
    if (plan.splits == 1) plan.whole = tiles_of(ne01);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    __half* bmat = reinterpret_cast<__half*>(ws);
    float* ds = reinterpret_cast<float*>(ws + bmat_bytes(ne00, ne11));
    unsigned int* ctrl = reinterpret_cast<unsigned int*>(ws + bmat_bytes(ne00, ne11) + ds_bytes(ne00, ne11));
    const int ctrl_words = CTRL_WORDS;

    // activation kernel (programmatic dependent launch behind earlier work only when asked)
    {
        const int64_t items = (ne11 + 7) / 8 * 8 * (ne00 / QK) * 4;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)std::max<int64_t>(
            1, std::min<int64_t>((items + ACT_THREADS - 1) / ACT_THREADS, (int64_t)info.sm_count * 8)));
        cfg.blockDim = dim3(ACT_THREADS);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        if (cudaLaunchKernelEx(&cfg, act_to_rmma_kernel, src1, bmat, ds, (int)ne00, (int)ne11, ctrl, ctrl_words) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return Q4Q_ERR_CUDA;
        }
        const q4q_status st = launch_status();
        if (st != Q4Q_OK) return st;
    }

    const int NG = ng_of(ne11);
    CUtensorMap tw;
    if (!encode_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, src0, (uint64_t)(ne00 / QK * Q4_0_BYTES), (uint64_t)ne01,
                       (uint64_t)(ne00 / QK * Q4_0_BYTES), RAW_ROW, RM))
        return Q4Q_ERR_CUDA;

    RParams p;
    p.bmat = reinterpret_cast<const uint8_t*>(bmat);
    p.ds = reinterpret_cast<const uint8_t*>(ds);
    p.M = (int)ne01;
    p.N = (int)ne11;
    p.nst = (int)(ne00 / KST);
    p.tiles = (int)tiles_of(ne01);
    p.whole = (int)plan.whole;
    p.splits = plan.splits;
    p.items = p.whole + (p.tiles - p.whole) * p.splits;
    p.dst = dst;
    p.part = plan.splits > 1 ? reinterpret_cast<float*>(ws + base) : nullptr;
    p.abort_word = ctrl;
    p.limit_ns = dbg ? dbg->limit_ns : WAIT_LIMIT_NS;
    p.fault = dbg ? dbg->fault : 0;
    switch (NG) {
        case 1: return launch_ng<1>(tw, p, stream, info);
        case 2: return launch_ng<2>(tw, p, stream, info);
        case 3: return launch_ng<3>(tw, p, stream, info);
        default: return launch_ng<4>(tw, p, stream, info);
    }
}

}  // namespace q4q
