// q4q_mma.cu -- Q4_0 x Q8_0 mul_mat on the 5th-generation tensor cores (ne11 >= 8).
//
// The operation is "llama.cpp 深度解读" §3 "量化矩阵乘法 — 核心算子" as a GEMM:
//   dst[n][m] = sum_b fp32(d_w[m][b] * d_x[n][b]) * S_b[m][n],
//   S_b[m][n] = sum_{k in block b} (nibble[m][k] - 8) * q[n][k]     (exact integer).
// sm_103a has no integer tcgen05 MMA, so both operands are held as fp16 values
// that are exact small integers (weights in [-8, 7], activations in [-127, 127]).
// Each 32-wide K block is two K=16 tcgen05.mma (kind::f16) into a FRESH fp32 TMEM
// accumulator; |S_b| <= 32 * 8 * 127 < 2^24, so the accumulator holds S_b exactly.
// The per-block scales are then applied by CUDA-core warps reading the slab out of
// TMEM (tcgen05.ld), while the tensor core fills the other slab buffer.
//
// Warp roles (one CTA per 128-row x NT-token output tile, full K loop):
//   warp 0      : TMA producer of raw weight bytes (2-D tensor map over the block rows,
//                 box = 8 blocks (256 K; 144 bytes of Q4_0 or 272 of Q8_0) x 128 rows)
//                 into a 3-deep ring (2-deep for Q8_0)
//   warp 1      : TMEM allocator and the single MMA-issuing thread
//   warp 2      : TMA producer of the activation tile (fp16, 128-byte swizzle,
//                 box = 64 K x NT tokens) into a 4-deep ring
//   warps 4-7   : dequantizers: raw Q4_0 / Q8_0 -> fp16 A tile (128 rows x 64 K) written
//                 straight into tensor memory (tcgen05.st, row = TMEM lane), where the MMA
//                 reads it as its A operand, plus the fp32 block scales (shared memory)
//   warps 8..   : epilogue, NT/32 warps per TMEM lane quadrant: per 32-K slab each warp
//                 loads its 32 columns with one tcgen05.ld and applies acc += d_w d_x S
// K order inside every 8-element group is permuted the same way on both operands
// ([0,4,1,5,2,6,3,7]) so that a 32-bit word of nibbles turns into fp16 with a
// handful of bit operations; the dot product does not depend on that order.
// Every mbarrier wait is bounded; a wait that runs out records Q4Q_ERR_TIMEOUT in the
// library's status word, raises the call's abort word (in the workspace, zeroed by
// the activation kernel that precedes every GEMM launch, so an old timeout never
// reaches a later call), and the CTA winds down (waits for its own copies, frees its
// TMEM) and returns.  Other CTAs of the same call that find the abort word raised
// while they wait wind down the same way.
#include <algorithm>
#include <atomic>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "q4q_common.cuh"
#include "q4q_internal.h"

namespace q4q {
namespace {

__device__ unsigned int g_mma_status = 0;

// Bytes at the end of the GEMM's workspace operands that hold the call's abort word.
constexpr size_t CTRL_BYTES = 256;

constexpr int BM = 128;                 // weight rows per CTA tile (MMA M)
constexpr int KRAW = 256;               // K per raw-weight stage (8 blocks per row)
constexpr int KAB = 64;                 // K per A/B stage (2 blocks, one 128-byte swizzle row)
constexpr int A_COLS = KAB / 2;          // TMEM columns of one stage's A tile (2 fp16 per column)
constexpr int WQ4_0 = 0;                // weight block types
constexpr int WQ8_0 = 1;

// Bytes of one raw-stage row: 8 blocks of 18 (Q4_0) or 34 (Q8_0) bytes, a multiple
// of 16 either way (the TMA box's inner extent).
__host__ __device__ constexpr int raw_row_bytes(int wt) { return wt == WQ8_0 ? 8 * 34 : 8 * 18; }
// Bytes per element of the weight tensor map: a box dimension holds at most 256
// elements, so the 272-byte Q8_0 rows are mapped as 136 two-byte elements.
__host__ __device__ constexpr int raw_elem_bytes(int wt) { return wt == WQ8_0 ? 2 : 1; }
constexpr int NPAD = 128;               // activation-scale rows are padded to this

// ------------------------------------------------------------------ PTX ----

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}


// The same MMA with its A operand in tensor memory (M = 128 rows in the 128 lanes, K along
// the columns, two fp16 per 32-bit column).
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (its warp's lane quadrant).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

template <int CK>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[CK]) {
    if constexpr (CK == 8) tmem_ld8(taddr, r);
    else if constexpr (CK == 16) tmem_ld16(taddr, r);
    else tmem_ld32(taddr, r);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// one lane of the (converged) warp, the same on every call
__device__ __forceinline__ bool elect_one() {
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
    return pred != 0;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row atoms
// of 1024 bytes (stride-dimension offset 1024), version bits 46..48 = 0b001.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                 // leading-dimension offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride-dimension offset
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}



// Two words of Q8_0 codes (elements e0..e3, e4..e7) -> 8 fp16 values in the same
// order [e0, e4, e1, e5, e2, e6, e3, e7]: a byte permute puts e_k and e_{k+4} in
// the low bytes of the two halves, flipping their sign bits makes them e + 128,
// 0x64 in the high bytes makes the fp16 1024 + (e + 128), and subtracting 1152 is
// exact.
__device__ __forceinline__ uint4 codes_to_f16x8(uint32_t lo, uint32_t hi) {
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t sel = (uint32_t)(k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12));
        h[k] = (__byte_perm(lo, hi, sel) & 0x00FF00FFu) ^ 0x64806480u;
    }
    uint4 out;
    __half2 r;
    r = __hsub2(*reinterpret_cast<__half2*>(&h[0]), bias); out.x = *reinterpret_cast<uint32_t*>(&r);
    r = __hsub2(*reinterpret_cast<__half2*>(&h[1]), bias); out.y = *reinterpret_cast<uint32_t*>(&r);
    r = __hsub2(*reinterpret_cast<__half2*>(&h[2]), bias); out.z = *reinterpret_cast<uint32_t*>(&r);
    r = __hsub2(*reinterpret_cast<__half2*>(&h[3]), bias); out.w = *reinterpret_cast<uint32_t*>(&r);
    return out;
}

// position p of an 8-element group holds element PERM[p]
__host__ __device__ constexpr int perm8(int p) { return (p & 1) ? 4 + (p >> 1) : (p >> 1); }

struct MmaParams {
    int M, N, K, nb, Npad;
    int splits;           // split-K: blockIdx.z takes raw stages [z * n / splits, (z + 1) * n / splits)
    float* dst;           // [N][M]; with splits > 1 the partial sums go to dst + z * N * M
    const float* dx;      // [nb][Npad]
    int32_t* isums;       // debug: [N][M][nb]
    unsigned int* abort_word;   // this call's abort word (workspace; zero at launch)
    uint64_t limit_ns;    // bound of every wait
    int fault;            // test only: 1 = CTA (0, 0, 0) leaves out its first activation stage
};



template <int NT, int WT>
struct Cfg {
    // epilogue warps: NT/32 per TMEM lane quadrant (each owns 32 columns), at least one
    static constexpr int EPI_WARPS = NT >= 128 ? 16 : (NT >= 64 ? 8 : 4);
    // Narrow token tiles do little work per 32-K block, so a CTA is bound by the
    // latency of its per-block hand-offs: with shallower rings two CTAs fit on an
    // SM (shared memory, registers, TMEM) and their chains overlap.
    static constexpr int MIN_BLOCKS = NT <= 32 ? 2 : 1;
    // Q8_0 raw stages are 34816 bytes: two of them keep the widest tile in 227 KB
    static constexpr int RAW_STAGES = (NT <= 32 || WT == WQ8_0) ? 2 : 3;
    static constexpr int RAW_ROW = raw_row_bytes(WT);
    static constexpr int RAW_BYTES = BM * RAW_ROW;
    // 128-token tiles: 3 stages with 3 slab buffers, so that slab buffers repeat with the
    // stage ring (the loops are unrolled over it); narrower tiles: 4 stages, 2 slab pairs
    static constexpr int AB_STAGES = NT >= 128 ? 3 : 4;
    // Narrow tiles are bound by the single MMA-issuing thread: it hands TMEM over in
    // slab pairs (one check and one commit per A/B stage).  The widest tile is bound
    // by its epilogue, which frees each slab as soon as it has read it.
    static constexpr bool PAIRWISE = NT <= 64;
    static constexpr int CPW = NT * 4 / EPI_WARPS;       // columns per epilogue warp
    // Columns per tcgen05.ld: the widest tile reads its 32 columns per slab in two
    // 16-column loads, which keeps the epilogue within the 80 registers a thread of a
    // 768-thread CTA has (one 32-column load made it spill; measured 9% slower on the
    // 512-token lm_head).
    static constexpr int CH = NT >= 128 ? 16 : (CPW < 32 ? CPW : 32);
    static constexpr int THREADS = (8 + EPI_WARPS) * 32;
    static constexpr int B_BYTES = NT * KAB * 2;
    static constexpr int B_STRIDE = (B_BYTES + 1023) / 1024 * 1024;
    // TMEM: NBUF accumulator slabs of NT columns, then the A tiles of the A/B stages
    // (A_COLS columns each); the allocation is the power of two that holds both.
    static constexpr int NBUF = NT >= 128 ? 3 : 4;
    static constexpr int A_COL0 = NBUF * NT;
    static constexpr int TMEM_USED = A_COL0 + AB_STAGES * A_COLS;
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "tensor memory holds 512 columns");
    static constexpr int DX_BYTES = 2 * NT * 4;           // activation scales of one A/B stage
    // shared memory map (offsets from a 1024-aligned base)
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_B = OFF_RAW + RAW_STAGES * RAW_BYTES;                  // 1024-aligned
    static constexpr int OFF_DW = OFF_B + AB_STAGES * B_STRIDE;
    static constexpr int OFF_DX = OFF_DW + AB_STAGES * 2 * BM * 4;
    static constexpr int OFF_BAR = OFF_DX + AB_STAGES * DX_BYTES;
    static constexpr int NBARS = 2 * RAW_STAGES + 2 * AB_STAGES + 2 * NBUF + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;                                // + alignment slack
};

// WT: the weight block type (WQ4_0 or WQ8_0); only the raw stage and the
// dequantizers differ.
template <int NT, bool DEBUG, int WT>
__global__ void __launch_bounds__(Cfg<NT, WT>::THREADS, Cfg<NT, WT>::MIN_BLOCKS)
mma_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_b,
                const MmaParams p) {
    using C = Cfg<NT, WT>;
    constexpr int RAW_BYTES = C::RAW_BYTES;
    constexpr int NBUF = C::NBUF;
    constexpr int RAW_STAGES = C::RAW_STAGES;
    constexpr int AB_STAGES = C::AB_STAGES;
    extern __shared__ uint8_t smem_raw[];
    // align to 1024 bytes by pointer arithmetic on the shared array itself, so the
    // compiler keeps every derived pointer in the shared address space
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    const uint32_t raw_full = smem_u32(&bars[0]);
    const uint32_t raw_empty = smem_u32(&bars[RAW_STAGES]);
    const uint32_t ab_full = smem_u32(&bars[2 * RAW_STAGES]);
    const uint32_t ab_empty = smem_u32(&bars[2 * RAW_STAGES + AB_STAGES]);
    const uint32_t slab_full = smem_u32(&bars[2 * RAW_STAGES + 2 * AB_STAGES]);
    const uint32_t slab_empty = slab_full + 8 * NBUF;
    const uint32_t drain = slab_full + 16 * NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
    const Waiter wt{abort_flag, p.abort_word, p.limit_ns, &g_mma_status};
    float* dw_s = reinterpret_cast<float*>(smem + C::OFF_DW);
    const float* dx_s = reinterpret_cast<const float*>(smem + C::OFF_DX);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * NT;
    const int m0 = blockIdx.y * BM;
    // this CTA's share of the K loop (split-K: a contiguous range of raw stages)
    const int n_raw_all = p.K / KRAW;
    const int r_begin = (int)(((int64_t)blockIdx.z * n_raw_all) / p.splits);
    const int r_end = (int)(((int64_t)(blockIdx.z + 1) * n_raw_all) / p.splits);
    const int n_raw = r_end - r_begin, n_ab = n_raw * (KRAW / KAB), n_slab = n_raw * (KRAW / 32);
    const int ab_begin = r_begin * (KRAW / KAB);

    if (threadIdx.x == 0) {
        for (int s = 0; s < RAW_STAGES; ++s) {
            mbar_init(raw_full + 8 * s, 1);
            mbar_init(raw_empty + 8 * s, 4);
        }
        for (int s = 0; s < AB_STAGES; ++s) {
            mbar_init(ab_full + 8 * s, 4 + 1);
            // released by the MMA issuer's commit and every epilogue warp; with pairwise
            // hand-off by the epilogue warps alone (they release a stage only after
            // seeing the commit that follows its MMAs)
            mbar_init(ab_empty + 8 * s, (C::PAIRWISE && !DEBUG ? 0 : 1) + C::EPI_WARPS);
        }
        for (int s = 0; s < NBUF; ++s) {
            mbar_init(slab_full + 8 * s, 1);
            mbar_init(slab_empty + 8 * s, C::EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- raw Q4_0 producer
        if (lane == 0) {
            int r = 0;
            for (; r < n_raw; ++r) {
                const int st = r % RAW_STAGES;
                if (r >= RAW_STAGES && !wait_or_abort(raw_empty + 8 * st, ((r / RAW_STAGES) + 1) & 1, wt)) break;
                mbar_arrive_expect_tx(raw_full + 8 * st, RAW_BYTES);
                tma_load_2d(sbase + C::OFF_RAW + st * RAW_BYTES, &tmap_w, (r_begin + r) * (C::RAW_ROW / raw_elem_bytes(WT)), m0,
                            raw_full + 8 * st);
            }
            // let every load issued land before the CTA can exit: consumers that gave up
            // (this CTA's or another's abort) no longer wait for them
            for (int r2 = max(0, r - RAW_STAGES); r2 < r; ++r2)
                mbar_wait_bounded(raw_full + 8 * (r2 % RAW_STAGES), (r2 / RAW_STAGES) & 1, p.limit_ns);
        }
    } else if (warp == 2) {
        // ---------------- activation tile + activation scale producer
        if (lane == 0) {
            int i = 0;
            for (; i < n_ab; ++i) {
                const int s = i % AB_STAGES;
                if (i >= AB_STAGES && !wait_or_abort(ab_empty + 8 * s, ((i / AB_STAGES) + 1) & 1, wt)) break;
                // test only: the first CTA leaves out its first stage (no expected bytes, no
                // copies), so that stage never completes and every role's bounded wait runs out
                if (p.fault && i == 0 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) continue;
                const uint32_t bar = ab_full + 8 * s;
                mbar_arrive_expect_tx(bar, C::B_BYTES + C::DX_BYTES);
                tma_load_2d(sbase + C::OFF_B + s * C::B_STRIDE, &tmap_b, (ab_begin + i) * KAB, n0, bar);
                const uint32_t dxd = sbase + C::OFF_DX + s * C::DX_BYTES;
                bulk_g2s(dxd, p.dx + (size_t)(2 * (ab_begin + i)) * p.Npad + n0, NT * 4, bar);
                bulk_g2s(dxd + NT * 4, p.dx + (size_t)(2 * (ab_begin + i) + 1) * p.Npad + n0, NT * 4, bar);
            }
            const bool faulted = p.fault && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
            for (int i2 = max(0, i - AB_STAGES); i2 < i; ++i2)
                if (!(faulted && i2 == 0))   // the stage left out never completes
                    mbar_wait_bounded(ab_full + 8 * (i2 % AB_STAGES), (i2 / AB_STAGES) & 1, p.limit_ns);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        // One thread issues every MMA of the CTA, so its own instruction latency is on the
        // critical path.  The whole warp runs the stage loop (polls with a warp vote, forms
        // descriptors and addresses as warp-uniform values) and one elected lane issues the
        // MMAs and commits: 64 tokens 402 -> 383 us per Llama step against a lane-0-only
        // issuer.  The loop is unrolled over the ring, which makes every stage slot, slab
        // buffer and barrier parity a compile-time constant, and the B descriptors of the
        // stage slots are formed once.
        {
            const bool leader = elect_one();
            constexpr uint32_t IDESC = idesc_f16(BM, NT);
            bool ok = true;
            constexpr bool PAIRWISE = C::PAIRWISE && !DEBUG;
            // B descriptor of stage slot st at K offset `koff` bytes along the swizzled row:
            // the start-address field is the shared-memory byte address / 16 and stays far
            // from overflowing, so the slot and offset add to the first slot's descriptor
            const uint64_t bdesc0 = smem_desc_sw128(sbase + C::OFF_B);
#define Q4Q_BDESC(st, koff) (bdesc0 + (uint64_t)(((st) * C::B_STRIDE + (koff)) >> 4))
            if constexpr (PAIRWISE) {
                // One hand-off per A/B stage: its two K blocks go to the two slab buffers
                // of one pair, with one empty check and one commit for the pair.
                constexpr int NPAIR = NBUF / 2;
                static_assert(AB_STAGES % (2 * NPAIR) == 0, "slab pairs repeat with the stage ring");
                for (int i0 = 0; i0 < n_ab && ok; i0 += AB_STAGES) {
                    const uint32_t par_a = (uint32_t)((i0 / AB_STAGES) & 1);
#pragma unroll
                    for (int st = 0; st < AB_STAGES; ++st) {
                        const int i = i0 + st;
                        if (i >= n_ab) break;
                        const int pr = st % NPAIR;
                        const uint32_t par_e = (uint32_t)(((st / NPAIR) + 1) & 1);
                        const bool ra = mbar_try_wait(ab_full + 8 * st, par_a);
                        const bool re = i < NPAIR || mbar_try_wait(slab_empty + 8 * pr, par_e);
                        if (!__all_sync(0xffffffffu, ra && re) &&
                            (!warp_wait(ab_full + 8 * st, par_a, wt) ||
                             (i >= NPAIR && !warp_wait(slab_empty + 8 * pr, par_e, wt)))) {
                            ok = false;
                            break;
                        }
                        if (leader) {
                            tc_fence_after();
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk)
                                    mma_f16_tmem_a(tmem + (uint32_t)((2 * pr + j) * NT),
                                                   tmem + (uint32_t)(C::A_COL0 + st * A_COLS + 16 * j + 8 * kk),
                                                   Q4Q_BDESC(st, 64 * j + 32 * kk), IDESC, (uint32_t)kk);
                            }
                            mma_commit(slab_full + 8 * pr);
                        }
                        __syncwarp();
                    }
                }
            } else {
                // One slab per K block, each handed back by the epilogue on its own; the
                // slab buffers cycle with the stage ring (2 * AB_STAGES slabs a round).
                static_assert((2 * AB_STAGES) % NBUF == 0 && ((2 * AB_STAGES) / NBUF) % 2 == 0,
                              "slab buffers and their parities repeat with the stage ring");
                for (int i0 = 0; i0 < n_ab && ok; i0 += AB_STAGES) {
                    const uint32_t par_a = (uint32_t)((i0 / AB_STAGES) & 1);
#pragma unroll
                    for (int st = 0; st < AB_STAGES; ++st) {
                        const int i = i0 + st;
                        if (i >= n_ab) break;
                        if (!warp_wait(ab_full + 8 * st, par_a, wt)) { ok = false; break; }
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                                const int gg = 2 * st + j;                    // slab index within the round
                            const int buf = gg % NBUF;
                            const uint32_t par_e = (uint32_t)(((gg / NBUF) + 1) & 1);
                            if ((i0 > 0 || gg >= NBUF) && !warp_wait(slab_empty + 8 * buf, par_e, wt)) {
                                ok = false;
                                break;
                            }
                            if (leader) {
                                tc_fence_after();
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk)
                                    mma_f16_tmem_a(tmem + (uint32_t)(buf * NT),
                                                   tmem + (uint32_t)(C::A_COL0 + st * A_COLS + 16 * j + 8 * kk),
                                                   Q4Q_BDESC(st, 64 * j + 32 * kk), IDESC, (uint32_t)kk);
                                mma_commit(slab_full + 8 * buf);
                            }
                            __syncwarp();
                        }
                        if (!ok) break;
                        if (leader) mma_commit(ab_empty + 8 * st);
                        __syncwarp();
                    }
                }
            }
#undef Q4Q_BDESC
            if (!ok && leader) {
                // no MMA may still be reading shared memory or writing TMEM at exit
                mma_commit(drain);
                mbar_wait_bounded(drain, 0, p.limit_ns);
            }
            __syncwarp();
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- dequantizers: thread t <-> tile row t = TMEM lane t (warp 4 + q
        // owns lane quadrant q); each A/B stage needs one pair of the row's 8 raw blocks
        const int t = threadIdx.x - 128;
        const uint32_t a_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)C::A_COL0;
        bool ok = true;
        for (int r = 0; r < n_raw && ok; ++r) {
            const int st = r % RAW_STAGES;
            if (!warp_wait(raw_full + 8 * st, (r / RAW_STAGES) & 1, wt)) { ok = false; break; }
            const uint4* rowp = reinterpret_cast<const uint4*>(smem + C::OFF_RAW + st * RAW_BYTES + t * C::RAW_ROW);
#pragma unroll
            for (int a = 0; a < KRAW / KAB; ++a) {
                const int i = r * (KRAW / KAB) + a;
                const int s = i % AB_STAGES;
                if (i >= AB_STAGES && !warp_wait(ab_empty + 8 * s, ((i / AB_STAGES) + 1) & 1, wt)) {
                    ok = false;
                    break;
                }
                tc_fence_after();      // the MMAs that read this stage's A columns have completed
                const uint32_t a_stage = a_lane + (uint32_t)(s * A_COLS);
                if constexpr (WT == WQ4_0) {
                    // pair a = blocks 2a, 2a+1 = words 9a .. 9a+8 of the row, inside the three
                    // 16-byte chunks (9a)/4 .. (9a)/4 + 2 (16-byte loads keep the eight lanes
                    // of each load phase on distinct banks: the row pitch is 144 bytes)
                    uint32_t wv[12];
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        const uint4 v4 = rowp[(9 * a) / 4 + k];
                        wv[4 * k + 0] = v4.x; wv[4 * k + 1] = v4.y; wv[4 * k + 2] = v4.z; wv[4 * k + 3] = v4.w;
                    }
                    const int w0 = (9 * a) % 4;                  // first word of the pair (compile time)
                    uint32_t q[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) q[k] = __byte_perm(wv[w0 + k], wv[w0 + k + 1], 0x5432);   // block 2a
#pragma unroll
                    for (int k = 0; k < 4; ++k) q[4 + k] = wv[w0 + 5 + k];                              // block 2a+1
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint32_t av[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 h = nibbles_to_f16x8(q[4 * j + c]);
                            av[4 * c + 0] = h.x; av[4 * c + 1] = h.y; av[4 * c + 2] = h.z; av[4 * c + 3] = h.w;
                        }
                        tmem_st16(a_stage + (uint32_t)(16 * j), av);
                    }
                    dw_s[(s * 2 + 0) * BM + t] = fp16_to_f32(wv[w0]);
                    dw_s[(s * 2 + 1) * BM + t] = fp16_to_f32(wv[w0 + 4] >> 16);
                } else {
                    // pair a = blocks 2a, 2a+1 = words 17a .. 17a+16 of the row, inside the five
                    // 16-byte chunks (17a)/4 .. (17a)/4 + 4 (row pitch 272 bytes = 17 chunks:
                    // the eight lanes of a load phase hit distinct banks)
                    uint32_t wv[20];
#pragma unroll
                    for (int k = 0; k < 5; ++k) {
                        const uint4 v4 = rowp[(17 * a) / 4 + k];
                        wv[4 * k + 0] = v4.x; wv[4 * k + 1] = v4.y; wv[4 * k + 2] = v4.z; wv[4 * k + 3] = v4.w;
                    }
                    const int w0 = (17 * a) % 4;                 // first word of the pair (compile time)
                    uint32_t q[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) q[k] = __byte_perm(wv[w0 + k], wv[w0 + k + 1], 0x5432);   // block 2a
#pragma unroll
                    for (int k = 0; k < 8; ++k) q[8 + k] = wv[w0 + 9 + k];                              // block 2a+1
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint32_t av[16];
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint4 h = codes_to_f16x8(q[8 * j + 2 * c], q[8 * j + 2 * c + 1]);
                            av[4 * c + 0] = h.x; av[4 * c + 1] = h.y; av[4 * c + 2] = h.z; av[4 * c + 3] = h.w;
                        }
                        tmem_st16(a_stage + (uint32_t)(16 * j), av);
                    }
                    dw_s[(s * 2 + 0) * BM + t] = fp16_to_f32(wv[w0]);
                    dw_s[(s * 2 + 1) * BM + t] = fp16_to_f32(wv[w0 + 8] >> 16);
                }
                // the A columns are written before the stage is handed to the MMA issuer
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ab_full + 8 * s);
            }
            // Release the raw stage only now: every word loaded from it has been
            // consumed by the conversions above, so no load of this stage can still
            // be in flight when the producer's TMA starts overwriting it.
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(raw_empty + 8 * st);
        }
    } else if (warp >= 8) {
        // ---------------- epilogue
        const int q = warp & 3;                      // TMEM lane quadrant
        const int h = (warp - 8) >> 2;               // column group
        const int row = q * 32 + lane;
        const int m = m0 + row;
        const int col0 = h * C::CPW;
        const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
        if constexpr (DEBUG) {
            for (int g = 0; g < n_slab; ++g) {
                const int buf = g % NBUF;
                const int i = g >> 1, s = i % AB_STAGES, j = g & 1;
                if (!warp_wait(slab_full + 8 * buf, (g / NBUF) & 1, wt)) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < C::CPW; c0 += 8) {
                    uint32_t r[8];
                    tmem_ld8(tq + (uint32_t)(buf * NT + col0 + c0), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int n = n0 + col0 + c0 + c;
                        if (n < p.N && m < p.M)
                            p.isums[((size_t)n * p.M + m) * p.nb + r_begin * (KRAW / 32) + g] =
                                (int32_t)__uint_as_float(r[c]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(slab_empty + 8 * buf);
                    if (j == 1) mbar_arrive(ab_empty + 8 * s);
                }
            }
        } else {
            // Per slab each warp reads its CPW columns in loads of CH; the NT/32 warps that
            // share a lane quadrant overlap their load latencies.
            constexpr int CH = C::CH;
            static_assert(C::CPW % CH == 0 && (CH == 16 || CH == 32), "whole loads per slab");
            uint64_t acc[C::CPW / 2];
#pragma unroll
            for (int c = 0; c < C::CPW / 2; ++c) acc[c] = 0;
            bool aborted = false;
            constexpr int NPAIR = NBUF / 2;
            constexpr bool PAIRWISE = C::PAIRWISE;
            // per-thread bases; the stage loop is unrolled over the ring (as the issuer's),
            // so every stage slot, slab buffer and parity below is a compile-time constant
            const float* dw_row = dw_s + row;
            const float* dx_col = dx_s + col0;
            const uint32_t tq_col = tq + (uint32_t)col0;
            for (int i0 = 0; i0 < n_ab && !aborted; i0 += AB_STAGES) {
                const uint32_t par_a = (uint32_t)((i0 / AB_STAGES) & 1);
#pragma unroll
                for (int st = 0; st < AB_STAGES; ++st) {
                    const int i = i0 + st;
                    if (i >= n_ab) break;
                    const int pr = st % NPAIR;
                    {
                        // the stage's scales, and its slabs: pairwise, the commit of its slab
                        // pair; otherwise its second slab (the issuer commits it after the
                        // first, and a commit completes only once every earlier MMA of that
                        // thread has, so it implies the first)
                        const int g1 = 2 * st + 1;
                        const uint32_t bar_a = ab_full + 8 * st;
                        const uint32_t bar_b = PAIRWISE ? slab_full + 8 * pr : slab_full + 8 * (g1 % NBUF);
                        const uint32_t par_b = PAIRWISE ? (uint32_t)((st / NPAIR) & 1) : (uint32_t)((g1 / NBUF) & 1);
                        const bool ra = mbar_try_wait(bar_a, par_a);
                        const bool rb = mbar_try_wait(bar_b, par_b);
                        if (!__all_sync(0xffffffffu, ra && rb) &&
                            !(warp_wait(bar_a, par_a, wt) && warp_wait(bar_b, par_b, wt))) {
                            aborted = true;
                            break;
                        }
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int buf = PAIRWISE ? 2 * pr + j : (2 * st + j) % NBUF;
                        const float dwm = dw_row[(st * 2 + j) * BM];
                        const uint64_t dw2 = pack2(dwm, dwm);
                        const float4* dxs = reinterpret_cast<const float4*>(dx_col + (st * 2 + j) * NT);
#pragma unroll
                        for (int h = 0; h < C::CPW / CH; ++h) {
                            uint32_t r[CH];
                            tmem_ld_chunk<CH>(tq_col + (uint32_t)(buf * NT + h * CH), r);
                            tmem_ld_wait();
                            if (h == C::CPW / CH - 1 && (!PAIRWISE || j == 1)) {
                                tc_fence_before();
                                __syncwarp();
                                if (lane == 0) mbar_arrive(slab_empty + 8 * (PAIRWISE ? pr : buf));
                            }
#pragma unroll
                            for (int c = 0; c < CH / 4; ++c) {
                                const float4 d4 = dxs[h * (CH / 4) + c];
                                const int a = h * (CH / 2) + 2 * c;
                                acc[a] = ffma2(fmul2(dw2, pack2(d4.x, d4.y)),
                                               pack2(__uint_as_float(r[4 * c]), __uint_as_float(r[4 * c + 1])), acc[a]);
                                acc[a + 1] = ffma2(fmul2(dw2, pack2(d4.z, d4.w)),
                                                   pack2(__uint_as_float(r[4 * c + 2]), __uint_as_float(r[4 * c + 3])),
                                                   acc[a + 1]);
                            }
                        }
                    }
                    // the stage's scales have been read for both of its slabs
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ab_empty + 8 * st);
                }
            }
            if (!aborted && !*abort_flag && m < p.M) {
                float* out = p.dst + (size_t)blockIdx.z * p.N * p.M;
#pragma unroll
                for (int c = 0; c < C::CPW / 2; ++c) {
                    float x0, x1;
                    unpack2(acc[c], x0, x1);
                    const int n = n0 + col0 + 2 * c;
                    if (n < p.N) out[(size_t)n * p.M + m] = x0;
                    if (n + 1 < p.N) out[(size_t)(n + 1) * p.M + m] = x1;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------- activation operands --
// Q8_0 quantization of each src1 row (same recipe as q4q_quantize_q8_0), written
// as exact-integer fp16 in the permuted K order, plus the widened block scales
// d_x[b][n] (zero for the padding rows n >= N).
__global__ void __launch_bounds__(256)
act_to_mma_kernel(const float* __restrict__ x, __half* __restrict__ bmat, float* __restrict__ dx, int K, int N,
                  int Npad, unsigned int* __restrict__ abort_word) {
    const int nb = K / QK;
    if (blockIdx.x == 0 && threadIdx.x == 0) *abort_word = 0u;   // the GEMM launched next starts un-aborted
    const int64_t total = (int64_t)N * nb * 4;
    for (int64_t m0 = (int64_t)blockIdx.x * 256; m0 < total; m0 += (int64_t)gridDim.x * 256) {
        const int64_t m = m0 + threadIdx.x;
        const bool ok = m < total;
        const int64_t blk = ok ? m >> 2 : 0;
        const int i = (int)(m & 3);
        const int n = (int)(blk / nb), b = (int)(blk % nb);
        float v[8];
        if (ok) {
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
        if (ok) {
            uint32_t hw[4];
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const int q0 = qv[perm8(2 * pp)];
                const int q1 = qv[perm8(2 * pp + 1)];
                const __half2 hv = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
                hw[pp] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            *reinterpret_cast<uint4*>(bmat + (int64_t)n * K + b * QK + i * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            if (i == 0) dx[(int64_t)b * Npad + n] = fp16_to_f32(fp16_bits(d));
        }
    }
    // padding rows of the scale table
    const int64_t pad = (int64_t)nb * (Npad - N);
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < pad; e += (int64_t)gridDim.x * 256) {
        const int64_t b = e / (Npad - N), n = N + e % (Npad - N);
        dx[b * Npad + n] = 0.0f;
    }
}

// Public Q8_0 blocks -> the same operands (debug path).
__global__ void __launch_bounds__(256)
q8_to_mma_kernel(const uint8_t* __restrict__ yq, __half* __restrict__ bmat, float* __restrict__ dx, int K, int N,
                 int Npad, unsigned int* __restrict__ abort_word) {
    const int nb = K / QK;
    if (blockIdx.x == 0 && threadIdx.x == 0) *abort_word = 0u;
    const int64_t total = (int64_t)N * nb * 4;
    for (int64_t m = (int64_t)blockIdx.x * 256 + threadIdx.x; m < total; m += (int64_t)gridDim.x * 256) {
        const int64_t blk = m >> 2;
        const int i = (int)(m & 3);
        const int n = (int)(blk / nb), b = (int)(blk % nb);
        const uint8_t* y = yq + blk * Q8_0_BYTES;
        uint32_t hw[4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            const int q0 = (int8_t)y[2 + i * 8 + perm8(2 * pp)];
            const int q1 = (int8_t)y[2 + i * 8 + perm8(2 * pp + 1)];
            const __half2 hv = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
            hw[pp] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        *reinterpret_cast<uint4*>(bmat + (int64_t)n * K + b * QK + i * 8) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        if (i == 0) dx[(int64_t)b * Npad + n] = fp16_to_f32((uint32_t)y[0] | ((uint32_t)y[1] << 8));
    }
    const int64_t pad = (int64_t)nb * (Npad - N);
    for (int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x; e < pad; e += (int64_t)gridDim.x * 256) {
        const int64_t b = e / (Npad - N), n = N + e % (Npad - N);
        dx[b * Npad + n] = 0.0f;
    }
}

// dst[i] = sum over the splits of part[s][i], in split order (deterministic).
__global__ void __launch_bounds__(256)
split_reduce_kernel(const float* __restrict__ part, float* __restrict__ dst, int splits, int64_t nm) {
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < nm; i += (int64_t)gridDim.x * 256) {
        float acc = __ldcs(part + i);
        for (int z = 1; z < splits; ++z) acc = __fadd_rn(acc, __ldcs(part + (int64_t)z * nm + i));
        dst[i] = acc;
    }
}

// ------------------------------------------------------------------ host ----

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

int pick_nt(int64_t N) {
    if (N <= 16) return 16;
    if (N <= 32) return 32;
    if (N <= 64) return 64;
    return 128;
}

int64_t npad_of(int64_t N) { return (N + NPAD - 1) / NPAD * NPAD; }

size_t b_bytes_of(int64_t K, int64_t N) { return ((size_t)N * K * 2 + 255) / 256 * 256; }

// Workspace of one GEMM call: the fp16 activation operand, the activation scales
// ([nb][Npad] fp32, a multiple of 512 bytes), then the call's control block (its
// abort word).  Split-K partial sums, when used, follow.
size_t ctrl_offset_of(int64_t K, int64_t N) { return b_bytes_of(K, N) + (size_t)(K / QK) * (size_t)npad_of(N) * 4; }

template <int NT, bool DEBUG, int WT>
q4q_status launch_mma_t(const CUtensorMap& tw, const CUtensorMap& tb, const MmaParams& p, cudaStream_t stream,
                        int device) {
    using C = Cfg<NT, WT>;
    static std::atomic<int> configured[64];
    auto kern = mma_gemm_kernel<NT, DEBUG, WT>;
    if (device < 0 || device >= 64) return Q4Q_ERR_CUDA;
    if (!configured[device].load()) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return Q4Q_ERR_CUDA;
        configured[device].store(1);
    }
    dim3 grid((unsigned)((p.N + NT - 1) / NT), (unsigned)((p.M + BM - 1) / BM), (unsigned)p.splits);
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(tw, tb, p);
    return launch_status();
}

template <bool DEBUG, int WT>
q4q_status run_mma(const void* src0, int64_t ne00, int64_t ne01, int64_t ne11, const __half* bmat, const float* dx,
                   unsigned int* abort_word, float* dst, int32_t* isums, int splits, cudaStream_t stream,
                   const DeviceInfo& info, const KernelDebug* dbg = nullptr) {
    if (!get_encode()) return Q4Q_ERR_CUDA;
    const int NT = pick_nt(ne11);
    const int64_t row_bytes = ne00 / QK * (WT == WQ8_0 ? Q8_0_BYTES : Q4_0_BYTES);
    CUtensorMap tw, tb;
    {
        const int eb = raw_elem_bytes(WT);
        const cuuint64_t dims[2] = {(cuuint64_t)(row_bytes / eb), (cuuint64_t)ne01};
        const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)(raw_row_bytes(WT) / eb), BM};
        const cuuint32_t estr[2] = {1, 1};
        const CUtensorMapDataType dt = eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
        if (g_encode(&tw, dt, 2, const_cast<void*>(src0), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return Q4Q_ERR_CUDA;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)ne00, (cuuint64_t)ne11};
        const cuuint64_t strides[1] = {(cuuint64_t)(ne00 * 2)};
        const cuuint32_t box[2] = {KAB, (cuuint32_t)NT};
        const cuuint32_t estr[2] = {1, 1};
        if (g_encode(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(bmat), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return Q4Q_ERR_CUDA;
    }
    MmaParams p;
    p.M = (int)ne01;
    p.N = (int)ne11;
    p.K = (int)ne00;
    p.nb = (int)(ne00 / QK);
    p.Npad = (int)npad_of(ne11);
    p.splits = splits;
    p.dst = dst;
    p.dx = dx;
    p.isums = isums;
    p.abort_word = abort_word;
    p.limit_ns = dbg ? dbg->limit_ns : WAIT_LIMIT_NS;
    p.fault = dbg ? dbg->fault : 0;
    switch (NT) {
        case 16: return launch_mma_t<16, DEBUG, WT>(tw, tb, p, stream, info.device);
        case 32: return launch_mma_t<32, DEBUG, WT>(tw, tb, p, stream, info.device);
        case 64: return launch_mma_t<64, DEBUG, WT>(tw, tb, p, stream, info.device);
        default: return launch_mma_t<128, DEBUG, WT>(tw, tb, p, stream, info.device);
    }
}

}  // namespace

unsigned int mma_take_device_status() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_mma_status, sizeof(v)) != cudaSuccess) return Q4Q_ERR_CUDA;
    if (v) cudaMemcpyToSymbol(g_mma_status, &z, sizeof(z));
    return v;
}

bool mma_supported(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info) {
    if (info.cc_major != 10) return false;
    if (ne00 < KRAW || ne00 % KRAW != 0 || ne01 <= 0 || ne11 <= 0 || ne11 >= (1 << 20)) return false;
    if (ne01 >= (1ll << 31) || ne00 >= (1 << 20)) return false;
    return std::max(Cfg<128, WQ4_0>::SMEM, Cfg<128, WQ8_0>::SMEM) <= info.max_smem_optin && get_encode();
}

size_t mma_workspace_bytes(int64_t ne00, int64_t ne11) { return ctrl_offset_of(ne00, ne11) + CTRL_BYTES; }

// Split-K: when the output tiles alone leave most SMs idle (few tokens, few rows),
// the K loop of every tile is split over blockIdx.z, each split writing fp32 partial
// sums that split_reduce_kernel adds in split order.  Each split keeps at least two
// raw stages (512 K).  Fewer than 4 splits do not pay for the partial sums' traffic
// and the extra launch: timed on the Llama set, 2 or 3 splits made gate/up (112
// tiles at 8-64 tokens) and q/o/down (128 tiles at 512 tokens) slower, while 5-10
// splits made the 8- and 32-tile matrices 1.3-2.4x faster.
int mma_desired_splits(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info) {
    const int NT = pick_nt(ne11);
    const int64_t tiles = ((ne11 + NT - 1) / NT) * ((ne01 + BM - 1) / BM);
    const int64_t target = (int64_t)info.sm_count * (NT <= 32 ? 2 : 1);
    if (tiles <= 0) return 1;
    const int64_t want = (target + tiles - 1) / tiles;
    const int64_t most = (ne00 / KRAW) / 2;
    const int64_t s = std::min<int64_t>(want, most);
    return s >= 4 ? (int)s : 1;
}

size_t split_partial_bytes(int64_t ne01, int64_t ne11, int splits) {
    return splits > 1 ? ((size_t)splits * (size_t)ne01 * (size_t)ne11 * 4 + 255) / 256 * 256 : 0;
}

size_t mma_workspace_bytes_split(int64_t ne00, int64_t ne01, int64_t ne11, const DeviceInfo& info) {
    return mma_workspace_bytes(ne00, ne11) + split_partial_bytes(ne01, ne11, mma_desired_splits(ne00, ne01, ne11, info));
}

q4q_status mma_mul_mat(const void* src0, int64_t ne00, int64_t ne01, const float* src1, int64_t ne11, float* dst,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream, const DeviceInfo& info,
                       bool q8_weights, const KernelDebug* dbg) {
    const size_t base = mma_workspace_bytes(ne00, ne11);
    if (workspace_bytes < base) return Q4Q_ERR_WORKSPACE;
    // as many K splits as wanted and as the workspace holds partial sums for
    int splits = mma_desired_splits(ne00, ne01, ne11, info);
    while (splits > 1 && base + split_partial_bytes(ne01, ne11, splits) > workspace_bytes) --splits;
    if (splits < 4) splits = 1;   // 2 or 3 splits measured slower than none (see mma_desired_splits)
    float* part = splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + base) : nullptr;
    __half* bmat = static_cast<__half*>(workspace);
    float* dx = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + b_bytes_of(ne00, ne11));
    unsigned int* abort_word =
        reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + ctrl_offset_of(ne00, ne11));
    const int64_t items = ne11 * (ne00 / QK) * 4;
    const int grid = (int)std::min<int64_t>((items + 255) / 256, (int64_t)info.sm_count * 8);
    act_to_mma_kernel<<<grid, 256, 0, stream>>>(src1, bmat, dx, (int)ne00, (int)ne11, (int)npad_of(ne11), abort_word);
    q4q_status st = launch_status();
    if (st != Q4Q_OK) return st;
    float* out = splits > 1 ? part : dst;
    st = q8_weights
             ? run_mma<false, WQ8_0>(src0, ne00, ne01, ne11, bmat, dx, abort_word, out, nullptr, splits, stream, info, dbg)
             : run_mma<false, WQ4_0>(src0, ne00, ne01, ne11, bmat, dx, abort_word, out, nullptr, splits, stream, info, dbg);
    if (st != Q4Q_OK || splits == 1) return st;
    const int64_t nm = ne01 * ne11;
    const int rgrid = (int)std::max<int64_t>(1, std::min<int64_t>((nm + 255) / 256, (int64_t)info.sm_count * 8));
    split_reduce_kernel<<<rgrid, 256, 0, stream>>>(part, dst, splits, nm);
    return launch_status();
}

size_t mma_debug_workspace_bytes(int64_t ne00, int64_t ne11) { return mma_workspace_bytes(ne00, ne11); }

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t dim0, uint64_t dim1,
                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1) {
    if (!get_encode()) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)dim0, (cuuint64_t)dim1};
    const cuuint64_t strides[1] = {(cuuint64_t)stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

q4q_status mma_debug_isums(const void* src0, const void* src1_q8_0, int64_t ne00, int64_t ne01, int64_t ne11,
                           int32_t* out, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                           const DeviceInfo& info, bool q8_weights) {
    if (!mma_supported(ne00, ne01, std::max<int64_t>(ne11, 8), info)) return Q4Q_ERR_SHAPE;
    if (!aligned(src0, 16)) return Q4Q_ERR_ALIGN;
    if (workspace_bytes < mma_workspace_bytes(ne00, ne11)) return Q4Q_ERR_WORKSPACE;
    if (!workspace) return Q4Q_ERR_NULL;
    if (!aligned(workspace, 256)) return Q4Q_ERR_ALIGN;
    __half* bmat = static_cast<__half*>(workspace);
    float* dx = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + b_bytes_of(ne00, ne11));
    unsigned int* abort_word =
        reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(workspace) + ctrl_offset_of(ne00, ne11));
    const int64_t items = ne11 * (ne00 / QK) * 4;
    const int grid = (int)std::min<int64_t>((items + 255) / 256, (int64_t)info.sm_count * 8);
    q8_to_mma_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(src1_q8_0), bmat, dx, (int)ne00,
                                               (int)ne11, (int)npad_of(ne11), abort_word);
    q4q_status st = launch_status();
    if (st != Q4Q_OK) return st;
    return q8_weights ? run_mma<true, WQ8_0>(src0, ne00, ne01, ne11, bmat, dx, abort_word, nullptr, out, 1, stream, info)
                      : run_mma<true, WQ4_0>(src0, ne00, ne01, ne11, bmat, dx, abort_word, nullptr, out, 1, stream, info);
}

}  // namespace q4q
