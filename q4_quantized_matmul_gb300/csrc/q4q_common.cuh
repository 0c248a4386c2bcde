// q4q_common.cuh -- device helpers shared by the CUDA kernels of libq4q.
//
// Block quantization follows "llama.cpp 深度解读" (luoboask.github.io) §2
// "量化数据结构 — Q4_0 格式详解": per 32-element block, amax -> fp32 scale ->
// round(x / scale) -> clamp -> fp16 scale stored.  Rounding is half away from
// zero (roundf), the division is IEEE (__fdiv_rn), the fp16 store rounds to
// nearest even (__float2half_rn).  No fast-math anywhere in this library.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/q4q.h"

namespace q4q {

constexpr int QK = 32;
constexpr int Q4_0_BYTES = 18;
constexpr int Q8_0_BYTES = 34;

// device status codes (stored in a per-library status word, first error wins)
constexpr unsigned int DEV_OK = 0;
constexpr unsigned int DEV_TIMEOUT = Q4Q_ERR_TIMEOUT;

// ------------------------------------------------------------ quantization --

__device__ __forceinline__ float warp_max4(float v) {
    // max over the 4 consecutive lanes that hold one 32-element block
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
    return v;
}

__device__ __forceinline__ int warp_sum4(int v) {
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    return v;
}

// q = clamp(round_half_away(x / d), lo, hi); 0 when d == 0.  The quotient is
// the IEEE one (fl(x / d)), exactly as the encoder defines it.
__device__ __forceinline__ int quant_one(float x, float d, float lo, float hi) {
    if (d == 0.0f) return 0;
    float r = roundf(__fdiv_rn(x, d));
    r = fminf(fmaxf(r, lo), hi);
    return (int)r;
}

// Block scales without a division.  amax / 8 is exactly amax * 0.125 (a power of
// two).  For amax / 127 this is the division by a constant known in advance of
// N. Brisebarre, J.-M. Muller and S. K. Raina, "Accelerating correctly rounded
// floating-point division when the divisor is known in advance", IEEE Trans.
// Computers 53(8), 2004: with C = fl(1/127), q = fl(amax * C) and the exact
// remainder r = fma(-q, 127, amax), fma(r, C, q) is the correctly rounded
// quotient.  Their condition for the divisor was not relied on: the identity was
// checked against IEEE division for every positive finite binary32 amax (the CPU
// test suite re-checks a strided sample of them).
__device__ __forceinline__ float scale_q4(float amax) { return __fmul_rn(amax, 0.125f); }

__device__ __forceinline__ float scale_q8(float amax) {
    const float C = 0x1.020408p-7f;                  // fl(1/127)
    const float q = __fmul_rn(amax, C);
    const float r = __fmaf_rn(-q, 127.0f, amax);
    return __fmaf_rn(r, C, q);
}

// Hardware reciprocal (about 1 ulp); only ever used inside quant8's error
// budget, never as a stored value.
__device__ __forceinline__ float recip_approx(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// quant_one for N groups of 8 values (group n belongs to a block with scale
// d[n]), without a division on the common path.  inv = rcp.approx(d) is within
// 1 ulp (2^-23 relative) of 1/d, so t = fl(x * inv) is within 1.8e-7 |x / d| of
// x / d, and fl(x / d) within half an ulp (<= 3.9e-6 for |x / d| <= 128) of
// x / d: |t - fl(x / d)| <= 2.7e-5, since |x| <= amax and d = amax / 8 or amax /
// 127 give |x / d| <= 127.0001.  Round-half-away and round-to-nearest-even differ
// only at half-integers, and both are constant between them, so where t is more
// than NEAR_BAND = 5e-5 away from every half-integer, round-to-nearest-even(t)
// == roundf(fl(x / d)).  Elements inside that band (or with a non-finite t, e.g.
// a reciprocal flushed to infinity) take the exact quotient; one warp vote over
// all N groups keeps those divisions off the common path.  Must be called by all
// 32 lanes of the warp.
constexpr float NEAR_LIMIT = 0.49995f;            // 0.5 - NEAR_BAND
//
// RAW: the codes are only right in their low byte (the caller packs bytes and
// handles d == 0 itself); for Q8_0, whose common path needs no clamp.
template <int N, bool RAW = false>
__device__ __forceinline__ void quant8n(const float (&v)[N][8], const float (&d)[N], float lo, float hi,
                                        int (&q)[N][8]) {
    // Round to nearest even by adding 1.5 * 2^23 (|t| <= 2^22 here): the integer
    // lands in the low mantissa bits, so the code is the float's bit pattern minus
    // that of the constant -- full-rate adds instead of rint/convert instructions.
    constexpr float MAGIC = 12582912.0f;
    constexpr int MAGIC_BITS = 0x4B400000;
    float inv[N];
#pragma unroll
    for (int n = 0; n < N; ++n) inv[n] = recip_approx(d[n]);
    bool near = false;
#pragma unroll
    for (int n = 0; n < N; ++n) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float t = v[n][e] * inv[n];
            const float rm = __fadd_rn(t, MAGIC);
            // MAGIC_BITS has zero low bytes: the raw bits already hold the code's low byte
            q[n][e] = RAW ? __float_as_int(rm) : __float_as_int(rm) - MAGIC_BITS;
            near |= !(fabsf(__fsub_rn(t, __fsub_rn(rm, MAGIC))) <= NEAR_LIMIT) && d[n] != 0.0f;
        }
    }
    if (__any_sync(0xffffffffu, near)) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float t = v[n][e] * inv[n];
                const float r = __fsub_rn(__fadd_rn(t, MAGIC), MAGIC);
                if (d[n] != 0.0f && !(fabsf(__fsub_rn(t, r)) <= NEAR_LIMIT))
                    q[n][e] = (int)fminf(fmaxf(roundf(__fdiv_rn(v[n][e], d[n])), lo), hi);
            }
        }
    }
    // Codes stay inside [lo, hi] by construction on the common path: where d is an
    // fp32 normal, |x / d| <= 127.0001 never rounds past 127 (Q8_0) and x / d >= -8
    // never below -8 (Q4_0); x = +amax gives +8 in Q4_0, which the format stops at 7
    // (below).  Where d is an fp32 subnormal it carries too few bits for that bound
    // (amax = 11 * 2^-149 gives d = fl(amax / 8) = 2^-149 and quotients up to 11),
    // but then the flushed reciprocal is infinite, every element takes the exact
    // division above, and that path clamps to [lo, hi] itself.
    if constexpr (RAW) return;
    const int ihi = (int)hi;
#pragma unroll
    for (int n = 0; n < N; ++n) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            int c = q[n][e];
            if (hi < 127.0f) c = min(c, ihi);
            q[n][e] = (d[n] == 0.0f) ? 0 : c;
        }
    }
}

__device__ __forceinline__ void quant8(const float (&v)[8], float d, float lo, float hi, int (&q)[8]) {
    quant8n<1>(reinterpret_cast<const float (&)[1][8]>(v), reinterpret_cast<const float (&)[1]>(d), lo, hi,
               reinterpret_cast<int (&)[1][8]>(q));
}

__device__ __forceinline__ uint16_t fp16_bits(float d) {
    return __half_as_ushort(__float2half_rn(d));
}

__device__ __forceinline__ float fp16_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}

// Eight consecutive elements of one block -> one 32-bit word of Q4_0 nibbles.
// Byte j of the block's qs holds element 2j (low) and 2j+1 (high), so the 8
// elements e = 0..7 of this word land at bit 4e.  All 32 lanes of the warp must
// call it (see quant8).
__device__ __forceinline__ uint32_t pack_q4_word(const float (&v)[8], float d) {
    int q[8];
    quant8(v, d, -8.0f, 7.0f, q);
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) w |= (uint32_t)(q[e] + 8) << (4 * e);
    return w;
}

// ------------------------------------------------------ output activations --

// GELU(v) = v * Phi(v), Phi the standard normal CDF, written with erfc so that
// the small tail values keep their relative accuracy (1 + erf(v / sqrt 2) would
// cancel for negative v).  The pages name GELU for the GPT-2 MLP without a
// formula; this is its definition.
__device__ __forceinline__ float gelu_f32(float v) {
    return __fmul_rn(__fmul_rn(0.5f, v), erfcf(__fmul_rn(-v, 0.70710678118654752f)));
}

// SiLU(g) = g * sigmoid(g) = g / (1 + exp(-g)) ("llama.cpp 深度解读" §4, the Llama
// MLP); exp(-g) overflowing to infinity gives -0 for very negative g.
__device__ __forceinline__ float silu_f32(float g) {
    return __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
}

// SwiGLU of the same MLP: silu(gate) * up.
__device__ __forceinline__ float swiglu_f32(float gate, float up) {
    return __fmul_rn(silu_f32(gate), up);
}

// ------------------------------------------------------- operand unpacking --

// Q4_0 nibble word (elements e0..e7 at bits 4e) -> 8 fp16 values (e - 8) in the
// order [e0, e4, e1, e5, e2, e6, e3, e7].  A low nibble n OR-ed into 0x6400 is the
// fp16 1024 + n, and subtracting 1032 is exact; a high nibble left in place gives
// 1024 + 16 n, and (1024 + 16 n) / 16 - 72 = n - 8 is one exact HFMA2.
__device__ __forceinline__ uint4 nibbles_to_f16x8(uint32_t q) {
    const uint32_t MAGIC = 0x64006400u;
    const uint32_t q8 = q >> 8;
    uint32_t h[4];
    h[0] = (q & 0x000F000Fu) | MAGIC;    // {1024 + e0, 1024 + e4}
    h[1] = (q & 0x00F000F0u) | MAGIC;    // {1024 + 16 e1, 1024 + 16 e5}
    h[2] = (q8 & 0x000F000Fu) | MAGIC;   // {1024 + e2, 1024 + e6}
    h[3] = (q8 & 0x00F000F0u) | MAGIC;   // {1024 + 16 e3, 1024 + 16 e7}
    const __half2 bias = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));       // 1032
    const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));  // 1/16
    const __half2 m72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));        // -72
    uint4 out;
    __half2 r;
    r = __hsub2(*reinterpret_cast<__half2*>(&h[0]), bias); out.x = *reinterpret_cast<uint32_t*>(&r);
    r = __hfma2(*reinterpret_cast<__half2*>(&h[1]), sixteenth, m72); out.y = *reinterpret_cast<uint32_t*>(&r);
    r = __hsub2(*reinterpret_cast<__half2*>(&h[2]), bias); out.z = *reinterpret_cast<uint32_t*>(&r);
    r = __hfma2(*reinterpret_cast<__half2*>(&h[3]), sixteenth, m72); out.w = *reinterpret_cast<uint32_t*>(&r);
    return out;
}

__device__ __forceinline__ uint64_t pack2(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}

__device__ __forceinline__ void unpack2(uint64_t r, float& x, float& y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}

// two fp32 lanes at once: d = a * b, d = a * b + c (each lane rounded as fmul / fmaf)
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// ------------------------------------------------------------- async copy --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Same test, but the thread may be suspended in hardware for up to `hint_ns`
// while the phase is incomplete (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}

constexpr uint32_t SLEEP_HINT_NS = 100000;   // 0.1 ms per suspended try

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, for at most about `limit_ns`
// nanoseconds, or until *stop becomes non-zero (stop may be null).  Polls with the
// plain try_wait, which suspends the thread in hardware while the phase is
// incomplete, so a waiting warp takes almost no issue slots from working ones; the
// stop flag and the clock are looked at every 64 polls.
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, volatile int* stop,
                                                uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0u) {
            if (stop && *stop) return false;
            const uint64_t t = global_timer_ns();
            if (t0 == 0) t0 = t;
            else if (t - t0 > limit_ns) return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    return mbar_wait_until(bar, parity, nullptr, limit_ns);
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// ------------------------------------------------------ thread-block clusters --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the shared::cluster window, of shared-memory address `addr` of this
// CTA mapped into the CTA of rank `rank` of the cluster (same offset there).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
    return d;
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Cluster barrier (not .aligned: threads of one warp may take it separately).
// arrive has release semantics, wait acquire: shared-memory stores a thread made
// into any CTA of the cluster before its arrive are visible to every thread of
// the cluster after its wait.  wait returns once every non-exited thread of the
// cluster has arrived.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }

__device__ __forceinline__ void record_error(unsigned int* word, unsigned int code) {
    atomicCAS(word, 0u, code);
}

constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;   // one second

// What a bounded wait looks at besides its barrier: the CTA's abort flag (shared
// memory), the call's abort word (global memory) and the time limit.
struct Waiter {
    volatile int* flag;
    volatile unsigned int* word;
    uint64_t limit_ns;
    unsigned int* status;   // the translation unit's device status word
};

// bounded wait that also gives up as soon as another role of the CTA, or another CTA
// of the same call, has aborted
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, const Waiter& w) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, SLEEP_HINT_NS)) return true;
        if (*w.flag) return false;
        if (*w.word != 0) {   // another CTA of this call gave up
            *w.flag = 1;
            return false;
        }
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.flag = 1;
            atomicExch(const_cast<unsigned int*>(w.word), 1u);
            record_error(w.status, DEV_TIMEOUT);
            return false;
        }
    }
}

// Every lane polls the barrier itself (each gets its own acquire of the completed
// phase, which cannot advance before this warp arrives on the matching "empty"
// barrier); a single vote makes the verdict warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Waiter& w) {
    const bool ok = mbar_try_wait(bar, parity) || wait_or_abort(bar, parity, w);
    return __all_sync(0xffffffffu, ok);
}

}  // namespace q4q
