/*
 * q4q_oracle.c -- CPU oracle for the Q4_0 x Q8_0 quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY (see q4q_oracle.h).  Plain C99, built with
 * -O2 -ffp-contract=off so that every fp32 product and sum below is rounded
 * exactly where the source says, on x86-64 and on aarch64 alike.
 *
 * Method: "llama.cpp 深度解读" (luoboask.github.io) §2 and §3.  Each function
 * below names the passage it restates.  Every function here is pinned by a
 * CPU test against something other than itself (hand-derived golden block,
 * numpy's float16 cast, exact-grid round trips, fp64 brute force, numpy
 * float64 dot products of lossless inputs).
 */
#include "q4q_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ fp16 -- */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* binary32 -> binary16 round-to-nearest-even (IEEE 754-2008 §4.3.1).
 * The value m * 2^(e-23) (m = significand with hidden bit) is divided by the
 * binary16 quantum at its magnitude -- 2^(e-10) for normal results, 2^-24 for
 * subnormal ones -- and the integer quotient is rounded to nearest even. */
uint16_t orc_fp16_from_f32(float x)
{
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    int32_t  exp8 = (int32_t)((u >> 23) & 0xffu);
    uint32_t mant = u & 0x7fffffu;

    if (exp8 == 0xff) {                           /* inf or NaN */
        if (mant != 0) return (uint16_t)(sign | 0x7e00u);
        return (uint16_t)(sign | 0x7c00u);
    }
    int32_t  e;
    uint32_t m;
    if (exp8 == 0) { e = -126; m = mant; }        /* binary32 subnormal or zero */
    else           { e = exp8 - 127; m = mant | 0x800000u; }
    if (m == 0) return sign;

    int32_t q = (e - 10 > -24) ? e - 10 : -24;    /* log2 of the binary16 quantum */
    int32_t shift = 23 + q - e;                   /* >= 13 */
    uint32_t h;
    if (shift > 25) {
        h = 0;                                    /* below half the smallest subnormal */
    } else {
        uint32_t rem  = m & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        h = m >> shift;
        if (rem > half || (rem == half && (h & 1u))) h += 1u;
    }
    if (q == -24 && e - 10 < -24) {
        /* subnormal result (h <= 1024; h == 1024 is the smallest normal) */
        return (uint16_t)(sign | h);
    }
    /* normal result: h in [1024, 2048] */
    int32_t ee = e;
    if (h == 2048u) { h = 1024u; ee += 1; }
    if (ee + 15 >= 31) return (uint16_t)(sign | 0x7c00u);   /* overflow */
    return (uint16_t)(sign | (uint16_t)((ee + 15) << 10) | (uint16_t)(h - 1024u));
}

/* binary16 -> binary32: exact widening of sign, exponent and significand. */
float orc_f32_from_fp16(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t exp5 = ((uint32_t)h >> 10) & 0x1fu;
    uint32_t mant = (uint32_t)h & 0x3ffu;
    if (exp5 == 0x1f) return bits_f32(sign | 0x7f800000u | (mant << 13));
    if (exp5 == 0) {
        /* subnormal: mant * 2^-24, exact in binary32 */
        float v = (float)mant * (1.0f / 16777216.0f);
        return sign ? -v : v;
    }
    return bits_f32(sign | ((exp5 - 15u + 127u) << 23) | (mant << 13));
}

void orc_fp16_from_f32_n(const float* x, uint16_t* h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = orc_fp16_from_f32(x[i]);
}

void orc_f32_from_fp16_n(const uint16_t* h, float* x, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) x[i] = orc_f32_from_fp16(h[i]);
}

static uint16_t load_u16le(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void store_u16le(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

size_t orc_sizeof_block_q4_0(void) { return ORC_Q4_0_BYTES; }   /* 2 + 32/2 */
size_t orc_sizeof_block_q8_0(void) { return ORC_Q8_0_BYTES; }   /* 2 + 32   */

/* ---------------------------------------------------------- quantizers -- */

/* One Q4_0 block, following the four encode steps of §2:
 *   1. amax = largest |w| in the block
 *   2. scale = amax / 8
 *   3. q = round(w / scale) + 8  (clamped so that q - 8 stays in [-8, 7])
 *   4. qs[i/2] = q[i] | q[i+1] << 4
 * and the block layout { fp16 d; uint8 qs[16]; }. */
static void quantize_block_q4_0(const float* w, uint8_t* out)
{
    float amax = 0.0f;
    for (int k = 0; k < ORC_QK; ++k) {
        float a = fabsf(w[k]);
        if (a > amax) amax = a;
    }
    float scale = amax / 8.0f;
    uint8_t q[ORC_QK];
    for (int k = 0; k < ORC_QK; ++k) {
        int v = 0;
        if (scale != 0.0f) {
            float r = roundf(w[k] / scale);        /* half away from zero */
            if (r < -8.0f) r = -8.0f;
            if (r > 7.0f) r = 7.0f;
            v = (int)r;
        }
        q[k] = (uint8_t)(v + 8);
    }
    store_u16le(out, orc_fp16_from_f32(scale));
    for (int j = 0; j < ORC_QK / 2; ++j)
        out[2 + j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
}

/* One Q8_0 block: same recipe with the signed 8-bit range, scale = amax/127,
 * q in [-127, 127]; layout { fp16 d; int8 qs[32]; } (the activation side of
 * §3's dot product, whose struct the pages do not print). */
static void quantize_block_q8_0(const float* x, uint8_t* out)
{
    float amax = 0.0f;
    for (int k = 0; k < ORC_QK; ++k) {
        float a = fabsf(x[k]);
        if (a > amax) amax = a;
    }
    float scale = amax / 127.0f;
    store_u16le(out, orc_fp16_from_f32(scale));
    for (int k = 0; k < ORC_QK; ++k) {
        int v = 0;
        if (scale != 0.0f) {
            float r = roundf(x[k] / scale);
            if (r < -127.0f) r = -127.0f;
            if (r > 127.0f) r = 127.0f;
            v = (int)r;
        }
        out[2 + k] = (uint8_t)(int8_t)v;
    }
}

void orc_quantize_q4_0(const float* src, uint8_t* dst, int64_t ncols, int64_t nrows)
{
    int64_t nb = ncols / ORC_QK;
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block_q4_0(src + r * ncols + b * ORC_QK, dst + (r * nb + b) * ORC_Q4_0_BYTES);
}

void orc_quantize_q8_0(const float* src, uint8_t* dst, int64_t ncols, int64_t nrows)
{
    int64_t nb = ncols / ORC_QK;
    for (int64_t r = 0; r < nrows; ++r)
        for (int64_t b = 0; b < nb; ++b)
            quantize_block_q8_0(src + r * ncols + b * ORC_QK, dst + (r * nb + b) * ORC_Q8_0_BYTES);
}

/* Decode of §2: v0 = (qs[j/2] & 0x0F) - 8, v1 = (qs[j/2] >> 4) - 8, w = v * d. */
void orc_dequantize_q4_0(const uint8_t* src, float* dst, int64_t ncols, int64_t nrows)
{
    int64_t nb = ncols / ORC_QK;
    for (int64_t i = 0; i < nrows * nb; ++i) {
        const uint8_t* blk = src + i * ORC_Q4_0_BYTES;
        float d = orc_f32_from_fp16(load_u16le(blk));
        for (int j = 0; j < ORC_QK / 2; ++j) {
            int lo = (blk[2 + j] & 0x0F) - 8;
            int hi = (blk[2 + j] >> 4) - 8;
            dst[i * ORC_QK + 2 * j + 0] = (float)lo * d;
            dst[i * ORC_QK + 2 * j + 1] = (float)hi * d;
        }
    }
}

void orc_dequantize_q8_0(const uint8_t* src, float* dst, int64_t ncols, int64_t nrows)
{
    int64_t nb = ncols / ORC_QK;
    for (int64_t i = 0; i < nrows * nb; ++i) {
        const uint8_t* blk = src + i * ORC_Q8_0_BYTES;
        float d = orc_f32_from_fp16(load_u16le(blk));
        for (int k = 0; k < ORC_QK; ++k)
            dst[i * ORC_QK + k] = (float)(int8_t)blk[2 + k] * d;
    }
}

/* ------------------------------------------------------------- the dot -- */

/* Integer part of one block of §3's loop: byte j of the Q4_0 block carries
 * elements 2j (low nibble) and 2j+1 (high nibble); each nibble is offset by
 * -8 (the signed value of §2's decode) and multiplied by the matching int8. */
static int32_t block_isum(const uint8_t* xb, const uint8_t* yb)
{
    const uint8_t* qs = xb + 2;
    const int8_t* y = (const int8_t*)(yb + 2);
    int32_t sumi = 0;
    for (int j = 0; j < ORC_QK / 2; ++j) {
        int32_t v0 = (int32_t)(qs[j] & 0x0F) - 8;
        int32_t v1 = (int32_t)((qs[j] >> 4) & 0x0F) - 8;
        sumi += v0 * (int32_t)y[2 * j + 0] + v1 * (int32_t)y[2 * j + 1];
    }
    return sumi;
}

/* §3 ggml_vec_dot_q4_0_q8_0: sumf += (d0 * d1) * sumi over blocks in order. */
float orc_vec_dot_q4_0_q8_0(int64_t n, const uint8_t* vx, const uint8_t* vy)
{
    int64_t nb = n / ORC_QK;
    float sumf = 0.0f;
    for (int64_t i = 0; i < nb; ++i) {
        const uint8_t* xb = vx + i * ORC_Q4_0_BYTES;
        const uint8_t* yb = vy + i * ORC_Q8_0_BYTES;
        float d0 = orc_f32_from_fp16(load_u16le(xb));
        float d1 = orc_f32_from_fp16(load_u16le(yb));
        float d = d0 * d1;
        int32_t sumi = block_isum(xb, yb);
        sumf += d * (float)sumi;
    }
    return sumf;
}

static double vec_dot_abs_scale(int64_t n, const uint8_t* vx, const uint8_t* vy)
{
    int64_t nb = n / ORC_QK;
    double s = 0.0;
    for (int64_t i = 0; i < nb; ++i) {
        const uint8_t* xb = vx + i * ORC_Q4_0_BYTES;
        const uint8_t* yb = vy + i * ORC_Q8_0_BYTES;
        float d = orc_f32_from_fp16(load_u16le(xb)) * orc_f32_from_fp16(load_u16le(yb));
        s += fabs((double)d * (double)block_isum(xb, yb));
    }
    return s;
}

void orc_block_isums(const uint8_t* src0_q4_0, const uint8_t* src1_q8_0,
                     int64_t ne00, int64_t ne01, int64_t ne11, int32_t* out)
{
    int64_t nb = ne00 / ORC_QK;
    for (int64_t i11 = 0; i11 < ne11; ++i11)
        for (int64_t i01 = 0; i01 < ne01; ++i01)
            for (int64_t b = 0; b < nb; ++b)
                out[(i11 * ne01 + i01) * nb + b] =
                    block_isum(src0_q4_0 + (i01 * nb + b) * ORC_Q4_0_BYTES,
                               src1_q8_0 + (i11 * nb + b) * ORC_Q8_0_BYTES);
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int orc_mul_mat_q8(const uint8_t* src0_q4_0, int64_t ne00, int64_t ne01,
                   const uint8_t* src1_q8_0, int64_t ne11,
                   float* dst, double* abs_scale, int nthreads)
{
    if (ne00 <= 0 || ne00 % ORC_QK != 0 || ne01 < 0 || ne11 < 0) return -1;
    int64_t nb = ne00 / ORC_QK;
    for (int64_t i11 = 0; i11 < ne11; ++i11) {
        const uint8_t* yrow = src1_q8_0 + i11 * nb * ORC_Q8_0_BYTES;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 1 ? nthreads : 1) if (nthreads > 1)
#endif
        for (int64_t i01 = 0; i01 < ne01; ++i01) {
            const uint8_t* xrow = src0_q4_0 + i01 * nb * ORC_Q4_0_BYTES;
            dst[i11 * ne01 + i01] = orc_vec_dot_q4_0_q8_0(ne00, xrow, yrow);
            if (abs_scale) abs_scale[i11 * ne01 + i01] = vec_dot_abs_scale(ne00, xrow, yrow);
        }
    }
    return 0;
}

/* ggml_mul_mat as §3 states it: activations are quantized to Q8_0 row by row
 * ("激活值通常是 Q8_0 量化"), then every (i01, i11) pair is one vec_dot. */
int orc_mul_mat(const uint8_t* src0_q4_0, int64_t ne00, int64_t ne01,
                const float* src1, int64_t ne10, int64_t ne11,
                float* dst, double* abs_scale, int nthreads)
{
    if (ne00 <= 0 || ne00 % ORC_QK != 0 || ne10 != ne00 || ne01 < 0 || ne11 < 0) return -1;
    int64_t nb = ne00 / ORC_QK;
    uint8_t* q8 = (uint8_t*)malloc((size_t)(ne11 > 0 ? ne11 : 1) * (size_t)nb * ORC_Q8_0_BYTES);
    if (!q8) return -1;
    orc_quantize_q8_0(src1, q8, ne10, ne11);
    int rc = orc_mul_mat_q8(src0_q4_0, ne00, ne01, q8, ne11, dst, abs_scale, nthreads);
    free(q8);
    return rc;
}

/* Plain definition over decoded reals, fp64: dst = sum_k w_k * x_k with
 * w_k = (nibble-8)*d0 and x_k = q*d1 decoded independently of block_isum. */
void orc_mul_mat_decoded_f64(const uint8_t* src0_q4_0, int64_t ne00, int64_t ne01,
                             const uint8_t* src1_q8_0, int64_t ne11, double* dst)
{
    int64_t nb = ne00 / ORC_QK;
    for (int64_t i11 = 0; i11 < ne11; ++i11) {
        for (int64_t i01 = 0; i01 < ne01; ++i01) {
            double acc = 0.0;
            for (int64_t k = 0; k < ne00; ++k) {
                int64_t b = k / ORC_QK, e = k % ORC_QK;
                const uint8_t* xb = src0_q4_0 + (i01 * nb + b) * ORC_Q4_0_BYTES;
                const uint8_t* yb = src1_q8_0 + (i11 * nb + b) * ORC_Q8_0_BYTES;
                uint8_t byte = xb[2 + e / 2];
                int nib = (e % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
                double w = (double)(nib - 8) * (double)orc_f32_from_fp16(load_u16le(xb));
                double x = (double)(int8_t)yb[2 + e] * (double)orc_f32_from_fp16(load_u16le(yb));
                acc += w * x;
            }
            dst[i11 * ne01 + i01] = acc;
        }
    }
}

/* ------------------------------------------------------ row gather -- */

/* ggml_get_rows on a quantized table: the embedding lookup at the start of
 * the Llama graph of "llama.cpp 深度解读" §4 (ggml_get_rows(tok_embeddings,
 * inp_tokens)), with the token-embedding tensor stored as Q4_0 (the GGUF
 * tensor-info example of §1).  Output row i is the decode (§2) of table row
 * ids[i].  An id outside [0, nrows) leaves a row of zeros and makes the call
 * return -2; bad shapes return -1. */
static int get_rows(const uint8_t* src, int64_t ncols, int64_t nrows, const int32_t* ids, int64_t n,
                    float* dst, int64_t block_bytes, int q4)
{
    if (ncols <= 0 || ncols % ORC_QK != 0 || nrows < 0 || n < 0) return -1;
    int64_t row_bytes = ncols / ORC_QK * block_bytes;
    int bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t id = ids[i];
        if (id < 0 || id >= nrows) {
            memset(dst + i * ncols, 0, (size_t)ncols * sizeof(float));
            bad = 1;
            continue;
        }
        if (q4) orc_dequantize_q4_0(src + id * row_bytes, dst + i * ncols, ncols, 1);
        else    orc_dequantize_q8_0(src + id * row_bytes, dst + i * ncols, ncols, 1);
    }
    return bad ? -2 : 0;
}

int orc_get_rows_q4_0(const uint8_t* src, int64_t ncols, int64_t nrows, const int32_t* ids, int64_t n, float* dst)
{
    return get_rows(src, ncols, nrows, ids, n, dst, ORC_Q4_0_BYTES, 1);
}

int orc_get_rows_q8_0(const uint8_t* src, int64_t ncols, int64_t nrows, const int32_t* ids, int64_t n, float* dst)
{
    return get_rows(src, ncols, nrows, ids, n, dst, ORC_Q8_0_BYTES, 0);
}

/* ------------------------------------------------------- epilogues -- */

/* SiLU(x) = x * sigmoid(x), as the Llama MLP of "llama.cpp 深度解读" §4
 * (Step I) defines it, in fp64. */
double orc_silu(double x)
{
    return x * (1.0 / (1.0 + exp(-x)));
}

/* GELU, named by the GPT-2 MLP of the "ggml GPT-2 117M inference
 * walkthrough" (§3.5, F1 = GELU(Y W_fc + b_fc)) without a formula: taken as
 * its definition x * Phi(x), Phi the standard normal CDF = erfc(-x/sqrt 2)/2. */
double orc_gelu(double x)
{
    return 0.5 * x * erfc(-x / sqrt(2.0));
}

/* The bias add after a projection (ggml_add(ggml_repeat(b, cur), cur) in the
 * GPT-2 walkthrough §3.2/§3.5: the [ne01] bias is repeated over the ne11
 * tokens and added in fp32), then optionally GELU (act == 1), rounded to fp32.
 * y is [ne11][ne01], updated in place; bias may be NULL. */
void orc_bias_act(float* y, const float* bias, int act, int64_t ne01, int64_t ne11)
{
    for (int64_t t = 0; t < ne11; ++t) {
        for (int64_t r = 0; r < ne01; ++r) {
            float v = y[t * ne01 + r];
            if (bias) v = v + bias[r];
            if (act == 1) v = (float)orc_gelu((double)v);
            y[t * ne01 + r] = v;
        }
    }
}

/* SwiGLU of the Llama MLP (§4 Step I): gate_silu = silu(gate) as an fp32
 * tensor, then cur = gate_silu * up, an fp32 elementwise product. */
void orc_swiglu(const float* gate, const float* up, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        float s = (float)orc_silu((double)gate[i]);
        y[i] = s * up[i];
    }
}

/* ------------------------------------------------ Q8_0 weights -- */

/* Integer part of one block of the Q8_0 x Q8_0 dot: both blocks hold 32
 * signed 8-bit codes in element order (the Q8_0 type listed beside Q4_0 in
 * "llama.cpp 深度解读" §2's type table; block layout as for the activations). */
static int32_t block_isum_w8(const uint8_t* xb, const uint8_t* yb)
{
    const int8_t* x = (const int8_t*)(xb + 2);
    const int8_t* y = (const int8_t*)(yb + 2);
    int32_t sumi = 0;
    for (int k = 0; k < ORC_QK; ++k) sumi += (int32_t)x[k] * (int32_t)y[k];
    return sumi;
}

/* The same block loop as §3's vec_dot with Q8_0 weights:
 * sumf += fp32(d0 * d1) * sumi over blocks in order. */
float orc_vec_dot_q8_0_q8_0(int64_t n, const uint8_t* vx, const uint8_t* vy)
{
    int64_t nb = n / ORC_QK;
    float sumf = 0.0f;
    for (int64_t i = 0; i < nb; ++i) {
        const uint8_t* xb = vx + i * ORC_Q8_0_BYTES;
        const uint8_t* yb = vy + i * ORC_Q8_0_BYTES;
        float d = orc_f32_from_fp16(load_u16le(xb)) * orc_f32_from_fp16(load_u16le(yb));
        sumf += d * (float)block_isum_w8(xb, yb);
    }
    return sumf;
}

static double vec_dot_w8_abs_scale(int64_t n, const uint8_t* vx, const uint8_t* vy)
{
    int64_t nb = n / ORC_QK;
    double s = 0.0;
    for (int64_t i = 0; i < nb; ++i) {
        const uint8_t* xb = vx + i * ORC_Q8_0_BYTES;
        const uint8_t* yb = vy + i * ORC_Q8_0_BYTES;
        float d = orc_f32_from_fp16(load_u16le(xb)) * orc_f32_from_fp16(load_u16le(yb));
        s += fabs((double)d * (double)block_isum_w8(xb, yb));
    }
    return s;
}

void orc_block_isums_w8(const uint8_t* src0_q8_0, const uint8_t* src1_q8_0,
                        int64_t ne00, int64_t ne01, int64_t ne11, int32_t* out)
{
    int64_t nb = ne00 / ORC_QK;
    for (int64_t i11 = 0; i11 < ne11; ++i11)
        for (int64_t i01 = 0; i01 < ne01; ++i01)
            for (int64_t b = 0; b < nb; ++b)
                out[(i11 * ne01 + i01) * nb + b] =
                    block_isum_w8(src0_q8_0 + (i01 * nb + b) * ORC_Q8_0_BYTES,
                                  src1_q8_0 + (i11 * nb + b) * ORC_Q8_0_BYTES);
}

int orc_mul_mat_w8_q8(const uint8_t* src0_q8_0, int64_t ne00, int64_t ne01,
                      const uint8_t* src1_q8_0, int64_t ne11,
                      float* dst, double* abs_scale, int nthreads)
{
    if (ne00 <= 0 || ne00 % ORC_QK != 0 || ne01 < 0 || ne11 < 0) return -1;
    int64_t nb = ne00 / ORC_QK;
    for (int64_t i11 = 0; i11 < ne11; ++i11) {
        const uint8_t* yrow = src1_q8_0 + i11 * nb * ORC_Q8_0_BYTES;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads > 1 ? nthreads : 1) if (nthreads > 1)
#endif
        for (int64_t i01 = 0; i01 < ne01; ++i01) {
            const uint8_t* xrow = src0_q8_0 + i01 * nb * ORC_Q8_0_BYTES;
            dst[i11 * ne01 + i01] = orc_vec_dot_q8_0_q8_0(ne00, xrow, yrow);
            if (abs_scale) abs_scale[i11 * ne01 + i01] = vec_dot_w8_abs_scale(ne00, xrow, yrow);
        }
    }
    return 0;
}

/* ggml_mul_mat(Q8_0 src0, F32 src1): src1 rows quantized to Q8_0, then one
 * Q8_0 x Q8_0 vec_dot per output. */
int orc_mul_mat_w8(const uint8_t* src0_q8_0, int64_t ne00, int64_t ne01,
                   const float* src1, int64_t ne10, int64_t ne11,
                   float* dst, double* abs_scale, int nthreads)
{
    if (ne00 <= 0 || ne00 % ORC_QK != 0 || ne10 != ne00 || ne01 < 0 || ne11 < 0) return -1;
    int64_t nb = ne00 / ORC_QK;
    uint8_t* q8 = (uint8_t*)malloc((size_t)(ne11 > 0 ? ne11 : 1) * (size_t)nb * ORC_Q8_0_BYTES);
    if (!q8) return -1;
    orc_quantize_q8_0(src1, q8, ne10, ne11);
    int rc = orc_mul_mat_w8_q8(src0_q8_0, ne00, ne01, q8, ne11, dst, abs_scale, nthreads);
    free(q8);
    return rc;
}
