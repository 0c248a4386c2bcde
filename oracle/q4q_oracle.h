/*
 * q4q_oracle.h -- the CPU oracle for the Q4_0 x Q8_0 quantized matmul.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, obviously-correct C99
 * restatement of what the method computes.  It shares no code, header, table
 * or helper with the CUDA library under q4_quantized_matmul_gb300/; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 *
 * Source of the method: "llama.cpp 深度解读" (luoboask.github.io),
 *   §2 "量化数据结构 — Q4_0 格式详解"  (block layout, encode, decode)
 *   §3 "量化矩阵乘法 — 核心算子"        (ggml_vec_dot_q4_0_q8_0, operand shapes)
 * Operand convention (src0 [ne00, ne01], src1 [ne10, ne11], dst [ne01, ne11],
 * ne[0] innermost): same page §3, and "ggml GPT-2 117M inference walkthrough"
 * (aicoding.csdn.net) §3.2 "QKV 线性投影".
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - Q4_0 quantizes with the fp32 scale d32 = amax/8 (IEEE division), stores
 *    fp16(d32) rounded to nearest-even, rounds w/d32 half away from zero and
 *    clamps to [-8, 7] before adding 8.  amax == 0 or d32 == 0 -> all nibbles 8.
 *  - Q8_0 (not printed on the pages) is the same recipe with d32 = amax/127 and
 *    clamp to [-127, 127]; block = fp16 d + 32 int8 = 34 bytes.
 *  - Byte j of qs holds element 2j in its low nibble and 2j+1 in its high one.
 *  - The dot subtracts 8 from each nibble (the printed loop elides it).
 *  - dst accumulates fp32(d0*d1) * (float)isum over blocks in order, in fp32.
 *
 * All buffers are host memory owned by the caller.  Nothing is allocated
 * except the per-row Q8_0 scratch inside orc_mul_mat (malloc, freed).
 */
#ifndef Q4Q_ORACLE_H
#define Q4Q_ORACLE_H

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_QK 32
#define ORC_Q4_0_BYTES 18
#define ORC_Q8_0_BYTES 34

/* IEEE 754 binary32 -> binary16, round to nearest even, subnormals kept,
 * overflow to infinity, NaN stays NaN.  Written from the format definition. */
uint16_t orc_fp16_from_f32(float x);
/* binary16 -> binary32, exact. */
float orc_f32_from_fp16(uint16_t h);
/* Bulk versions for tests. */
void orc_fp16_from_f32_n(const float* x, uint16_t* h, int64_t n);
void orc_f32_from_fp16_n(const uint16_t* h, float* x, int64_t n);

size_t orc_sizeof_block_q4_0(void);
size_t orc_sizeof_block_q8_0(void);

/* src: nrows x ncols fp32 row-major; dst: nrows * ncols/32 blocks. ncols % 32 == 0. */
void orc_quantize_q4_0(const float* src, uint8_t* dst, int64_t ncols, int64_t nrows);
void orc_quantize_q8_0(const float* src, uint8_t* dst, int64_t ncols, int64_t nrows);
/* decode (value = (nibble - 8) * d, resp. q * d), fp32 */
void orc_dequantize_q4_0(const uint8_t* src, float* dst, int64_t ncols, int64_t nrows);
void orc_dequantize_q8_0(const uint8_t* src, float* dst, int64_t ncols, int64_t nrows);

/* The pages' ggml_vec_dot_q4_0_q8_0: n elements, one Q4_0 row, one Q8_0 row. */
float orc_vec_dot_q4_0_q8_0(int64_t n, const uint8_t* vx, const uint8_t* vy);

/* Per-block integer sums: out[(i11*ne01 + i01)*nb + b] = sum_k (nib-8)*q. */
void orc_block_isums(const uint8_t* src0_q4_0, const uint8_t* src1_q8_0,
                     int64_t ne00, int64_t ne01, int64_t ne11, int32_t* out);

/* ggml_mul_mat(Q4_0 src0 [ne00, ne01], F32 src1 [ne10, ne11]) -> dst [ne01, ne11].
 * Quantizes each src1 row to Q8_0, then dst[i11*ne01 + i01] = vec_dot(row i01, q8 row i11).
 * If abs_scale != NULL it also receives sum_b |fp32(d0*d1) * isum_b| (fp64), the
 * per-element scale of the parity tolerance.  nthreads <= 1 runs serially;
 * otherwise OpenMP over output rows (same scalar code, same results).
 * Returns 0, or -1 on bad shapes / allocation failure. */
int orc_mul_mat(const uint8_t* src0_q4_0, int64_t ne00, int64_t ne01,
                const float* src1, int64_t ne10, int64_t ne11,
                float* dst, double* abs_scale, int nthreads);

/* Same contraction with src1 already in Q8_0 blocks. */
int orc_mul_mat_q8(const uint8_t* src0_q4_0, int64_t ne00, int64_t ne01,
                   const uint8_t* src1_q8_0, int64_t ne11,
                   float* dst, double* abs_scale, int nthreads);

/* Brute force in fp64 over decoded reals: dst = sum_k deq(w_k) * deq(x_k). */
void orc_mul_mat_decoded_f64(const uint8_t* src0_q4_0, int64_t ne00, int64_t ne01,
                             const uint8_t* src1_q8_0, int64_t ne11, double* dst);

/* ggml_get_rows on a Q4_0 / Q8_0 table [nrows][ncols]: dst[i] = decode(row ids[i]).
 * Returns 0; -2 if some id is outside [0, nrows) (that output row is zeroed);
 * -1 on bad shapes. */
int orc_get_rows_q4_0(const uint8_t* src, int64_t ncols, int64_t nrows, const int32_t* ids, int64_t n, float* dst);
int orc_get_rows_q8_0(const uint8_t* src, int64_t ncols, int64_t nrows, const int32_t* ids, int64_t n, float* dst);

/* Epilogues next to the matmul, fp64 activations rounded to fp32:
 * silu(x) = x * sigmoid(x); gelu(x) = x * Phi(x) (a reading: the pages name GELU only). */
double orc_silu(double x);
double orc_gelu(double x);
/* y[t][r] = act(fp32(y[t][r] + bias[r])), act 0 = identity, 1 = gelu; bias may be NULL. */
void orc_bias_act(float* y, const float* bias, int act, int64_t ne01, int64_t ne11);
/* y[i] = fp32(fp32(silu(gate[i])) * up[i]). */
void orc_swiglu(const float* gate, const float* up, float* y, int64_t n);

/* Q8_0 weights: the same contraction with 34-byte weight blocks, isum = sum_k qw_k * qx_k. */
float orc_vec_dot_q8_0_q8_0(int64_t n, const uint8_t* vx, const uint8_t* vy);
void orc_block_isums_w8(const uint8_t* src0_q8_0, const uint8_t* src1_q8_0,
                        int64_t ne00, int64_t ne01, int64_t ne11, int32_t* out);
int orc_mul_mat_w8_q8(const uint8_t* src0_q8_0, int64_t ne00, int64_t ne01,
                      const uint8_t* src1_q8_0, int64_t ne11,
                      float* dst, double* abs_scale, int nthreads);
int orc_mul_mat_w8(const uint8_t* src0_q8_0, int64_t ne00, int64_t ne01,
                   const float* src1, int64_t ne10, int64_t ne11,
                   float* dst, double* abs_scale, int nthreads);

int orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
