/*
 * q4q.h -- C ABI of the GB300 (sm_103a) Q4_0 x Q8_0 quantized matmul library
 * (libq4q.so).
 *
 * The operation is ggml's quantized weight matmul as described in
 * "llama.cpp 深度解读" (luoboask.github.io):
 *   §2 "量化数据结构 — Q4_0 格式详解"  -- the 18-byte Q4_0 block and its encode/decode,
 *   §3 "量化矩阵乘法 — 核心算子"        -- ggml_vec_dot_q4_0_q8_0, with activations
 *                                         quantized to Q8_0 so that the inner sum is integer.
 * Operand convention (ggml, ne[0] innermost, all buffers contiguous):
 *   src0  Q4_0   [ne00, ne01]  ne01 rows of ne00/32 blocks (weights)
 *   src1  F32    [ne10, ne11]  ne11 rows (tokens) of ne10 = ne00 floats
 *   dst   F32    [ne01, ne11]  dst[i11 * ne01 + i01]
 * as in the same page §3 and "ggml GPT-2 117M inference walkthrough"
 * (aicoding.csdn.net) §3.2 "QKV 线性投影" (c_attn_attn_w [768, 2304] x cur [768, N]
 * -> [2304, N]).
 *
 * Conventions shared by every call:
 *  - Memory: every pointer is DEVICE memory (cudaMalloc / a torch CUDA tensor)
 *    owned by the caller.  The library never allocates device memory and never
 *    frees caller memory; scratch space is passed in as `workspace`.
 *  - Streams: every call enqueues work on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and returns without synchronizing.  Outputs are
 *    valid once the stream has reached the call.
 *  - Errors: argument errors are detected on the host, returned synchronously,
 *    and nothing is launched.  A failed launch returns Q4Q_ERR_CUDA.  Kernels
 *    that wait on asynchronous copies bound every wait (about one second); a
 *    wait that runs out records Q4Q_ERR_TIMEOUT in a device status word that
 *    q4q_device_status() returns (and clears), and that call's kernel returns
 *    early, leaving its output incomplete.  The abort is scoped to the call:
 *    later calls run normally whether or not the word has been read.
 *  - Empty problems (ne01 == 0 or ne11 == 0, or nrows == 0) are valid and launch
 *    nothing.
 *  - Out of contract (not checked): non-finite inputs, and inputs whose block
 *    scale overflows fp16 (|x| > 65504 * 8 for Q4_0, 65504 * 127 for Q8_0).
 *  - Thread safety: calls may be made from several host threads; calls that
 *    overlap on the GPU must not share output or workspace buffers.
 */
#ifndef Q4Q_H
#define Q4Q_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define Q4Q_API __attribute__((visibility("default")))
#else
#define Q4Q_API
#endif

typedef struct CUstream_st* q4q_stream_t;   /* identical to cudaStream_t */

typedef enum {
    Q4Q_OK = 0,
    Q4Q_ERR_NULL = 1,       /* a required pointer is NULL                          */
    Q4Q_ERR_SHAPE = 2,      /* ne00 <= 0, ne00 % 32 != 0, ne10 != ne00, size < 0,
                               or a size beyond the documented limits              */
    Q4Q_ERR_ALIGN = 3,      /* a pointer is not aligned as the call requires       */
    Q4Q_ERR_WORKSPACE = 4,  /* workspace smaller than the call needs (see each call) */
    Q4Q_ERR_CUDA = 5,       /* a CUDA runtime call or kernel launch failed          */
    Q4Q_ERR_TIMEOUT = 6,    /* a bounded device wait ran out (see q4q_device_status) */
    Q4Q_ERR_ARG = 7         /* any other invalid argument (e.g. unknown path)       */
} q4q_status;

#define Q4Q_QK 32                    /* weights per block                          */
#define Q4Q_BLOCK_Q4_0_BYTES 18      /* fp16 d + 16 bytes of nibbles               */
#define Q4Q_BLOCK_Q8_0_BYTES 34      /* fp16 d + 32 int8                           */

/* Block layouts (little endian; `d` is the IEEE binary16 bit pattern).
 * Q4_0 (§2): qs[j] holds element 2j in its low nibble and element 2j+1 in its
 * high nibble; element value = (nibble - 8) * d.
 * Q8_0: qs[k] is element k; element value = qs[k] * d. */
typedef struct { uint16_t d; uint8_t qs[16]; } q4q_block_q4_0;
typedef struct { uint16_t d; int8_t  qs[32]; } q4q_block_q8_0;

/* Q4_0 encode (§2 "编码过程"): for each 32-element block of each row,
 *   amax = max |w|, d32 = amax / 8 (fp32, IEEE division),
 *   q = clamp(round_half_away(w / d32), -8, 7) + 8   (all 8 when d32 == 0),
 *   qs[j] = q[2j] | q[2j+1] << 4,  d = fp16_round_to_nearest_even(d32).
 * src: fp32 [nrows][ncols] row-major, device; dst: nrows * ncols/32 blocks
 * (18 bytes each, contiguous, no padding), device.
 * Requires ncols > 0, ncols % 32 == 0, nrows >= 0, ncols * nrows < 2^40.
 * Any alignment is accepted; 16-byte aligned src and dst take the fast path. */
Q4Q_API q4q_status q4q_quantize_q4_0(const float* src, void* dst, int64_t ncols, int64_t nrows,
                             q4q_stream_t stream);

/* Q8_0 encode: the same recipe on the signed 8-bit range (the activation side
 * of §3's dot product; the pages name the type but do not print its encoder):
 *   d32 = amax / 127, q = clamp(round_half_away(x / d32), -127, 127), d = fp16(d32).
 * Layout, requirements and alignment as q4q_quantize_q4_0; 34-byte blocks. */
Q4Q_API q4q_status q4q_quantize_q8_0(const float* src, void* dst, int64_t ncols, int64_t nrows,
                             q4q_stream_t stream);

/* Bytes of device workspace q4q_mul_mat wants for this problem.  The answer
 * depends only on the shapes and on the current device.  The tensor-core path
 * (ne11 > 32) runs in
 *   B = round_up(2 * ne00 * ne11, 256) + (ne00 / 32) * round_up(ne11, 128) * 4 + 256
 * bytes (fp16 activation codes, block scales, a control word) and the warp-MMA
 * kernel (2 <= ne11 <= 32) in round_up(2 * ne00 * n8, 256) + round_up(ne00 / 2 * n8,
 * 256) + 256 bytes, n8 = round_up(ne11, 8); the size returned adds room for split-K
 * (used when the output tiles alone leave SMs idle: few tokens or few rows): the
 * tensor-core path's fp32 partial sums, round_up(s * ne01 * ne11 * 4, 256) for
 * s <= ne00 / 512 splits, or the warp-MMA kernel's, s * T * 128 * n8 * 4 bytes for T
 * split 128-row tiles and s <= min(ne00 / 512, 64) splits.  The generic path needs
 * (ne00 / 32) * ne11 * 34 bytes, the GEMV none. */
Q4Q_API q4q_status q4q_mul_mat_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes);

/* ggml_mul_mat(src0 Q4_0 [ne00, ne01], src1 F32 [ne10, ne11]) -> dst F32 [ne01, ne11]
 * (§3): each src1 row is quantized to Q8_0 (as q4q_quantize_q8_0 does), then
 *   dst[i11*ne01 + i01] = sum_b fp32(d_w[i01,b] * d_x[i11,b]) * isum(i01, i11, b),
 *   isum = sum_{j<16} (lo_j - 8) * q[2j] + (hi_j - 8) * q[2j+1]   (exact int32).
 * The block sums are exact; the fp32 sum over blocks may be taken in any order
 * (results differ from a serial sum by rounding only).
 * src0: device, 2-byte aligned; src1 / dst: device, 4-byte aligned.
 * Paths (ne00 % 256 == 0 and 16-byte aligned src0 / src1 for all but the generic):
 *   ne11 = 1, and 2..3 on matrices of at most 2^24 weights (where it is faster): a
 *     fused GEMV that streams the weights once (no workspace);
 *   2 <= ne11 <= 32 otherwise: the warp-MMA kernel (an activation kernel, then
 *     per-warp mma.sync on nibbles unpacked in registers), given at least its
 *     split-free minimum of 256-byte aligned workspace (else the GEMV below 8
 *     tokens, Q4Q_ERR_WORKSPACE from 8);
 *   ne11 > 32: the tensor-core GEMM (tcgen05) on 256-byte aligned workspace.
 * With q4q_mul_mat_workspace_size(...) bytes K is split as planned; with less (down
 * to the split-free minimum) fewer splits are used, the splits' partial sums being
 * added in a fixed order, so a given workspace size gives the same bits every time.
 * Limits: 0 < ne00 < 2^20 (ne00 % 32 == 0), 0 <= ne01 < 2^31, 0 <= ne11 < 2^20. */
Q4Q_API q4q_status q4q_mul_mat(const void* src0, int64_t ne00, int64_t ne01,
                       const float* src1, int64_t ne10, int64_t ne11,
                       float* dst, void* workspace, size_t workspace_bytes,
                       q4q_stream_t stream);

/* Bytes of workspace q4q_debug_block_isums needs for `path` (0 for path 0). */
Q4Q_API q4q_status q4q_debug_workspace_size(int64_t ne00, int64_t ne11, int path, size_t* bytes);

/* Launch flags of q4q_mul_mat_ex. */
#define Q4Q_MUL_MAT_PDL 1u   /* programmatic dependent launch (see below) */

/* q4q_mul_mat with launch flags (0 = exactly q4q_mul_mat).
 * Q4Q_MUL_MAT_PDL: the kernel is launched with programmatic dependent launch, so
 * that it can be scheduled, set up and start streaming src0 while the work queued
 * before it on `stream` is still running; it waits for that work to complete
 * before it reads src1 or writes dst.  Valid only when no work still in flight on
 * the stream writes src0 (true for resident model weights).  Used by chains of
 * projections; honoured by the GEMV and the warp-MMA kernel (whose activation kernel
 * then waits for the work before it), ignored by the tensor-core GEMM. */
Q4Q_API q4q_status q4q_mul_mat_ex(const void* src0, int64_t ne00, int64_t ne01,
                          const float* src1, int64_t ne10, int64_t ne11,
                          float* dst, void* workspace, size_t workspace_bytes,
                          unsigned int flags, q4q_stream_t stream);

/* ------------------------------------------------ next to the matmul ---- */

/* Activations of q4q_mul_mat_bias_act. */
#define Q4Q_ACT_NONE 0
#define Q4Q_ACT_GELU 1   /* GELU(v) = v * Phi(v), Phi the standard normal CDF */

/* The projection, its bias and its activation in one call: the GPT-2 graph of
 * the "ggml GPT-2 117M inference walkthrough" adds a bias after every projection
 * (§3.2, §3.5: ggml_add(ggml_repeat(b, cur), cur)) and applies GELU after the
 * MLP's first one (§3.5, F1 = GELU(Y W_fc + b_fc)); "llama.cpp 深度解读" §4 names
 * "matmul + bias + activation" as the fusion a graph allows.  The page names
 * GELU without a formula; this library uses its definition v * Phi(v).
 *   dst[i11*ne01 + i01] = act(fp32(mul_mat[i11][i01] + bias[i01]))
 * with mul_mat exactly as q4q_mul_mat computes it.  bias: device fp32 [ne01]
 * (4-byte aligned) or NULL for none; act: Q4Q_ACT_NONE or Q4Q_ACT_GELU, else
 * Q4Q_ERR_ARG.  Everything else (arguments, workspace, flags, limits, errors)
 * as q4q_mul_mat_ex; under Q4Q_MUL_MAT_PDL the bias, like src0, may be read before
 * the work queued ahead of the call completes, so no work still in flight on the
 * stream may write it (true for a model's resident biases).  For ne11 < 8 the epilogue runs inside the GEMV (one launch);
 * other paths apply it with one elementwise kernel over dst after the matmul. */
Q4Q_API q4q_status q4q_mul_mat_bias_act(const void* src0, int64_t ne00, int64_t ne01,
                                const float* src1, int64_t ne10, int64_t ne11,
                                const float* bias, int act, float* dst,
                                void* workspace, size_t workspace_bytes,
                                unsigned int flags, q4q_stream_t stream);

/* Bytes of device workspace q4q_mul_mat_swiglu needs: q4q_mul_mat_workspace_size
 * rounded up to 256, plus 4 * ne01 * ne11 for the gate projection on the paths
 * that do not fuse it. */
Q4Q_API q4q_status q4q_mul_mat_swiglu_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes);

/* The Llama MLP's gate and up projections with SwiGLU ("llama.cpp 深度解读" §4,
 * Step I: up = ffn_up x, gate = ffn_gate x, cur = silu(gate) * up with SiLU(x) =
 * x * sigmoid(x)):
 *   dst[i11*ne01 + i01] = fp32(silu(g) * u),  g = mul_mat(gate)[i11][i01],
 *                                             u = mul_mat(up)[i11][i01].
 * gate, up: Q4_0 weights of the same shape [ne00, ne01] (layout and alignment as
 * q4q_mul_mat's src0); src1, dst, flags, limits and errors as q4q_mul_mat_ex;
 * workspace: q4q_mul_mat_swiglu_workspace_size bytes, 256-byte aligned (the fused
 * path does not touch it).  For ne11 < 8 with 16-byte aligned operands and
 * ne00 % 256 == 0 both matrices stream through one GEMV launch and only the
 * product is written; otherwise the two projections run as q4q_mul_mat calls
 * (gate into the workspace) followed by one elementwise kernel. */
Q4Q_API q4q_status q4q_mul_mat_swiglu(const void* gate, const void* up, int64_t ne00, int64_t ne01,
                              const float* src1, int64_t ne10, int64_t ne11, float* dst,
                              void* workspace, size_t workspace_bytes, unsigned int flags,
                              q4q_stream_t stream);

/* Most matrices one q4q_mul_mat_group call takes. */
#define Q4Q_GROUP_MAX 4

/* Bytes of device workspace q4q_mul_mat_group needs: the largest
 * q4q_mul_mat_workspace_size over the n matrices. */
Q4Q_API q4q_status q4q_mul_mat_group_workspace_size(int n, const int64_t* ne01, int64_t ne00, int64_t ne11,
                                            size_t* bytes);

/* Several Q4_0 projections of one input: for m < n,
 *   dst[m] = ggml_mul_mat(src0[m] [ne00, ne01[m]], src1 [ne10, ne11]),  dst[m] F32 [ne01[m], ne11],
 * each exactly as q4q_mul_mat computes it.  This is the q, k and v projections
 * of a layer with separate wq / wk / wv weights ("llama.cpp 深度解读" §3.2 of the
 * Gemma3 graph: llm_build_mul_mat_qkv takes either a fused wqkv or the three
 * tensors); a fused wqkv is a single q4q_mul_mat over concatenated rows.
 * n: 1 .. Q4Q_GROUP_MAX, else Q4Q_ERR_ARG.  src0, ne01, dst: HOST arrays of n
 * entries (src0[m], dst[m] are device pointers, aligned as q4q_mul_mat requires;
 * the outputs must not overlap each other or src1).  Matrices with ne01[m] == 0
 * are skipped.  workspace: q4q_mul_mat_group_workspace_size bytes.  flags and
 * errors as q4q_mul_mat_ex.  For ne11 < 8 with ne00 % 256 == 0 and 16-byte aligned
 * weights and src1, all matrices stream through one GEMV launch that quantizes
 * src1 once; otherwise one q4q_mul_mat_ex call per matrix. */
Q4Q_API q4q_status q4q_mul_mat_group(int n, const void* const* src0, const int64_t* ne01, int64_t ne00,
                             const float* src1, int64_t ne10, int64_t ne11, float* const* dst,
                             void* workspace, size_t workspace_bytes, unsigned int flags,
                             q4q_stream_t stream);

/* ggml_get_rows on a quantized table (the embedding lookup that starts the Llama
 * graph of "llama.cpp 深度解读" §4, ggml_get_rows(tok_embeddings, inp_tokens), with
 * the token-embedding tensor stored as Q4_0 as §1's GGUF example shows):
 *   dst[i*ne00 + k] = decode(src0 row ids[i])[k],  decode as §2: (nibble - 8) * d
 *   (Q4_0) or q * d (Q8_0), exact in fp32.
 * src0: ne01 rows of ne00/32 blocks (2-byte aligned); ids: device int32 [n_ids]
 * (4-byte aligned), or NULL for rows 0 .. n_ids-1 (the whole-table decode, which
 * then requires n_ids <= ne01); dst: device fp32 [n_ids][ne00], 16-byte aligned.
 * An id outside [0, ne01) is not read: its output row is written as zeros and
 * Q4Q_ERR_ARG is recorded in the device status word (q4q_device_status).
 * Limits: 0 < ne00 < 2^20, ne00 % 32 == 0, 0 <= ne01, n_ids < 2^31. */
Q4Q_API q4q_status q4q_get_rows_q4_0(const void* src0, int64_t ne00, int64_t ne01, const int32_t* ids,
                             int64_t n_ids, float* dst, q4q_stream_t stream);
Q4Q_API q4q_status q4q_get_rows_q8_0(const void* src0, int64_t ne00, int64_t ne01, const int32_t* ids,
                             int64_t n_ids, float* dst, q4q_stream_t stream);

/* Bytes of device workspace q4q_mul_mat_q8_0 needs for this problem on the current
 * device (the tensor-core GEMM's operands for ne11 >= 8, the Q8_0 activations of
 * the generic path otherwise; the GEMV needs none). */
Q4Q_API q4q_status q4q_mul_mat_q8_0_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, size_t* bytes);

/* ggml_mul_mat with Q8_0 weights (the Q8_0 type of "llama.cpp 深度解读" §2's type
 * table; block {fp16 d; int8 qs[32]}, element k = qs[k] * d):
 *   dst[i11*ne01 + i01] = sum_b fp32(d_w * d_x) * isum,  isum = sum_k qw_k * qx_k,
 * src1 rows quantized to Q8_0 as q4q_quantize_q8_0 does.  src0: ne01 rows of
 * ne00/32 34-byte blocks (2-byte aligned); everything else as q4q_mul_mat_ex.
 * With ne00 % 256 == 0 and 16-byte aligned src0 / src1: ne11 < 8 runs the GEMV,
 * ne11 >= 8 the tensor-core GEMM of q4q_mul_mat with a Q8_0 dequantizer (256-byte
 * aligned workspace of q4q_mul_mat_q8_0_workspace_size bytes); otherwise a generic
 * kernel over Q8_0 activations in the workspace. */
Q4Q_API q4q_status q4q_mul_mat_q8_0(const void* src0, int64_t ne00, int64_t ne01,
                            const float* src1, int64_t ne10, int64_t ne11,
                            float* dst, void* workspace, size_t workspace_bytes,
                            unsigned int flags, q4q_stream_t stream);

/* Debug: per-block integer sums of Q8_0 weights and Q8_0 activations, out int32
 * [ne11][ne01][ne00/32], from the device routine of `path`: 0 = the Q8_0 GEMV's
 * block dot (requires ne00 % 64 == 0, 2-byte aligned inputs; no workspace),
 * 1 = the tensor-core GEMM with the Q8_0 dequantizer (requires ne00 % 256 == 0,
 * a 16-byte aligned src0 and q4q_debug_workspace_size(ne00, ne11, 1) bytes of
 * 256-byte aligned workspace).  Small shapes only (tests). */
Q4Q_API q4q_status q4q_debug_block_isums_q8_0(const void* src0_q8_0, const void* src1_q8_0, int64_t ne00,
                                      int64_t ne01, int64_t ne11, int path, int32_t* out,
                                      void* workspace, size_t workspace_bytes, q4q_stream_t stream);

/* Most links one q4q_mul_mat_chain call takes. */
#define Q4Q_CHAIN_MAX 64

/* One projection of a chain (one token): dst = ggml_mul_mat(src0 Q4_0 [ne00, ne01],
 * src1 F32 [ne00, 1]) -> F32 [ne01], computed as q4q_mul_mat computes it. */
typedef struct {
    const void* src0;     /* Q4_0 weights, ne01 rows of ne00/32 blocks; device, 16-byte aligned */
    int64_t ne00, ne01;   /* 0 < ne00 < 2^20 with ne00 % 256 == 0; 0 < ne01 < 2^31 */
    const float* src1;    /* fp32 [ne00]; device, 16-byte aligned; may be an earlier link's dst */
    float* dst;           /* fp32 [ne01]; device, 4-byte aligned */
} q4q_chain_link;

/* Bytes of device workspace q4q_mul_mat_chain needs for n links (a completion
 * count per link and an abort word); n: 1 .. Q4Q_CHAIN_MAX, else Q4Q_ERR_ARG. */
Q4Q_API q4q_status q4q_mul_mat_chain_workspace_size(int n, size_t* bytes);

/* A chain of dependent one-token projections in one launch: for i = 0 .. n-1, in
 * order, links[i].dst = ggml_mul_mat(links[i].src0, links[i].src1), each exactly as
 * q4q_mul_mat computes it.  This is the shape of a decode step: the "ggml GPT-2 117M
 * inference walkthrough" runs every layer's QKV projection (§3.2), its output
 * projection and MLP (§3.5) and finally the lm_head (§3.6) one after another, each
 * a ggml_mul_mat ("llama.cpp 深度解读" §3) whose input an earlier step produced.
 * Link i reads its src1 only after every earlier link has written all of its dst,
 * so src1 of link i may be (or overlap) the dst of any earlier link; it must not
 * overlap its own dst, and no dst may overlap any link's src0 (the weights of
 * later links are read ahead).  One persistent grid is launched cooperatively (all
 * of its CTAs resident at once): its CTAs stream every link's weights back to back
 * and meet at device-side completion counts between links, instead of one launch
 * per matrix.
 * links: HOST array of n entries (read during the call); n: 1 .. Q4Q_CHAIN_MAX;
 * ne11: must be 1 (one token), else Q4Q_ERR_SHAPE; flags: 0, else Q4Q_ERR_ARG;
 * workspace: device, 4-byte aligned, q4q_mul_mat_chain_workspace_size(n) bytes,
 * zeroed by the call on `stream` (calls that overlap on the GPU must not share it).
 * Every wait between links and on the weight stages is bounded (about one second):
 * one that runs out records Q4Q_ERR_TIMEOUT (q4q_device_status), raises the call's
 * abort and the remaining links are not computed. */
Q4Q_API q4q_status q4q_mul_mat_chain(const q4q_chain_link* links, int n, int64_t ne11, void* workspace,
                             size_t workspace_bytes, unsigned int flags, q4q_stream_t stream);

/* Size of the library-owned scratch array used by q4q_mul_mat_noalloc (per GPU). */
#define Q4Q_NOALLOC_SCRATCH_BYTES (8u << 20)

/* q4q_mul_mat for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for callers such as a plugin inside a host
 * application that owns every device allocation (an inference server with its
 * own memory pool, a runtime that forbids allocation after start-up) and so has
 * no workspace to pass.  It computes what q4q_mul_mat computes, with the same
 * arguments minus the workspace -- the same result within the library's output
 * bound (1e-5 of sum_b |d_w d_x isum_b|; the tensor-core path may split K fewer
 * ways than with a full workspace, which changes the fp32 summation order) --
 * and allocates nothing: the scratch space
 * that the tensor-core and generic paths need comes from one static device array
 * of Q4Q_NOALLOC_SCRATCH_BYTES that the library owns on every GPU that loads it,
 * until the process exits.
 *  - Limit: problems that need more than Q4Q_NOALLOC_SCRATCH_BYTES of scratch
 *    even without split-K partial sums are rejected with Q4Q_ERR_WORKSPACE before
 *    any launch (e.g. ne11 = 512 tokens fits up to ne00 = 7680; ne11 = 2048 does
 *    not fit at ne00 = 4096); others use as many K splits as the array holds.
 *  - Set-up: the first call on a device, made while that device is current,
 *    looks up the array's device address (cudaGetSymbolAddress) and caches it;
 *    make that first call before any stream capture.  A device reset
 *    (cudaDeviceReset) discards the array and with it the cached address: after
 *    one, the process must not call q4q_mul_mat_noalloc on that device again.
 *  - Sharing: every call on a device uses the same array, which keeps whatever
 *    the last call left in it (no call needs it to start at zero: each call
 *    rewrites every scratch byte it reads).  Calls that overlap on the GPU (on
 *    different streams, or from several host threads) race on it; serialize them. */
Q4Q_API q4q_status q4q_mul_mat_noalloc(const void* src0, int64_t ne00, int64_t ne01,
                               const float* src1, int64_t ne10, int64_t ne11,
                               float* dst, q4q_stream_t stream);

/* Debug: per-block integer sums isum(i01, i11, b) (§3's `sumi`) of Q4_0 weights
 * and already-quantized Q8_0 activations, computed by the device routine of the
 * chosen path: path 0 = the GEMV block-dot routine (dp4a on nibble words),
 * path 1 = the tensor-core GEMM (one 32-wide K block per fresh TMEM accumulator,
 * read back exactly as fp32 and converted to int32).
 * src0: ne01 rows x ne00/32 Q4_0 blocks; src1_q8_0: ne11 rows x ne00/32 Q8_0
 * blocks; out: int32 [ne11][ne01][ne00/32].  All device memory.
 * Path 0 requires ne00 % 64 == 0 and 2-byte aligned inputs; path 1 requires
 * ne00 % 256 == 0, a 16-byte aligned src0 and q4q_debug_workspace_size bytes of
 * 256-byte aligned workspace (path 0 ignores workspace).
 * Meant for small shapes (tests); it is not optimized. */
Q4Q_API q4q_status q4q_debug_block_isums(const void* src0, const void* src1_q8_0,
                                 int64_t ne00, int64_t ne01, int64_t ne11, int path,
                                 int32_t* out, void* workspace, size_t workspace_bytes,
                                 q4q_stream_t stream);

/* Debug, host only (no GPU needed): the GEMV launch plan for 1..7 tokens on a
 * device with sm_count SMs and smem_optin bytes of opt-in shared memory per CTA,
 * for weight blocks of weight_block_bytes (18: Q4_0, 34: Q8_0) and mats matrices
 * streamed side by side (1, or 2 for the SwiGLU kernel).  On Q4Q_OK, out[0 ..
 * Q4Q_DEBUG_GEMV_PLAN_FIELDS-1] receives: rows per unit, ring stages, bytes per
 * stage, dynamic shared memory, grid (without clusters), cluster size, lanes per
 * row, register-resident block pairs per lane, units, and the shared-memory
 * offsets of the activations, of the ring and of the second matrix's rows in a
 * stage, the row bytes, and the offsets of the activation scales and code sums.
 * Q4Q_ERR_SHAPE when the GEMV takes no such problem (the generic kernel runs it). */
#define Q4Q_DEBUG_GEMV_PLAN_FIELDS 15
Q4Q_API q4q_status q4q_debug_gemv_plan(int64_t ne00, int64_t ne01, int64_t ne11, int weight_block_bytes, int mats,
                               int sm_count, int smem_optin, int64_t* out);

/* Debug, host only: how many ways the tensor-core GEMM splits K for this problem
 * on a device with sm_count SMs, given enough workspace (1 = no split).  Requires
 * ne00 % 256 == 0, ne11 >= 8 and ne01 > 0, else Q4Q_ERR_ARG. */
Q4Q_API q4q_status q4q_debug_mma_splits(int64_t ne00, int64_t ne01, int64_t ne11, int sm_count, int* splits);

/* Debug: the failure path of the library's bounded waits, on its own.  Launches
 * one CTA whose thread waits, for at most limit_ns nanoseconds, on an mbarrier
 * phase that nothing completes (the wait every kernel uses for its copies and
 * hand-offs), then records Q4Q_ERR_TIMEOUT in the device status word and returns;
 * q4q_device_status reports it.  No GPU fault or hang is involved, and the context
 * stays usable.  limit_ns: 1 .. 1e9, else Q4Q_ERR_ARG. */
Q4Q_API q4q_status q4q_debug_wait_timeout(uint64_t limit_ns, q4q_stream_t stream);

/* Debug: the failure path of the matmul kernels' own bounded waits.  Runs the
 * kernel q4q_mul_mat would run for this problem -- path 0: the GEMV (ne11 1..7),
 * path 1: the tensor-core GEMM (ne11 >= 8), path 3: the warp-MMA kernel (ne11
 * 1..32) -- with every wait bounded by limit_ns nanoseconds and one hand-off left
 * out in its first CTA: that CTA's first stage of weights (GEMV), of activations
 * (GEMM) or of both (warp-MMA) is never copied, so the waits on it run out.  Path 2 (ne11 = 1): q4q_mul_mat_chain over two links of this matrix on
 * the same input, whose first CTA never reports the first link finished, so the
 * other CTAs' waits before the second link run out (workspace: that of a
 * two-link chain).  The CTA that gives up records Q4Q_ERR_TIMEOUT in the device status
 * word (read by q4q_device_status) and raises the call's abort; it and every CTA
 * of the call that then finds the abort raised wait (bounded) for their own copies
 * in flight, free their tensor memory and return.  No GPU fault or hang is
 * involved and the context stays usable; dst is left incomplete.  Arguments as
 * q4q_mul_mat (paths 1 and 3: its workspace); the problem must take the chosen path
 * (ne00 % 256 == 0, 16-byte aligned src0 and src1), else Q4Q_ERR_SHAPE.
 * limit_ns: 1 .. 1e9, path: 0, 1, 2 or 3, else Q4Q_ERR_ARG. */
Q4Q_API q4q_status q4q_debug_mul_mat_timeout(const void* src0, int64_t ne00, int64_t ne01, const float* src1,
                                     int64_t ne11, float* dst, void* workspace, size_t workspace_bytes,
                                     int path, uint64_t limit_ns, q4q_stream_t stream);

/* Debug: run one named path of q4q_mul_mat on a problem it accepts, whatever
 * q4q_mul_mat itself would pick -- path 0: the GEMV (ne11 1..7, no workspace), path
 * 1: the tensor-core GEMM (ne11 >= 8), path 3: the warp-MMA kernel (ne11 1..32).
 * Same operation, outputs and tolerance as q4q_mul_mat.  Requires ne00 % 256 == 0 and
 * 16-byte aligned src0 and src1 (else Q4Q_ERR_ALIGN / Q4Q_ERR_SHAPE); paths 1 and 3 take
 * 256-byte aligned workspace of at least their split-free minimum (see
 * q4q_mul_mat_workspace_size), and
 * split K as far as the workspace given allows.  path: 0, 1 or 3, else Q4Q_ERR_ARG;
 * ne01 == 0 or ne11 == 0: Q4Q_ERR_SHAPE. */
Q4Q_API q4q_status q4q_debug_mul_mat_path(const void* src0, int64_t ne00, int64_t ne01, const float* src1,
                                  int64_t ne11, float* dst, void* workspace, size_t workspace_bytes,
                                  int path, q4q_stream_t stream);

/* Bytes of workspace q4q_debug_mul_mat_path's `path` plans its split-K for (0 for path 0). */
Q4Q_API q4q_status q4q_debug_mul_mat_path_workspace_size(int64_t ne00, int64_t ne01, int64_t ne11, int path,
                                                 size_t* bytes);

/* Synchronizes the device, returns (in *status) the first device-side error
 * recorded since the last call (Q4Q_OK if none) and clears it.  This is where a
 * bounded wait that ran out (Q4Q_ERR_TIMEOUT) or an out-of-range row id of
 * q4q_get_rows_* (Q4Q_ERR_ARG) is reported: the call whose kernel recorded it has
 * already returned, and its output is incomplete.  A recorded error does not
 * affect later calls. */
Q4Q_API q4q_status q4q_device_status(q4q_status* status);

/* Static string for a status code. */
Q4Q_API const char* q4q_status_string(q4q_status status);

/* Library ABI version: (major << 16) | minor. */
Q4Q_API int q4q_version(void);

#ifdef __cplusplus
}
#endif
#endif /* Q4Q_H */
