/*
 * qdecode.h — C ABI of libqdecode, the single-token decode path of a llama-style
 * transformer over block-quantised weights, for NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (the pages on quantized decode GEMV; each entry point
 * below names its passage):
 *   [llmoxide]  "Running an LLM, then forgetting it" (llmoxide blog), sections
 *               1 "A neuron is a dot product", 2 "Layers, and the bend between them",
 *               3 "Text in, vectors out", 4 "Keeping the numbers in range",
 *               5 "Attention", 6 "Where things are: RoPE", 7 "The block, and the
 *               residual stream", 10 "Loading weights", 11 "Prefill and decode",
 *               12 "The KV cache".
 *   [go-llm]    "llm" Go package documentation (go-wasmcontainers/llm v0.1.0):
 *               package overview, "Design points", "Oracle tolerances", index
 *               (Argmax, F16ToF32, RoundF16, type CPU and ExactGGML, CPU.Forward,
 *               CPU.Reset, CPU.Pos, Config).
 *   [llamini]   "Building llamini.cpp: a from-scratch llama.cpp core in C99",
 *               summary table ("Quants"), "What I reimplemented" (Q4_K
 *               scale/min unpacking), "Optimizing for CPU, and finding out what
 *               was actually true".
 *   [dasLLAMA]  "dasLLAMA-00 - The Problem Statement", 8.7.1.4 "Five small
 *               functions", 8.7.1.6.2 "Attention", 8.7.1.6.3 "Feed-forward",
 *               8.7.1.6.4 "Logits", 8.7.1.7 "Prompting is repeated forward".
 *   [minillm]   minillm-cpp README, "Loader", "Direct INT8 loading", "NEON
 *               kernels", "Quantization".
 *
 * Conventions for every entry point:
 *  - Device pointers unless stated "host".  The caller owns and allocates every
 *    buffer; no entry point calls cudaMalloc or frees caller memory.  (The model
 *    object is a small host struct; the first qd_decode_step of each batch size
 *    captures and instantiates a CUDA graph, which the driver allocates for itself.)
 *  - All device work is enqueued on `stream` and is asynchronous; host-side
 *    results (sizes, statuses) are synchronous.
 *  - Every call validates its arguments before enqueuing anything.  A failed check
 *    returns a status other than QD_OK and enqueues nothing.  Launch failures
 *    return QD_ERR_CUDA.  Kernels never trap: a condition only the device can see
 *    (a token id or position out of range inside a captured step) sets a bit in the
 *    model's device error word and the kernel skips the access; qd_model_check
 *    reports it.
 *  - Activations are f32, batch-major: x[batch][n].  Batch is 1..QD_MAX_BATCH.
 *  - Every device buffer must be 16-byte aligned.
 *  - No entry point is thread-safe on the same model or buffers.
 */
#ifndef QDECODE_H
#define QDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* qd_stream_t;

#define QD_MAX_BATCH 16

typedef enum {
    QD_OK = 0,
    QD_ERR_INVALID_ARG = 1, /* null pointer, bad enum, negative size          */
    QD_ERR_SHAPE = 2,       /* size not allowed for the format / operation     */
    QD_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned         */
    QD_ERR_UNSUPPORTED = 4, /* unknown format, pairing or configuration        */
    QD_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed     */
    QD_ERR_NOMEM = 6,       /* a caller-provided buffer is too small           */
    QD_ERR_DEVICE_FLAG = 7  /* a kernel flagged an out-of-range token/position */
} qd_status;

/* Weight formats ([llmoxide] 10; [go-llm] "Design points"; [llamini]; [minillm]
 * "Quantization"):
 *  QD_Q4_0   blocks of 32 weights, 18 B: f16 d, 16 B of 4-bit codes; value (q-8)*d.
 *            Element j (0..15) is the low nibble of code byte j, element j+16 its
 *            high nibble.
 *  QD_Q8_0   blocks of 32 weights, 34 B: f16 d, 32 int8 codes; value q*d.
 *  QD_Q4_K   super-blocks of 256 weights, 144 B: f16 d, f16 dmin, 12 B of packed
 *            6-bit (scale, min) for 8 sub-blocks of 32, 128 B of 4-bit codes;
 *            value d*sc*q - dmin*m.  Code byte 32c+l holds element 64c+l (low
 *            nibble, sub-block 2c) and element 64c+32+l (high nibble, sub-block 2c+1).
 *  QD_I8_ROW per-row symmetric INT8: int8 codes [rows][cols], then one f32 scale
 *            per row; value q*s_row.
 * The formats a Q4_K_M-class file mixes in ([go-llm] package overview: its first
 * model's Q4_0 file holds Q4_0, Q4_1 and Q8_0 tensors; [llamini] summary table,
 * "Quants": Q4_K, Q6_K, Q5_0, Q5_K, Q4_0, Q4_1, Q8_0, F16; [llmoxide] 10: Q6_K).  The pages name them and give Q6_K's 6.6 bits per weight; the
 * byte layouts (not on the pages) are the GGUF ones:
 *  QD_Q4_1   blocks of 32, 20 B: f16 d, f16 m, 16 B of 4-bit codes (order as Q4_0);
 *            value d*q + m.
 *  QD_Q5_0   blocks of 32, 22 B: f16 d, 4 B qh (little-endian; bit j is the fifth bit
 *            of element j), 16 B of low nibbles (order as Q4_0); value (q-16)*d.
 *  QD_Q5_K   super-blocks of 256, 176 B: f16 d, f16 dmin, 12 B of 6-bit (scale, min)
 *            as Q4_K, 32 B qh, 128 B of low nibbles (order as Q4_K); element 64c+l
 *            takes bit 2c of qh[l] as its fifth bit, element 64c+32+l bit 2c+1;
 *            value d*sc*q - dmin*m.
 *  QD_Q6_K   super-blocks of 256, 210 B: 128 B ql (low nibbles), 64 B qh (two-bit
 *            high parts), 16 int8 scales (one per 16 weights), f16 d; in half h
 *            (elements 128h..128h+127) element 128h+32k+l (k 0..3, l 0..31) takes the
 *            low (k < 2) or high (k >= 2) nibble of ql[64h + l + 32 (k & 1)], bits
 *            2k, 2k+1 of qh[32h + l] above it, and scale 8h + 2k + l/16;
 *            value d*sc*(q-32).
 *  QD_F16    binary16 weights, 2 B each (little-endian).
 *  QD_I4_ROW per-row symmetric INT4 ([minillm] "Quantization": INT8 and INT4, one
 *            scale per output row): codes [rows][cols/2], two per byte (element 2i in
 *            the low nibble, two's complement, -7..7), then one f32 scale per row;
 *            value q*s_row.
 * The "source" layout of a tensor is the model-file layout above, rows in order
 * (for QD_I8_ROW: all codes, then all scales, in one buffer).  The decode step
 * (qd_model_*) takes every format but QD_I4_ROW, for each class of layer matrix and for
 * the embedding; the layout calls, qd_dequant, qd_embed and qd_q_gemv take every format. */
typedef enum {
    QD_Q4_0 = 0,
    QD_Q8_0 = 1,
    QD_Q4_K = 2,
    QD_I8_ROW = 3,
    QD_Q4_1 = 4,
    QD_Q5_0 = 5,
    QD_Q5_K = 6,
    QD_Q6_K = 7,
    QD_F16 = 8,
    QD_I4_ROW = 9
} qd_fmt;

/* RoPE pairing ([llmoxide] 6): ADJACENT rotates (2i, 2i+1) (llama files), HALF
 * rotates (i, i + head_dim/2) (NeoX/Qwen). */
typedef enum { QD_ROPE_ADJACENT = 0, QD_ROPE_HALF = 1 } qd_rope_pairing;

const char* qd_status_str(qd_status s);
int qd_abi_version(void);

/* ------------------------------------------------------------------------- */
/* Scalar conversions ([go-llm] index F16ToF32; [minillm] "Loader").          */
/* ------------------------------------------------------------------------- */

/* Device kernels converting n binary16 / bfloat16 bit patterns to f32 (exact;
 * bf16 is the zero-extension bits << 16).  in, out: device, n >= 0. */
qd_status qd_f16_to_f32(const uint16_t* in, float* out, int64_t n, qd_stream_t stream);
qd_status qd_bf16_to_f32(const uint16_t* in, float* out, int64_t n, qd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Load-time repacking ([go-llm] "Design points": blocks are repacked into    */
/* aligned quants and scales on upload).                                      */
/* Packed layouts (all regions 16-byte aligned, rows in order):               */
/*  Q4_0: codes [rows][cols/32][16 B], then f16 d [rows][cols/32].            */
/*  Q8_0: codes [rows][cols/32][32 B], then f16 d [rows][cols/32].            */
/*  Q4_K: codes [rows][cols/256][128 B], then headers [rows][cols/256][16 B]  */
/*        (d, dmin, 12 scale bytes).                                          */
/*  I8_ROW: codes [rows][cols], then f32 scales [rows].                       */
/*  Q4_1: codes [rows][cols/32][16 B], then (d, m) [rows][cols/32][4 B].      */
/*  Q5_0: low nibbles [rows][cols/32][16 B], then (d, qh) [rows][cols/32][6 B]. */
/*  Q5_K: (qh, low nibbles) [rows][cols/256][160 B], then headers            */
/*        [rows][cols/256][16 B] (d, dmin, 12 scale bytes).                   */
/*  Q6_K: (ql, qh) [rows][cols/256][192 B], then (16 scales, d)               */
/*        [rows][cols/256][18 B].                                             */
/*  F16:  weights [rows][cols] (2 B each); no scale region.                   */
/*  I4_ROW: codes [rows][cols/32][16 B], each 32-element unit in Q4_0's order  */
/*        (element j: low nibble of byte j, j+16: its high nibble) and in      */
/*        offset binary (q + 8); then f32 scales [rows].                      */
/* The repack is lossless: qd_unpack restores the source bytes exactly.       */
/* ------------------------------------------------------------------------- */

/* Bytes of the source / packed layout; 0 for a shape the format does not allow
 * (rows < 1, cols < 1, cols % 32 for Q4_0/Q8_0/Q4_1/Q5_0/F16/I4_ROW, cols % 256
 * for Q4_K/Q5_K/Q6_K, cols % 16 for I8_ROW). */
size_t qd_src_bytes(qd_fmt fmt, int64_t rows, int64_t cols);
size_t qd_packed_bytes(qd_fmt fmt, int64_t rows, int64_t cols);

/* src (device, source layout, qd_src_bytes) -> dst (device, packed layout,
 * dst_bytes >= qd_packed_bytes).  src and dst must not overlap. */
qd_status qd_repack(qd_fmt fmt, const void* src, int64_t rows, int64_t cols, void* dst, size_t dst_bytes,
                    qd_stream_t stream);
/* Inverse of qd_repack (for tests): packed -> source layout (dst_bytes >= qd_src_bytes). */
qd_status qd_unpack(qd_fmt fmt, const void* packed, int64_t rows, int64_t cols, void* dst, size_t dst_bytes,
                    qd_stream_t stream);
/* Dequantised values of a packed tensor: out f32 [rows][cols] (device), each value
 * rounded once to f32 (for the bit-exact block-value tests). */
qd_status qd_dequant(qd_fmt fmt, const void* packed, int64_t rows, int64_t cols, float* out, qd_stream_t stream);

/* Load-time per-row INT8 quantisation of BF16 weights ([minillm] "Direct INT8
 * loading": each matrix quantised row by row from the BF16 checkpoint;
 * "Quantization": symmetric, one scale per output row).  The page prints no rule;
 * the one implemented: s_r = max_c |w_rc| / 127 in f32, q_rc = w_rc / s_r (f32)
 * rounded to nearest with ties away from zero, clamped to [-127, 127]; a row of
 * zeros gets s_r = 0 and codes 0, a row holding a non-finite value codes 0 and a NaN
 * scale.  w_bf16: device bf16 bit patterns [rows][cols] (16-byte aligned; value =
 * bits << 16 as f32).  out: device, the QD_I8_ROW source layout (codes [rows][cols],
 * then f32 scales [rows]; out_bytes >= qd_src_bytes(QD_I8_ROW, rows, cols)), ready for
 * qd_repack or a model's INT8 weights; must not overlap w_bf16.  cols % 16 == 0. */
qd_status qd_quantize_i8_rows(const uint16_t* w_bf16, int64_t rows, int64_t cols, void* out, size_t out_bytes,
                              qd_stream_t stream);

/* The same for per-row INT4 ([minillm] "Quantization"): s_r = max_c |w_rc| / 7 (f32),
 * q_rc = w_rc / s_r (f32) rounded to nearest with ties away from zero, clamped to
 * [-7, 7]; zero and non-finite rows as above.  out: the QD_I4_ROW source layout (codes
 * [rows][cols/2], then f32 scales [rows]; out_bytes >= qd_src_bytes(QD_I4_ROW, rows,
 * cols)).  cols % 32 == 0. */
qd_status qd_quantize_i4_rows(const uint16_t* w_bf16, int64_t rows, int64_t cols, void* out, size_t out_bytes,
                              qd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Fused dequantise-and-dot GEMV ([llmoxide] 1 matvec, 10 (the Q8_0 row dot), */
/* 11 (t rows of x through one read of W); [dasLLAMA] 8.7.1.4 matmul;         */
/* [minillm] "NEON kernels": fused, no f32 temporary).                        */
/* y[b][r] = sum_c deq(W)[r][c] * x[b][c], for b < batch, r < rows.           */
/* W: packed layout (qd_repack).  x: f32 [batch][cols].  y: f32 [batch][rows], */
/* must not overlap x.  batch 1..16.  workspace: currently unused (pass NULL, 0);*/
/* qd_q_gemv_workspace returns the bytes a call needs.                         */
/* Arithmetic: codes meet x through integer dot products, x held per 32-element */
/* unit as 24-bit integers with a power-of-two scale (at most 2^-23 of the      */
/* unit's largest |x| per element); sums are f32.  Batch 3-16 with Q4_0, Q8_0  */
/* or INT8 rows runs on the tensor cores instead: codes exact in binary16, x   */
/* per 256-element stage scaled by a power of two and split into two binary16 */
/* parts (at most 2^-22 of the stage's largest |x| per element), products     */
/* summed in f32; x rows wider than one CTA's shared memory holds split their */
/* columns over a thread-block cluster (partial sums added in a fixed order), */
/* or run as several launches over column ranges (added in a fixed order), or */
/* (batch 9-16) as two passes of up to 8 batch rows.  Batch 9-16 INT8 rows    */
/* that fit none of these run on the 5th-generation tensor cores (the same    */
/* split of x).  Results are the same bits on every run.  A non-finite x      */
/* gives NaN in its batch row.                                                 */
/* ------------------------------------------------------------------------- */
size_t qd_q_gemv_workspace(qd_fmt fmt, int64_t rows, int64_t cols, int batch);
qd_status qd_q_gemv(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                    void* workspace, size_t workspace_bytes, qd_stream_t stream);

/* qd_q_gemv with launch flags.  QD_GEMV_OVERLAP: the kernel may start streaming W
 * while the kernel before it on `stream` is still running (programmatic dependent
 * launch), as the decode step launches its projections; x and y are still read and
 * written only after that kernel has finished.  Only valid when no kernel that can
 * still be running on `stream` writes W.  No flags: same as qd_q_gemv.  Unknown
 * flag bits: QD_ERR_INVALID_ARG. */
#define QD_GEMV_OVERLAP 1u

/* Roofline calibration (no counterpart on the pages: measurement support).  Reads every
 * byte of buf (device, 16-byte aligned, bytes a multiple of 16) once with 16-byte streaming
 * loads and computes nothing: the bandwidth one launch of a plain read reaches on this GPU
 * for a buffer of that size, the ceiling a GEMV streaming the same bytes can be compared
 * with.  Grid: ctas_per_sm (1..8) CTAs per SM of `threads` (128, 256 or 512) threads, each
 * CTA one contiguous run.  flags: QD_GEMV_OVERLAP launches it as a programmatic dependent
 * that waits for its predecessor only before its last write, as a GEMV waits before it
 * reads x.  sink: device word that the kernel writes only on an improbable XOR value. */
qd_status qd_read_ceiling(const void* buf, size_t bytes, int ctas_per_sm, int threads, unsigned flags,
                          uint32_t* sink, qd_stream_t stream);
qd_status qd_q_gemv_ex(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                       unsigned int flags, qd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Batched prefill product ([llmoxide] 11 "Prefill and decode": the decode     */
/* product with t rows of x through one read of the weights, compute-bound;    */
/* its Metal GEMM dequantises a weight tile once into on-chip memory for the   */
/* matrix units).  y[n][r] = sum_c deq(W)[r][c] * x[n][c] for n < t, r < rows. */
/* fmt: QD_Q4_0, QD_Q8_0 or QD_I8_ROW (others: QD_ERR_UNSUPPORTED).  W: packed  */
/* layout (qd_repack).  x: f32 [t][cols].  y: f32 [t][rows], must not overlap  */
/* x or the workspace.  cols a multiple of 64, 1 <= t <= QD_MAX_GEMM_TOKENS.     */
/* workspace: device, 16-byte aligned, >= qd_q_gemm_workspace bytes (0 for an  */
/* unsupported format or shape; a smaller one: QD_ERR_NOMEM, as for the other */
/* workspaces); it holds the split x between the call's two kernels and may be */
/* reused once the call has completed on `stream`.                              */
/* Arithmetic (5th-generation tensor cores, f32 accumulation): each token's x  */
/* is scaled by a power of two and split into two binary16 parts (about 2^-22  */
/* relative); Q4_0 / Q8_0 weights enter as the binary16 rounding of d * q       */
/* (relative error at most 2^-11 per weight; for |d * q| below 2^-14 the        */
/* binary16 subnormal step 2^-24 bounds it); INT8 codes enter exactly and the   */
/* row scale is applied in f32.  A non-finite x row gives NaN in its y row.     */
/* ------------------------------------------------------------------------- */
#define QD_MAX_GEMM_TOKENS 65536
size_t qd_q_gemm_workspace(qd_fmt fmt, int64_t rows, int64_t cols, int t);
qd_status qd_q_gemm(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int t,
                    void* workspace, size_t workspace_bytes, qd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* ggml-exact activations ([go-llm] type CPU, "ExactGGML": activations are     */
/* quantised to Q8_0, Q8_1 for Q4_1 weights, before every quantised product)  */
/* and the product over them in integers ([llamini] "Optimizing for CPU, and  */
/* finding out what was actually true": ggml multiplies packed bytes and      */
/* converts only the scaled sum to float).                                     */
/* Quantisation (the page prints no rule), per 32 values of a row of x:       */
/* d = max|x| / 127 and q = x / d rounded to nearest, ties away from zero,    */
/* clamped to +-127, both divisions IEEE round-to-nearest in f32; d is kept   */
/* as binary16 and, with with_sum (Q8_1), s = d * sum(q) as binary16.  A zero */
/* block has d = 0 and codes 0; a block holding a non-finite value codes 0    */
/* and d = s = NaN.  Buffer layout (device, each region 16-byte aligned):     */
/* int8 codes [batch][cols], then f16 d [batch][cols/32], then (with_sum)      */
/* f16 s [batch][cols/32]; qd_q8_bytes gives its size (0: bad shape).          */
/* batch 1..QD_MAX_BATCH, cols a multiple of 32.                               */
/* qd_q_gemv_q8: y[b][r] = sum over blocks k of d_w d_x sum_j q_w q_x (Q4_0:  */
/* q_w - 8; Q4_1: plus m_w s_x, so its activations need with_sum = 1), f32.   */
/* fmt: QD_Q4_0, QD_Q8_0 or QD_Q4_1.  y: f32 [batch][rows].                    */
/* ------------------------------------------------------------------------- */
size_t qd_q8_bytes(int batch, int64_t cols, int with_sum);
qd_status qd_quantize_q8(const float* x, int batch, int64_t cols, int with_sum, void* out, size_t out_bytes,
                         qd_stream_t stream);
qd_status qd_q_gemv_q8(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const void* xq, size_t xq_bytes,
                       float* y, int batch, qd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Decode-step operations                                                      */
/* ------------------------------------------------------------------------- */

/* RMSNorm ([llmoxide] 4 rms_norm_mul; [dasLLAMA] 8.7.1.6.2 rmsnorm):
 * out[b][i] = x[b][i] * g[i] / sqrt(mean_i(x[b][i]^2) + eps).  x, out: f32
 * [batch][n] (may alias); g: f32 [n].  n 1..65536, eps >= 0. */
qd_status qd_rmsnorm(const float* x, const float* g, float* out, int n, int batch, float eps, qd_stream_t stream);

/* Host: fill dst_host f32 [ctx][head_dim/2][2] with (cos, sin) of the angle
 * p * theta^(-2i/head_dim), computed in double and rounded to f32 ([go-llm]
 * "Design points": RoPE angles on the CPU in double precision).  head_dim even. */
qd_status qd_rope_table(float theta, int head_dim, int ctx, float* dst_host);

/* RoPE in place ([llmoxide] 6 rope; [dasLLAMA] 8.7.1.6.2 rope): rotate each of the
 * n_heads heads of row b of v (v + b*batch_stride, f32 [n_heads][head_dim]) by the
 * angles of position pos[b] (device int32 [batch]) from cos_sin (device, the table
 * of qd_rope_table for max_ctx positions).  A pos[b] outside [0, max_ctx) leaves
 * that row unchanged. */
qd_status qd_rope(float* v, int n_heads, int head_dim, int64_t batch_stride, const int32_t* pos,
                  qd_rope_pairing pairing, const float* cos_sin, int max_ctx, int batch, qd_stream_t stream);

/* KV-cache append ([llmoxide] 12; [dasLLAMA] 8.7.1.6.2: the rotated K and the V of
 * the current token go to the layer's cache at its position).  k, v: rows
 * b*src_batch_stride of f32 [n_kv_heads][head_dim]; caches: f32
 * [batch][n_kv_heads][max_ctx][head_dim]; position pos[b] (device).  A pos[b]
 * outside [0, max_ctx) writes nothing for that row. */
qd_status qd_kv_append(const float* k, const float* v, int64_t src_batch_stride, float* k_cache, float* v_cache,
                       int n_kv_heads, int head_dim, const int32_t* pos, int max_ctx, int batch,
                       qd_stream_t stream);

/* Causal grouped-query decode attention ([llmoxide] 5; [dasLLAMA] 8.7.1.6.2 score,
 * softmax and weighted sum).  For row b and q head h: kvh = h / (n_heads /
 * n_kv_heads); s_p = q.k_p / sqrt(head_dim) over p = 0..pos[b]; out = sum_p
 * softmax(s)_p v_p.  q: f32 [batch][n_heads][head_dim] (row stride q_batch_stride);
 * caches as in qd_kv_append; out: f32 [batch][n_heads][head_dim].  head_dim 64
 * (the models here); n_heads % n_kv_heads == 0, group size <= 8.  The context is
 * split across CTAs and merged with log-sum-exp weights; workspace (device) holds
 * the partial results, qd_gqa_decode_attn_workspace bytes.  A pos[b] outside
 * [0, max_ctx) yields zeros for that row. */
size_t qd_gqa_decode_attn_workspace(int n_heads, int head_dim, int max_ctx, int batch);
qd_status qd_gqa_decode_attn(const float* q, int64_t q_batch_stride, const float* k_cache, const float* v_cache,
                             float* out, int n_heads, int n_kv_heads, int head_dim, const int32_t* pos, int max_ctx,
                             int batch, void* workspace, size_t workspace_bytes, qd_stream_t stream);

/* Allocation-free variant of qd_gqa_decode_attn.  The pages have no counterpart: this is
 * an interface convenience, not part of the method.  Some callers cannot allocate device
 * memory for a workspace: code that runs after a fixed memory budget has been handed out
 * (another allocator or runtime owns the rest of the device), and loops that must not
 * call cudaMalloc because it can synchronise the device or fail at an unpredictable
 * moment.  This entry point takes the same inputs and outputs as qd_gqa_decode_attn
 * (same meaning, layout and validation) but keeps its partial results in a fixed 8 MiB
 * device array inside the library.  It calls no cudaMalloc or cudaFree.
 *  - When the array is reserved: the CUDA driver reserves it when it loads the library's
 *    module holding this function on a device, and keeps it until the process exits.
 *    Under CUDA's lazy module loading (the default since CUDA 12.2) that load can happen
 *    on the first call of this entry point on a device, and is itself a driver-side
 *    allocation that may synchronise.  So make one warm-up call on each device at set-up,
 *    before any stream capture and before any loop that must not allocate.
 *  - Size limit: calls whose workspace (qd_gqa_decode_attn_workspace) would exceed
 *    8 MiB return QD_ERR_NOMEM and enqueue nothing.  The largest configuration here,
 *    32 heads at context 4096 with batch 16, needs 4.3 MB.
 *  - The first call on each device also looks up the array's device address (with that
 *    device current); the warm-up call above covers it.
 *  - All calls share the one array and leave their partials in it.  Nothing needs to
 *    start at zero, but calls that overlap on the GPU (e.g. on two streams) race on it:
 *    order them on one stream. */
qd_status qd_gqa_decode_attn_noalloc(const float* q, int64_t q_batch_stride, const float* k_cache,
                                     const float* v_cache, float* out, int n_heads, int n_kv_heads, int head_dim,
                                     const int32_t* pos, int max_ctx, int batch, qd_stream_t stream);

/* SwiGLU gate ([llmoxide] 2; [dasLLAMA] 8.7.1.6.3): out = silu(gate) * up with
 * silu(z) = z / (1 + exp(-z)).  f32 [batch][n] each. */
qd_status qd_swiglu(const float* gate, const float* up, float* out, int64_t n, int batch, qd_stream_t stream);

/* Greedy argmax ([go-llm] index Argmax; [dasLLAMA] 8.7.1.6.4 most_likely): the
 * index of the largest of logits[b][0..n), the first such index on ties.
 * out_idx: device int32 [batch].  NaN never wins (inputs are expected NaN-free). */
qd_status qd_argmax(const float* logits, int64_t n, int batch, int32_t* out_idx, qd_stream_t stream);

/* Embedding lookup ([llmoxide] 3; [dasLLAMA] 8.7.1.6.1): x[b] = deq(E)[tokens[b]].
 * E: packed [vocab][dim]; tokens: device int32 [batch]; an id outside [0, vocab)
 * writes zeros. */
qd_status qd_embed(qd_fmt fmt, const void* E, int64_t vocab, int64_t dim, const int32_t* tokens, int batch,
                   float* x, qd_stream_t stream);

/* ------------------------------------------------------------------------- */
/* Model and decode step ([llmoxide] 7, 11, 12; [dasLLAMA] 8.7.1.6 forward,    */
/* 8.7.1.7; [go-llm] CPU.Forward / Reset / Pos, "Design points").             */
/* ------------------------------------------------------------------------- */

typedef struct {
    int layers, dim, ffn, n_heads, n_kv_heads, head_dim, vocab;
    int max_ctx;   /* positions per sequence in the KV cache                  */
    int max_batch; /* independent sequences per step, 1..16                  */
    float rope_theta, eps;
    qd_rope_pairing pairing;
    qd_fmt w_fmt;   /* the seven matrices of every layer                        */
    qd_fmt emb_fmt; /* token embedding (and output head)                        */
    int tied;       /* 1: logits use the token embedding as output head         */
    int kv_f16;     /* 0: f32 KV cache; 1: binary16 KV cache (go-llm's ggml-exact  */
                    /* cache: k and v rounded to nearest binary16 when appended,  */
                    /* read back exactly; half the cache bytes)                   */
    int act_q8;     /* 0: products over f32 activations; 1: every quantised       */
                    /* product over Q8_0 activations (qd_quantize_q8 rule) in     */
                    /* integers (go-llm's ggml-exact products); the layer formats */
                    /* and emb_fmt must then be QD_Q4_0 or QD_Q8_0.  With kv_f16 = */
                    /* 1 this is the pages' whole ggml-exact mode.                 */
    int mixed_fmt;  /* 0: every layer matrix takes w_fmt; 1: each class takes its  */
                    /* own format below and w_fmt is unused (model files mix      */
                    /* formats by tensor, e.g. Q4_K with Q6_K: [llamini] "Quants", */
                    /* [go-llm] package overview)                                  */
    qd_fmt qkv_fmt;     /* wq, wk, wv (one fused matrix)                           */
    qd_fmt wo_fmt;      /* attention output                                       */
    qd_fmt gate_up_fmt; /* wg, wu (one fused matrix)                              */
    qd_fmt down_fmt;    /* wd                                                     */
} qd_config;

typedef struct qd_model qd_model;

/* Bytes of the caller-provided regions: packed weights, and state (KV cache,
 * activations, positions, error word, rope table; the flat-split attention's partials
 * and counters when the model takes it; with act_q8 one quantised-input slot per product,
 * 4 * layers + 1 of them).
 * 0 for an invalid config (including act_q8 with formats other than Q4_0 / Q8_0, and
 * the formats the decode step does not take). */
size_t qd_model_weight_bytes(const qd_config* cfg);
size_t qd_model_state_bytes(const qd_config* cfg);

/* Build a model.  src_tensors: 3 + 9*layers device pointers to source-layout
 * tensors: [0] token embedding (emb_fmt, vocab x dim), [1] output norm gains f32
 * [dim], [2] output head (emb_fmt) or NULL when tied, then for layer l at 3+9l:
 * attn_norm f32[dim], wq (n_heads*head_dim x dim), wk, wv (n_kv_heads*head_dim x
 * dim), wo (dim x n_heads*head_dim), ffn_norm f32[dim], wg, wu (ffn x dim), wd
 * (dim x ffn).  They are repacked into weight_mem (fused QKV rows and interleaved
 * gate/up rows) on `stream`; the sources may be freed once the stream has passed
 * this point.  state_mem is zeroed (empty caches, pos 0).  *out receives a host
 * object, freed by qd_model_destroy. */
qd_status qd_model_create(const qd_config* cfg, const void* const* src_tensors, void* weight_mem,
                          size_t weight_bytes, void* state_mem, size_t state_bytes, qd_stream_t stream,
                          qd_model** out);
void qd_model_destroy(qd_model* m);

/* One greedy decode step for sequences 0..batch-1 at their current positions:
 * embed tokens[b], run every layer (appending K, V at pos[b]), compute the logits,
 * write argmax to out_tokens[b], advance pos[b].  tokens / out_tokens may be host
 * or device pointers (int32 [batch]); logits_out (f32 [batch][vocab], host or
 * device) may be NULL.  The step is one CUDA graph replay on `stream` (captured on
 * the first step of each batch size); host pointers make the call wait for the
 * copies.  A prompt can run as this call once per token (the Go package's "Results"
 * section runs its prompt that way, one decode pass per token) or through qd_prefill. */
qd_status qd_decode_step(qd_model* m, const int32_t* tokens, int batch, int32_t* out_tokens, float* logits_out,
                         qd_stream_t stream);

/* Batched prefill ([llmoxide] 11 "Prefill and decode": the prompt's t tokens go through
 * every product as one t-row matrix, so each weight tile is read once for all of them).
 * Runs the t prompt tokens of sequence `seq` (0 <= seq < max_batch) at positions
 * pos[seq] .. pos[seq] + t - 1: embeds them, runs every layer over the t rows (RMSNorm,
 * QKV product, RoPE and the cache append at each token's position, causal attention of
 * token i over positions 0 .. pos[seq] + i, output projection and residual, SwiGLU
 * feed-forward and residual), then the output head on the last token: its greedy token
 * to *out_token and, if logits_out is not NULL, its logits (f32 [vocab]).  pos[seq]
 * advances by t.  The cache and the returned values equal those of t decode steps of that
 * sequence, up to the products' arithmetic:
 *  - flags 0: with Q4_0, Q8_0 or INT8 layer weights, column counts (dim, heads * 64, ffn)
 *    that are multiples of 64 and t > 16, the layer products run on qd_q_gemm's tensor-core
 *    GEMM (Q4_0 / Q8_0 weights rounded to binary16, see qd_q_gemm); otherwise as below.
 *  - QD_PREFILL_EXACT: the layer products run on the batched GEMV (qd_q_gemv's arithmetic,
 *    as the decode step), 16 tokens a launch.
 * The head always runs the decode step's GEMV.  tokens: host or device int32 [t]; ids
 * outside [0, vocab) embed zeros and set the device flag (qd_model_check), as do
 * positions past max_ctx.  out_token (int32) and logits_out: host or device.
 * workspace: device, 256-byte aligned, >= qd_prefill_workspace(cfg, t) bytes (smaller:
 * QD_ERR_NOMEM); it may be reused once the call has completed on `stream`.
 * 1 <= t <= min(max_ctx, QD_MAX_GEMM_TOKENS) (else QD_ERR_SHAPE); models with act_q8 = 1:
 * QD_ERR_UNSUPPORTED; unknown flag bits: QD_ERR_INVALID_ARG.  Kernels are launched
 * directly on `stream` (no graph). */
#define QD_PREFILL_EXACT 1u
size_t qd_prefill_workspace(const qd_config* cfg, int t);
qd_status qd_prefill(qd_model* m, int seq, const int32_t* tokens, int t, unsigned flags, void* workspace,
                     size_t workspace_bytes, int32_t* out_token, float* logits_out, qd_stream_t stream);

/* Zero the KV cache and set every position to 0 ([go-llm] CPU.Reset). */
qd_status qd_model_reset(qd_model* m, qd_stream_t stream);
/* Set the positions of sequences 0..batch-1 (host int32 [batch]) (e.g. after
 * filling the cache directly). */
qd_status qd_model_set_pos(qd_model* m, const int32_t* pos_host, int batch, qd_stream_t stream);
/* Read positions (host int32 [batch]); synchronises `stream` ([go-llm] CPU.Pos). */
qd_status qd_model_pos(qd_model* m, int32_t* pos_host, int batch, qd_stream_t stream);
/* Device pointers to the KV cache, [layers][max_batch][n_kv_heads][max_ctx][head_dim] of
 * f32 (kv_f16 == 0) or binary16 bit patterns (kv_f16 == 1). */
qd_status qd_model_kv_cache(qd_model* m, void** k_cache, void** v_cache);
/* The quantised inputs of the last step of a model created with act_q8 == 1 (buf NULL,
 * slot_bytes 0 and slots 0 otherwise): one slot per quantised input, slot k at
 * buf + k * slot_bytes, in step order -- for layer l the QKV input (4l), the attention
 * output (4l + 1), the feed-forward input (4l + 2) and the SwiGLU output (4l + 3) -- then
 * the head's input (slot 4 * layers).  After a step over `batch` sequences, a slot of an
 * input of length n holds it in the layout of qd_quantize_q8: int8 codes [batch][n], then,
 * from byte offset batch*n rounded up to 16, f16 d [batch][n/32].  For inspection (tests);
 * the next step overwrites them. */
qd_status qd_model_act_q8_buffer(qd_model* m, void** buf, size_t* slot_bytes, int* slots);
/* Synchronise `stream` and return QD_ERR_DEVICE_FLAG (and clear the word) if a
 * kernel met an out-of-range token or position since the last check. */
qd_status qd_model_check(qd_model* m, qd_stream_t stream);
/* Number of kernels one decode step launches (for launch accounting). */
int qd_model_launches_per_step(const qd_model* m);

/* How the decode step runs its layers (no counterpart on the pages; the same step either
 * way, parity-tested both ways):
 *  - QD_STEP_KERNEL_CHAIN: a CUDA graph of per-operation kernels over the whole GPU (the
 *    embedding, five kernels per layer, the head GEMV with the argmax).
 *  - QD_STEP_CLUSTER: the embedding and all layers in one kernel, one thread-block
 *    cluster of 8 or 16 CTAs per sequence that keeps each layer's intermediate vectors in
 *    distributed shared memory, then the head GEMV with the argmax over the whole GPU.
 *    Available for Q4_0 / Q8_0 layer weights with the f32 cache and f32 activations, when
 *    the shapes fit its shared memory (per sequence: a weight slice of each product, and
 *    the cached K/V rows of one attention chunk, max_ctx / (cluster size / n_kv_heads)
 *    positions) and the device can schedule the cluster.
 *  - QD_STEP_AUTO (the default): the kernel chain, the faster of the two on GB300 at the
 *    135M shape (0.45 against 0.65-0.69 ms per token: the cluster's 16 SMs are latency-
 *    bound on each layer's products, and a handoff through distributed shared memory costs
 *    about a round trip to L2).
 * qd_model_set_step_path: QD_ERR_UNSUPPORTED when QD_STEP_CLUSTER is asked for and not
 * available, QD_ERR_INVALID_ARG for another value.  qd_model_step_path: the path the
 * next step takes (QD_STEP_KERNEL_CHAIN or QD_STEP_CLUSTER; -1 for a null model).
 * qd_model_cluster_available: 1 when the model can take QD_STEP_CLUSTER, else 0. */
#define QD_STEP_AUTO 0
#define QD_STEP_KERNEL_CHAIN 1
#define QD_STEP_CLUSTER 2
qd_status qd_model_set_step_path(qd_model* m, int path);
int qd_model_step_path(const qd_model* m);
int qd_model_cluster_available(const qd_model* m);

#ifdef __cplusplus
}
#endif
#endif /* QDECODE_H */
