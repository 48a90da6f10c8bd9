// Internal declarations shared by the libqdecode translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/qdecode.h"

namespace qd {

constexpr int kWarp = 32;

// Bits of the device error word.
constexpr uint32_t kErrToken = 1u;     // token id outside [0, vocab)
constexpr uint32_t kErrPosition = 2u;  // position outside [0, max_ctx)
constexpr uint32_t kErrTimeout = 4u;   // a bounded wait inside a kernel gave up

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int64_t align16u(int64_t v) { return (v + 15) & ~(int64_t)15; }

inline qd_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Packed layout of one tensor (see qdecode.h, "Load-time repacking").
//   codes: per row, `row_code_bytes` contiguous bytes (16-byte aligned rows)
//   scales: per row, `row_scale_bytes` contiguous bytes (f16 d per block for
//           Q4_0/Q8_0, 16-byte headers per super-block for Q4_K, one f32 for I8)
// ---------------------------------------------------------------------------
struct PackedView {
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t rows, cols;
  int64_t row_code_bytes, row_scale_bytes;
};

__host__ __device__ inline int64_t row_code_bytes(int fmt, int64_t cols) {
  switch (fmt) {
    case QD_Q4_0:
    case QD_Q4_1:
    case QD_Q5_0:
    case QD_Q4_K: return cols / 2;
    case QD_Q8_0: return cols;
    case QD_Q5_K: return (cols / 256) * 160;  // qh, then low nibbles
    case QD_Q6_K: return (cols / 256) * 192;  // ql, then qh
    case QD_F16: return cols * 2;
    case QD_I4_ROW: return cols / 2;
    default: return cols;  // QD_I8_ROW
  }
}

__host__ __device__ inline int64_t row_scale_bytes(int fmt, int64_t cols) {
  switch (fmt) {
    case QD_Q4_0:
    case QD_Q8_0: return (cols / 32) * 2;
    case QD_Q4_1: return (cols / 32) * 4;    // d, m
    case QD_Q5_0: return (cols / 32) * 6;    // d, qh
    case QD_Q4_K:
    case QD_Q5_K: return (cols / 256) * 16;  // d, dmin, 12 scale bytes
    case QD_Q6_K: return (cols / 256) * 18;  // 16 int8 scales, d
    case QD_F16: return 0;
    default: return 4;
  }
}

inline bool shape_ok(int fmt, int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 1) return false;
  switch (fmt) {
    case QD_Q4_0:
    case QD_Q8_0:
    case QD_Q4_1:
    case QD_Q5_0:
    case QD_F16: return cols % 32 == 0;
    case QD_Q4_K:
    case QD_Q5_K:
    case QD_Q6_K: return cols % 256 == 0;
    case QD_I8_ROW: return cols % 16 == 0;
    case QD_I4_ROW: return cols % 32 == 0;
    default: return false;
  }
}

inline bool fmt_ok(int fmt) { return fmt >= QD_Q4_0 && fmt <= QD_I4_ROW; }
// The formats the decode step's fused kernels take.
inline bool model_fmt_ok(int fmt) { return fmt >= QD_Q4_0 && fmt <= QD_I8_ROW; }

inline size_t packed_code_region(int fmt, int64_t rows, int64_t cols) {
  return align_up((size_t)rows * (size_t)row_code_bytes(fmt, cols), 16);
}

inline size_t packed_bytes(int fmt, int64_t rows, int64_t cols) {
  if (!fmt_ok(fmt) || !shape_ok(fmt, rows, cols)) return 0;
  return packed_code_region(fmt, rows, cols) + align_up((size_t)rows * (size_t)row_scale_bytes(fmt, cols), 16);
}

inline size_t src_bytes(int fmt, int64_t rows, int64_t cols) {
  if (!fmt_ok(fmt) || !shape_ok(fmt, rows, cols)) return 0;
  switch (fmt) {
    case QD_Q4_0: return (size_t)rows * (cols / 32) * 18;
    case QD_Q8_0: return (size_t)rows * (cols / 32) * 34;
    case QD_Q4_K: return (size_t)rows * (cols / 256) * 144;
    case QD_Q4_1: return (size_t)rows * (cols / 32) * 20;
    case QD_Q5_0: return (size_t)rows * (cols / 32) * 22;
    case QD_Q5_K: return (size_t)rows * (cols / 256) * 176;
    case QD_Q6_K: return (size_t)rows * (cols / 256) * 210;
    case QD_F16: return (size_t)rows * cols * 2;
    case QD_I4_ROW: return (size_t)rows * (cols / 2) + 4 * (size_t)rows;
    default: return (size_t)rows * cols + 4 * (size_t)rows;
  }
}

inline PackedView packed_view(int fmt, const void* base, int64_t rows, int64_t cols) {
  PackedView v;
  v.codes = static_cast<const uint8_t*>(base);
  v.scales = v.codes + packed_code_region(fmt, rows, cols);
  v.rows = rows;
  v.cols = cols;
  v.row_code_bytes = row_code_bytes(fmt, cols);
  v.row_scale_bytes = row_scale_bytes(fmt, cols);
  return v;
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)));
}

// Streaming 16-byte load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Byte k of w (as an unsigned 0..255) turned into the float 2^23 + byte:
// the byte lands in the low mantissa bits of 0x4B000000.
__device__ __forceinline__ float byte_as_magic(uint32_t w, int k) {
  return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | (uint32_t)k));
}

constexpr float kMagic = 8388608.0f;  // 2^23

// Q4_K: 6-bit (scale, min) of sub-block j from the 12-byte field q.
__device__ __forceinline__ void q4k_scale_min(int j, const uint8_t* q, int& sc, int& m) {
  if (j < 4) {
    sc = q[j] & 63;
    m = q[j + 4] & 63;
  } else {
    sc = (q[j + 4] & 0x0F) | ((q[j - 4] >> 6) << 4);
    m = (q[j + 4] >> 4) | ((q[j] >> 6) << 4);
  }
}

// One dequantised weight (row r, column c) of a packed tensor, rounded once to
// f32.  Used by the embedding lookup and the test dequantiser; the GEMV kernels
// never materialise weights.
__device__ __forceinline__ float dequant_elem(int fmt, const PackedView& W, int64_t r, int64_t c) {
  const uint8_t* code_row = W.codes + r * W.row_code_bytes;
  const uint8_t* sc_row = W.scales + r * W.row_scale_bytes;
  if (fmt == QD_Q4_0) {
    const int64_t b = c >> 5;
    const int j = (int)(c & 31);
    const uint8_t byte = code_row[b * 16 + (j & 15)];
    const int q = (j < 16) ? (byte & 15) : (byte >> 4);
    const float d = f16_bits_to_f32(sc_row[2 * b] | (sc_row[2 * b + 1] << 8));
    return (float)(q - 8) * d;
  } else if (fmt == QD_Q8_0) {
    const int64_t b = c >> 5;
    const float d = f16_bits_to_f32(sc_row[2 * b] | (sc_row[2 * b + 1] << 8));
    return (float)(int8_t)code_row[c] * d;
  } else if (fmt == QD_Q4_K) {
    const int64_t s = c >> 8;
    const int e = (int)(c & 255);
    const int chunk = e >> 6, hi = (e >> 5) & 1, l = e & 31;
    const uint8_t* hdr = sc_row + s * 16;
    const float d = f16_bits_to_f32(hdr[0] | (hdr[1] << 8));
    const float dmin = f16_bits_to_f32(hdr[2] | (hdr[3] << 8));
    int sc, m;
    q4k_scale_min(2 * chunk + hi, hdr + 4, sc, m);
    const uint8_t byte = code_row[s * 128 + 32 * chunk + l];
    const int q = hi ? (byte >> 4) : (byte & 15);
    // d*sc is exact in f32; the fma rounds d*sc*q - dmin*m once.
    return fmaf(d * (float)sc, (float)q, -(dmin * (float)m));
  } else if (fmt == QD_Q4_1) {
    const int64_t b = c >> 5;
    const int j = (int)(c & 31);
    const uint8_t byte = code_row[b * 16 + (j & 15)];
    const int q = (j < 16) ? (byte & 15) : (byte >> 4);
    const uint8_t* h = sc_row + 4 * b;
    // d*q + m rounded once
    return fmaf(f16_bits_to_f32(h[0] | (h[1] << 8)), (float)q, f16_bits_to_f32(h[2] | (h[3] << 8)));
  } else if (fmt == QD_Q5_0) {
    const int64_t b = c >> 5;
    const int j = (int)(c & 31);
    const uint8_t byte = code_row[b * 16 + (j & 15)];
    const uint8_t* h = sc_row + 6 * b;
    const uint32_t qh = (uint32_t)h[2] | ((uint32_t)h[3] << 8) | ((uint32_t)h[4] << 16) | ((uint32_t)h[5] << 24);
    const int q = ((j < 16) ? (byte & 15) : (byte >> 4)) | (int)(((qh >> j) & 1u) << 4);
    return (float)(q - 16) * f16_bits_to_f32(h[0] | (h[1] << 8));
  } else if (fmt == QD_Q5_K) {
    const int64_t s = c >> 8;
    const int e = (int)(c & 255);
    const int chunk = e >> 6, hi = (e >> 5) & 1, l = e & 31;
    const uint8_t* hdr = sc_row + s * 16;
    const float d = f16_bits_to_f32(hdr[0] | (hdr[1] << 8));
    const float dmin = f16_bits_to_f32(hdr[2] | (hdr[3] << 8));
    int sc, m;
    q4k_scale_min(2 * chunk + hi, hdr + 4, sc, m);
    const uint8_t* blk = code_row + s * 160;
    const uint8_t byte = blk[32 + 32 * chunk + l];
    const int q = (hi ? (byte >> 4) : (byte & 15)) | (((blk[l] >> (2 * chunk + hi)) & 1) << 4);
    return fmaf(d * (float)sc, (float)q, -(dmin * (float)m));
  } else if (fmt == QD_Q6_K) {
    const int64_t s = c >> 8;
    const int e = (int)(c & 255);
    const int h = e >> 7, k = (e >> 5) & 3, l = e & 31;
    const uint8_t* blk = code_row + s * 192;
    const uint8_t lb = blk[64 * h + l + 32 * (k & 1)];
    const int q = ((k < 2) ? (lb & 15) : (lb >> 4)) | (((blk[128 + 32 * h + l] >> (2 * k)) & 3) << 4);
    const uint8_t* hdr = sc_row + s * 18;
    const int sc = (int8_t)hdr[8 * h + 2 * k + (l >> 4)];
    // d*sc*(q-32): at most 11 + 7 + 5 significant bits, exact in f32
    return f16_bits_to_f32(hdr[16] | (hdr[17] << 8)) * (float)sc * (float)(q - 32);
  } else if (fmt == QD_F16) {
    return f16_bits_to_f32(code_row[2 * c] | (code_row[2 * c + 1] << 8));
  } else if (fmt == QD_I4_ROW) {  // packed as Q4_0 codes in offset binary (q + 8)
    const int j = (int)(c & 31);
    const uint8_t byte = code_row[(c >> 5) * 16 + (j & 15)];
    float s;
    memcpy(&s, sc_row, 4);
    return s * (float)(((j < 16) ? (byte & 15) : (byte >> 4)) - 8);
  } else {
    float s;
    memcpy(&s, sc_row, 4);
    return (float)(int8_t)code_row[c] * s;
  }
}

// ---------------------------------------------------------------------------
// Launchers shared between translation units (return QD_OK or QD_ERR_CUDA)
// ---------------------------------------------------------------------------
enum GemvMode { kGemvStore = 0, kGemvAccumulate = 1, kGemvSwiGLU = 2, kGemvQKV = 3, kGemvArgmax = 4 };

// Fused epilogue of the QKV projection (mode kGemvQKV).  The packed QKV matrix holds
// q_rows query rows, k_rows key rows, then the value rows; in the q and k parts, the
// two rows of each RoPE pair are adjacent (pair i of a head at local rows 2i, 2i+1,
// see the repacker).  The epilogue rotates each pair by the angles of pos[b], writes
// q (natural order) to q_out[b*q_stride + ...], and appends k and v to the caches
// [batch][kv_head][max_ctx][head_dim] at pos[b].
struct QkvEpilogue {
  int q_rows = 0, k_rows = 0, head_dim = 64, pairing = QD_ROPE_HALF;
  const int32_t* pos = nullptr;
  const float* rope = nullptr;  // [max_ctx][head_dim/2][2] (cos, sin)
  float* q_out = nullptr;
  int64_t q_stride = 0;
  void* kc = nullptr;  // f32 or binary16 elements (kv_f16)
  void* vc = nullptr;
  int64_t cache_batch_stride = 0;  // elements
  int max_ctx = 0;
  bool kv_f16 = false;
};

// Store one cache element (index i) as f32 or binary16 (round to nearest even).
__device__ __forceinline__ void cache_store(void* base, bool f16, int64_t i, float v) {
  if (f16)
    reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
  else
    reinterpret_cast<float*>(base)[i] = v;
}

// Fused greedy argmax of the output head (mode kGemvArgmax): the logits are stored as
// in kGemvStore, every warp folds its rows into a 64-bit key (ordered value, then
// inverted index) merged with atomicMax into key[b]; the last CTA to finish writes the
// winning index to tok_out[b], advances pos[b] and resets key and counter to zero.
struct ArgmaxEpilogue {
  unsigned long long* key = nullptr;  // [batch], zero between steps
  unsigned int* counter = nullptr;    // zero between steps
  int32_t* tok_out = nullptr;
  int32_t* pos = nullptr;
};

__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);  // order-preserving for non-NaN floats
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t argmax_key_index(unsigned long long k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}

// Programmatic dependent launch: a kernel launched with the PDL attribute may start
// before its predecessor finishes; it must call pdl_wait() before it reads anything
// the predecessor writes or writes anything the predecessor reads.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
qd_status launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                   Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

// y = W x (mode store), y += W x (accumulate), or for rows interleaved as
// (gate_i, up_i) pairs: y[b][i] = silu(gate_i . x) * (up_i . x) (swiglu; y has
// rows/2 columns per batch row).  With norm_g set, x is first replaced by
// x * norm_g / sqrt(mean(x^2) + eps) (RMSNorm fused into the prologue).
struct GemvArgs {
  int fmt = QD_Q4_0;
  PackedView W{};
  const float* x = nullptr;
  float* y = nullptr;
  int batch = 1;
  GemvMode mode = kGemvStore;
  const float* norm_g = nullptr;
  float eps = 0.f;
  uint32_t* err = nullptr;  // device error word (may be null)
  bool pdl = false;         // launch as a programmatic dependent of the previous kernel
  QkvEpilogue qkv{};
  ArgmaxEpilogue am{};
};
qd_status launch_q_gemv(const GemvArgs& a, cudaStream_t stream);
qd_status launch_q_gemv_stream(const GemvArgs& a, cudaStream_t stream);
// Whether launch_q_gemv runs the streaming kernel for these arguments (and so can
// take norm_g and the pdl flag).
bool gemv_streams(const GemvArgs& a);
// Batch 3-16 on the tensor cores (mma.sync, binary16 codes times x split into two binary16
// parts; Q4_0, Q8_0, INT8 rows; every epilogue and the fused RMSNorm; store and accumulate
// over column ranges when x is wider than the shared memory holds).
bool gemv_mma_supported(const GemvArgs& a);
qd_status launch_q_gemv_mma(const GemvArgs& a, cudaStream_t stream);
// Whether launch_q_gemv fuses RMSNorm for these arguments with norm_g = gains.
bool gemv_fuses_norm(const GemvArgs& a, const float* gains);
// Batch 9-16 per-row INT8 on the tensor cores (store, accumulate or SwiGLU; no fused norm).
bool gemv_tc_supported(const GemvArgs& a);
qd_status launch_q_gemv_tc(const GemvArgs& a, cudaStream_t stream);

// Batched prefill product on the tensor cores (Q4_0, Q8_0, INT8 rows; cols % 64 == 0):
// y[n][r] = sum_c deq(W)[r][c] x[n][c] for n < t (kGemmStore), y[n][r] += that
// (kGemmAccumulate), or for rows interleaved as (gate_i, up_i) pairs y[n][i] =
// silu(gate_i . x[n]) * (up_i . x[n]) (kGemmSwiGLU; y has rows / 2 columns); ws holds
// gemm_workspace_bytes(cols, t).
constexpr int kGemmStore = 0, kGemmAccumulate = 1, kGemmSwiGLU = 2;
size_t gemm_workspace_bytes(int64_t cols, int t);
qd_status launch_q_gemm(int fmt, const PackedView& W, const float* x, float* y, int t, void* ws, uint32_t* err,
                        cudaStream_t stream, int mode = kGemmStore);

// ggml-exact activations: Q8_0 (Q8_1 with with_sum) quantisation of x [batch][cols] into
// out (codes, then f16 d, then f16 s; q8_buffer_bytes), and the product over them with the
// store / accumulate / SwiGLU epilogues (Q4_0, Q8_0, Q4_1).
size_t q8_buffer_bytes(int batch, int64_t cols, bool with_sum);
qd_status launch_quantize_q8(const float* x, int batch, int64_t cols, bool with_sum, void* out, cudaStream_t stream);
qd_status launch_q_gemv_q8(int fmt, const PackedView& W, const void* xq, int batch, float* y, int mode,
                           cudaStream_t stream);
// RMSNorm (the same f32 values as launch_rmsnorm) quantised to Q8_0 into out in one kernel.
qd_status launch_rmsnorm_q8(const float* x, const float* g, int n, float eps, int batch, void* out,
                            cudaStream_t stream);

qd_status launch_rmsnorm(const float* x, const float* g, float* out, int n, int batch, float eps,
                         cudaStream_t stream);
qd_status launch_rope(float* v, int n_heads, int head_dim, int64_t batch_stride, const int32_t* pos, int pairing,
                      const float* cos_sin, int max_ctx, int batch, uint32_t* err, cudaStream_t stream);
qd_status launch_kv_append(const float* k, const float* v, int64_t src_stride, float* kc, float* vc, int n_kv,
                           int head_dim, const int32_t* pos, int max_ctx, int batch, int64_t cache_batch_stride,
                           uint32_t* err, cudaStream_t stream);
size_t attn_workspace_bytes(int n_heads, int head_dim, int max_ctx, int batch);
qd_status launch_attention(const float* q, int64_t q_stride, const float* kc, const float* vc,
                           int64_t cache_batch_stride, float* out, int n_heads, int n_kv, int head_dim,
                           const int32_t* pos, int max_ctx, int batch, void* ws, uint32_t* err,
                           cudaStream_t stream);
qd_status launch_swiglu(const float* g, const float* u, float* out, int64_t n, int batch, cudaStream_t stream);
qd_status launch_argmax(const float* logits, int64_t n, int batch, int32_t* out, int32_t* pos_to_advance,
                        cudaStream_t stream);
qd_status launch_embed(int fmt, const PackedView& E, const int32_t* tokens, int batch, float* x, uint32_t* err,
                       cudaStream_t stream);
// Repack source rows [0, n_rows) into packed rows dst_row0 + i*dst_row_step.  With
// pair_hd > 0 the rows are taken in blocks of pair_hd (one head) and, inside a block,
// local row i goes to local row 2*(i % (pair_hd/2)) + i / (pair_hd/2): the two rows of
// each half-pairing RoPE pair (i, i + pair_hd/2) become adjacent.
qd_status launch_repack_rows(int fmt, const void* src, int64_t n_rows, int64_t cols, void* dst_base,
                             int64_t dst_rows, int64_t dst_row0, int64_t dst_row_step, cudaStream_t stream,
                             int pair_hd = 0);
// Standalone form of the kGemvQKV epilogue for the register-path GEMV: reads the
// packed-order projection qkv[b][rows] and does the rotation, q write and cache append.
qd_status launch_qkv_post(const float* qkv, int64_t qkv_stride, int batch, const QkvEpilogue& e, uint32_t* err,
                          cudaStream_t stream, bool pdl);
// Decode-step attention, one thread-block cluster per (sequence, kv head).  Cluster
// size and SM count used by its launcher.
int attn_cluster_size(int n_kv, int batch, int max_ctx);
int attn_sm_count();
qd_status launch_attention_cluster(const float* q, int64_t q_stride, const float* kc, const float* vc,
                                   int64_t cache_batch_stride, float* out, int n_heads, int n_kv, int head_dim,
                                   const int32_t* pos, int max_ctx, int batch, uint32_t* err, cudaStream_t stream,
                                   bool pdl);
// Decode-step attention for long walks: an even split of all pairs' positions over one
// CTA per SM (attn_flat_ctas), partials merged by the last CTA of each (sequence, kv
// head).  `ws` holds attn_flat_ws_floats(..., ctas) floats for the same `ctas`; `cnt`
// (batch * n_kv unsigned ints) must be zero and is left zero.  kc, vc hold f32 or
// (kv_f16) binary16 elements.  The decode step takes it when attn_use_flat says so (the f32
// cache of all pairs at full context holds at least kAttnFlatMinBytes) and always for a
// binary16 cache.
constexpr int64_t kAttnFlatMinBytes = 8ll << 20;
bool attn_use_flat(int n_kv, int batch, int max_ctx);
int attn_flat_ctas();
size_t attn_flat_ws_floats(int n_heads, int n_kv, int batch, int ctas);
qd_status launch_attention_flat(const float* q, int64_t q_stride, const void* kc, const void* vc, bool kv_f16,
                                int64_t cache_batch_stride, float* out, int n_heads, int n_kv, int head_dim,
                                const int32_t* pos, int max_ctx, int batch, int ctas, float* ws, unsigned int* cnt,
                                uint32_t* err, cudaStream_t stream, bool pdl);

// The decode step's layers (embedding to the last residual add) as one thread-block
// cluster per sequence (qd_step_cluster.cu).  What it needs from the model: formats,
// shapes, the weight layout (a uniform stride between layers, offsets inside a layer) and
// the cache.
struct StepClusterModel {
  int fmt = QD_Q4_0, emb_fmt = QD_Q8_0;
  PackedView emb{};
  const uint8_t* w = nullptr;
  int64_t layer0 = 0, layer_stride = 0;  // bytes
  int64_t off_attn_norm = 0, off_ffn_norm = 0, off_qkv = 0, off_wo = 0, off_gu = 0, off_wd = 0;  // in a layer
  int layers = 0, D = 0, F = 0, n_heads = 0, n_kv = 0, max_ctx = 0, pairing = QD_ROPE_HALF, vocab = 0;
  float eps = 0.f;
  float* kc = nullptr;  // f32 caches [layer][batch][kv_head][max_ctx][64]
  float* vc = nullptr;
  int64_t cache_layer_stride = 0, cache_batch_stride = 0;  // elements
  const float* rope = nullptr;
};
struct StepClusterPlan {
  int C = 0, S = 0, kvp = 0, nmax = 0;
  uint32_t wbuf_bytes = 0, smem = 0;
  uint32_t off_wbuf = 0, off_kv = 0, off_slot = 0, off_x = 0, off_v = 0, off_rec = 0, off_sc = 0, off_misc = 0,
           off_bar = 0;
};
// False when the model's shapes, formats or cache do not fit the kernel (shared memory,
// cluster scheduling on this device).
bool step_cluster_plan(const StepClusterModel& m, StepClusterPlan* plan);
// Embedding and every layer for `batch` sequences (tokens tok[b] at positions pos[b]); the
// residual stream after the last layer goes to x_out [batch][D].
qd_status launch_step_cluster(const StepClusterModel& m, const StepClusterPlan& plan, const int32_t* tok,
                              const int32_t* pos, float* x_out, uint32_t* err, int batch, cudaStream_t stream);

}  // namespace qd
