// ggml-exact activations (go-llm type CPU, "ExactGGML": activations are quantised to Q8_0,
// Q8_1 for Q4_1 weights, before every quantised matrix product) and the product over them
// in the blocks' own integers (llamini, "Optimizing for CPU, and finding out what was
// actually true": ggml multiplies the packed bytes and converts to float only for the
// scaled sum).
//
// Quantisation, per 32 values of a row of x: d = max|x| / 127, q = x / d rounded to nearest
// with ties away from zero, clamped to +-127 (both divisions IEEE round-to-nearest in f32);
// the block keeps d as binary16 and, for Q8_1, s = d * sum q as binary16.  A zero block
// has d = 0 and codes 0; a block holding a non-finite value codes 0 and d = s = NaN.
//
// Product: per weight block, an integer dot of its codes with the block's activation codes
// (dp4a over eight 4-byte words), then y += d_w d_x sum (Q4_0: sum (q_w - 8) q_x, taken as
// sum q_w q_x - 8 sum q_x; Q4_1: plus m_w s_x), in f32.
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kQ8Warps = 8;

// One block of 32 values (lane = value, whole warp): codes, d and s (s may be null).
__device__ __forceinline__ void quantize_block(float v, int lane, int8_t* q, __half* d, __half* s) {
  const bool bad = __any_sync(0xffffffffu, !isfinite(v));
  float m = fabsf(v);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (bad || m == 0.f) {
    q[lane] = 0;
    if (lane == 0) {
      const __half z = bad ? __float2half_rn(__int_as_float(0x7FC00000)) : __float2half_rn(0.f);
      *d = z;
      if (s) *s = z;
    }
    return;
  }
  const float dd = __fdiv_rn(m, 127.0f);
  float t = roundf(__fdiv_rn(v, dd));
  t = fminf(fmaxf(t, -127.0f), 127.0f);
  const int qi = (int)t;
  q[lane] = (int8_t)qi;
  int sum = qi;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane == 0) {
    *d = __float2half_rn(dd);
    if (s) *s = __float2half_rn(__fmul_rn(dd, (float)sum));
  }
}

// One warp per block of 32 values.
__global__ void __launch_bounds__(kQ8Warps * 32) k_quantize_q8(const float* __restrict__ x, int64_t blocks,
                                                                int8_t* __restrict__ q, __half* __restrict__ d,
                                                                __half* __restrict__ s) {
  const int lane = threadIdx.x & 31;
  const int64_t b = (int64_t)blockIdx.x * kQ8Warps + (threadIdx.x >> 5);
  if (b >= blocks) return;
  quantize_block(__ldg(x + 32 * b + lane), lane, q + 32 * b, d + b, s ? s + b : nullptr);
}

// RMSNorm of one row (one CTA per row, the same reduction and products as the RMSNorm
// kernel, so the normalised values are the same f32 numbers) quantised to Q8_0 as it is
// formed: out[b][i] = x[b][i] * g[i] / sqrt(mean(x^2) + eps), never stored as f32.
__global__ void __launch_bounds__(512) k_rmsnorm_q8(const float* __restrict__ x, const float* __restrict__ g, int n,
                                                    float eps, int8_t* __restrict__ q, __half* __restrict__ d) {
  __shared__ float red[32];
  const float* xr = x + (int64_t)blockIdx.x * n;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = 1.0f / sqrtf(v / (float)n + eps);
  }
  __syncthreads();
  const float scale = red[0];
  const int lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int64_t row_blocks = n / 32, b0 = (int64_t)blockIdx.x * row_blocks;
  for (int64_t k = threadIdx.x >> 5; k < row_blocks; k += nw) {
    const int i = (int)(32 * k) + lane;
    quantize_block(xr[i] * scale * g[i], lane, q + 32 * (b0 + k), d + b0 + k, nullptr);
  }
}

struct Q8View {
  const int8_t* q;      // [batch][cols]
  const __half* d;      // [batch][cols / 32]
  const __half* s;      // [batch][cols / 32] or null
};

__device__ __forceinline__ int dot_words(const uint32_t (&w)[8], const uint32_t (&x)[8]) {
  int acc = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) acc = __dp4a((int)w[k], (int)x[k], acc);
  return acc;
}

template <int FMT, int R, int NB>
__global__ void __launch_bounds__(256) k_gemv_q8(PackedView W, Q8View X, float* __restrict__ y, int batch, int mode) {
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * R;
  if (row0 >= W.rows) return;
  const int64_t nb = W.cols / 32;
  float acc[R][NB];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;
  for (int64_t k = lane; k < nb; k += 32) {
    uint32_t wq[R][8];
    float dw[R], mw[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int64_t r = row0 + i < W.rows ? row0 + i : row0;
      const uint8_t* cr = W.codes + r * W.row_code_bytes;
      const uint8_t* sr = W.scales + r * W.row_scale_bytes;
      if constexpr (FMT == QD_Q8_0) {
        const uint4 a = ld_stream_v4(cr + 32 * k), c = ld_stream_v4(cr + 32 * k + 16);
        wq[i][0] = a.x; wq[i][1] = a.y; wq[i][2] = a.z; wq[i][3] = a.w;
        wq[i][4] = c.x; wq[i][5] = c.y; wq[i][6] = c.z; wq[i][7] = c.w;
        dw[i] = f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(sr) + k));
        mw[i] = 0.f;
      } else {
        // nibble codes: element j of the block is the low nibble of byte j, element j + 16
        // its high nibble, so word t's low nibbles meet x word t and its high nibbles x word 4 + t
        const uint4 a = ld_stream_v4(cr + 16 * k);
        const uint32_t qw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          wq[i][t] = qw[t] & 0x0F0F0F0Fu;
          wq[i][4 + t] = (qw[t] >> 4) & 0x0F0F0F0Fu;
        }
        if constexpr (FMT == QD_Q4_0) {
          dw[i] = f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(sr) + k));
          mw[i] = 0.f;
        } else {  // Q4_1: (d, m)
          const uint32_t dm = __ldg(reinterpret_cast<const uint32_t*>(sr) + k);
          dw[i] = f16_bits_to_f32(dm & 0xFFFFu);
          mw[i] = f16_bits_to_f32(dm >> 16);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < batch) {
        const int8_t* xq = X.q + (int64_t)b * W.cols + 32 * k;
        const uint4 xa = __ldg(reinterpret_cast<const uint4*>(xq)), xb = __ldg(reinterpret_cast<const uint4*>(xq + 16));
        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
        const float dx = __half2float(X.d[(int64_t)b * nb + k]);
        int xsum = 0;
        if constexpr (FMT == QD_Q4_0) {
#pragma unroll
          for (int t = 0; t < 8; ++t) xsum = __dp4a((int)xw[t], 0x01010101, xsum);
        }
        const float sx = FMT == QD_Q4_1 ? __half2float(X.s[(int64_t)b * nb + k]) : 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const int sumi = dot_words(wq[i], xw) - (FMT == QD_Q4_0 ? 8 * xsum : 0);
          float v = dw[i] * dx * (float)sumi;
          if constexpr (FMT == QD_Q4_1) v = fmaf(mw[i], sx, v);
          acc[i][b] += v;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[i][b] = warp_sum(acc[i][b]);
  if (lane != 0) return;
  if (mode == kGemvSwiGLU) {  // rows (row0, row0 + 1) are (gate_i, up_i), i = row0 / 2
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b < batch) {
        const float g = acc[0][b];
        y[(int64_t)b * (W.rows / 2) + row0 / 2] = g / (1.0f + expf(-g)) * acc[R - 1][b];
      }
    return;
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (row0 + i >= W.rows) break;
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b < batch) {
        float* dst = y + (int64_t)b * W.rows + row0 + i;
        if (mode == kGemvAccumulate)
          *dst += acc[i][b];
        else
          *dst = acc[i][b];
      }
  }
}

template <int FMT, int R, int NB>
qd_status launch_q8_t(const PackedView& W, const Q8View& X, float* y, int batch, int mode, cudaStream_t stream) {
  const int64_t warps = (W.rows + R - 1) / R;
  k_gemv_q8<FMT, R, NB><<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(W, X, y, batch, mode);
  return launch_status();
}

// The SwiGLU epilogue needs each (gate, up) row pair in one warp: R = 2.
template <int FMT>
qd_status launch_q8_fmt(const PackedView& W, const Q8View& X, float* y, int batch, int mode, cudaStream_t stream) {
  const bool pair = mode == kGemvSwiGLU;
  if (batch <= 1) return launch_q8_t<FMT, 2, 1>(W, X, y, batch, mode, stream);
  if (batch <= 4) return launch_q8_t<FMT, 2, 4>(W, X, y, batch, mode, stream);
  if (batch <= 8) return pair ? launch_q8_t<FMT, 2, 8>(W, X, y, batch, mode, stream)
                              : launch_q8_t<FMT, 1, 8>(W, X, y, batch, mode, stream);
  return pair ? launch_q8_t<FMT, 2, 16>(W, X, y, batch, mode, stream)
              : launch_q8_t<FMT, 1, 16>(W, X, y, batch, mode, stream);
}

// Layout of a quantised activation buffer: codes [batch][cols], then f16 d [batch][cols/32],
// then (Q8_1) f16 s [batch][cols/32]; each region 16-byte aligned.
size_t q8_d_offset(int batch, int64_t cols) { return align_up((size_t)batch * (size_t)cols, 16); }
size_t q8_s_offset(int batch, int64_t cols) {
  return q8_d_offset(batch, cols) + align_up((size_t)batch * (size_t)(cols / 32) * 2, 16);
}
size_t q8_bytes(int batch, int64_t cols, bool with_sum) {
  return with_sum ? q8_s_offset(batch, cols) + align_up((size_t)batch * (size_t)(cols / 32) * 2, 16)
                  : q8_s_offset(batch, cols);
}

bool q8_shape_ok(int batch, int64_t cols) { return batch >= 1 && batch <= QD_MAX_BATCH && cols >= 32 && cols % 32 == 0; }

Q8View q8_view(const void* xq, int batch, int64_t cols, bool with_sum) {
  const uint8_t* base = static_cast<const uint8_t*>(xq);
  Q8View X;
  X.q = reinterpret_cast<const int8_t*>(base);
  X.d = reinterpret_cast<const __half*>(base + q8_d_offset(batch, cols));
  X.s = with_sum ? reinterpret_cast<const __half*>(base + q8_s_offset(batch, cols)) : nullptr;
  return X;
}

}  // namespace

size_t q8_buffer_bytes(int batch, int64_t cols, bool with_sum) { return q8_bytes(batch, cols, with_sum); }

qd_status launch_quantize_q8(const float* x, int batch, int64_t cols, bool with_sum, void* out, cudaStream_t stream) {
  uint8_t* base = static_cast<uint8_t*>(out);
  const int64_t blocks = (int64_t)batch * (cols / 32);
  k_quantize_q8<<<(unsigned)((blocks + kQ8Warps - 1) / kQ8Warps), kQ8Warps * 32, 0, stream>>>(
      x, blocks, reinterpret_cast<int8_t*>(base), reinterpret_cast<__half*>(base + q8_d_offset(batch, cols)),
      with_sum ? reinterpret_cast<__half*>(base + q8_s_offset(batch, cols)) : nullptr);
  return launch_status();
}

qd_status launch_rmsnorm_q8(const float* x, const float* g, int n, float eps, int batch, void* out,
                            cudaStream_t stream) {
  uint8_t* base = static_cast<uint8_t*>(out);
  const int threads = n >= 2048 ? 512 : 256;  // as the RMSNorm kernel: the same sums
  k_rmsnorm_q8<<<batch, threads, 0, stream>>>(x, g, n, eps, reinterpret_cast<int8_t*>(base),
                                              reinterpret_cast<__half*>(base + q8_d_offset(batch, n)));
  return launch_status();
}

qd_status launch_q_gemv_q8(int fmt, const PackedView& W, const void* xq, int batch, float* y, int mode,
                           cudaStream_t stream) {
  const Q8View X = q8_view(xq, batch, W.cols, fmt == QD_Q4_1);
  switch (fmt) {
    case QD_Q4_0: return launch_q8_fmt<QD_Q4_0>(W, X, y, batch, mode, stream);
    case QD_Q8_0: return launch_q8_fmt<QD_Q8_0>(W, X, y, batch, mode, stream);
    case QD_Q4_1: return launch_q8_fmt<QD_Q4_1>(W, X, y, batch, mode, stream);
    default: return QD_ERR_UNSUPPORTED;
  }
}

}  // namespace qd

using namespace qd;

extern "C" {

size_t qd_q8_bytes(int batch, int64_t cols, int with_sum) {
  if (!q8_shape_ok(batch, cols) || (with_sum != 0 && with_sum != 1)) return 0;
  return q8_bytes(batch, cols, with_sum != 0);
}

qd_status qd_quantize_q8(const float* x, int batch, int64_t cols, int with_sum, void* out, size_t out_bytes,
                         qd_stream_t stream) {
  if (!x || !out || (with_sum != 0 && with_sum != 1)) return QD_ERR_INVALID_ARG;
  if (!q8_shape_ok(batch, cols)) return QD_ERR_SHAPE;
  if (!aligned16(x) || !aligned16(out)) return QD_ERR_ALIGN;
  if (out_bytes < q8_bytes(batch, cols, with_sum != 0)) return QD_ERR_NOMEM;
  return launch_quantize_q8(x, batch, cols, with_sum != 0, out, (cudaStream_t)stream);
}

qd_status qd_q_gemv_q8(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const void* xq, size_t xq_bytes,
                       float* y, int batch, qd_stream_t stream) {
  if (fmt != QD_Q4_0 && fmt != QD_Q8_0 && fmt != QD_Q4_1) return QD_ERR_UNSUPPORTED;
  if (!W || !xq || !y) return QD_ERR_INVALID_ARG;
  if (!q8_shape_ok(batch, cols) || !shape_ok(fmt, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(y)) return QD_ERR_ALIGN;
  if (xq_bytes < q8_bytes(batch, cols, fmt == QD_Q4_1)) return QD_ERR_NOMEM;  // Q4_1 takes Q8_1 activations
  return launch_q_gemv_q8(fmt, packed_view(fmt, W, rows, cols), xq, batch, y, kGemvStore, (cudaStream_t)stream);
}

}  // extern "C"
