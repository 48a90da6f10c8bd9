// Load-time per-row INT8 quantisation of BF16 weights (minillm-cpp README, "Direct INT8
// loading": each weight matrix is quantised row by row straight from the BF16 checkpoint,
// never widened to f32 as a whole; "Quantization": symmetric, one scale per output row;
// "Loader": BF16 -> f32 is the zero-extension of the bit pattern).
//
// Row r: s_r = max_c |w_rc| / 127 (f32), q_rc = w_rc / s_r rounded to nearest with ties
// away from zero (roundf), clamped to [-127, 127].  A row of zeros gets s_r = 0 and codes
// 0; a row holding a non-finite value gets codes 0 and a NaN scale.  The output is the
// per-row INT8 source layout (codes [rows][cols], then f32 scales [rows]), which
// qd_repack and the model loader take as it is.
//
// One warp per row: a max pass over 16-byte chunks (8 values) of the row, then a second
// pass over the same chunks (now in L1) that writes 8 codes per lane and chunk; codes are
// computed from a reciprocal multiply, with the division kept for near-ties (code_byte).  HBM
// traffic: 2 bytes read and 1 byte written per weight, 4 bytes per row.
//
// Per-row INT4 ("Quantization" names symmetric per-channel INT8 and INT4 with one scale per
// output row): the same rule with the 4-bit range, s_r = max |w| / 7, codes clamped to
// [-7, 7], written as the INT4 source layout (two's-complement nibbles, element 2i in the
// low nibble of byte i, then f32 scales [rows]).
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kQuantWarps = 8;  // rows per CTA

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The code of value v in a row with scale s: roundf of the correctly rounded quotient
// v / s, clamped to [-127, 127].  t = v * rs (rs = 1/s, correctly rounded) is within
// 3 * 127 * 2^-24 < 3e-5 of that quotient (|v / s| <= 127 up to rounding), so wherever t is
// further than that from a half-way point both round to the same integer, and there
// truncating t + copysign(0.5, t) rounds it (the addition's own error, at most 2^-18, cannot
// reach an integer); the rare values closer to a half-way point (about 1 in 16,000) take
// the division itself.  The bound needs a normal s (1/s finite, both roundings relative):
// a row whose scale is subnormal (max |w| < 127 * 2^-126) always divides (fast == false).
// For a normal s the result is within [-127, 127] without a clamp.
__device__ __forceinline__ uint32_t code_byte(float v, float s, float rs, bool fast) {
  const float t = v * rs;
  const float a = fabsf(t);
  int q;
  if (!fast || fabsf(a - truncf(a) - 0.5f) < 3e-5f)
    q = (int)fminf(fmaxf(roundf(v / s), -127.f), 127.f);
  else
    q = __float2int_rz(t + copysignf(0.5f, t));
  return (uint32_t)q & 0xFFu;
}

__global__ void __launch_bounds__(kQuantWarps * 32)
    k_quantize_i8_rows(const uint16_t* __restrict__ w, int64_t rows, int64_t cols, uint8_t* __restrict__ codes,
                       float* __restrict__ scales) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kQuantWarps + warp;
  if (r >= rows) return;
  const uint4* src = reinterpret_cast<const uint4*>(w + r * cols);
  const int64_t n8 = cols / 8;  // chunks of 8 values (cols % 16 == 0)
  // max |w| as bf16 magnitude bits (sign cleared): for non-negative floats the bit
  // patterns order as the values, and NaN and infinity (>= 0x7F80) above every finite one
  uint32_t mb = 0u;
  for (int64_t i = lane; i < n8; i += 32) {
    const uint4 v = __ldg(src + i);
    mb = __vmaxu2(mb, v.x & 0x7FFF7FFFu);
    mb = __vmaxu2(mb, v.y & 0x7FFF7FFFu);
    mb = __vmaxu2(mb, v.z & 0x7FFF7FFFu);
    mb = __vmaxu2(mb, v.w & 0x7FFF7FFFu);
  }
  uint32_t m16 = max(mb & 0xFFFFu, mb >> 16);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m16 = max(m16, __shfl_xor_sync(0xffffffffu, m16, off));
  const bool finite = m16 < 0x7F80u;
  const float m = __uint_as_float(m16 << 16);
  const bool zero = !finite || m16 == 0u;
  const float s = m / 127.f;
  const bool fast = s >= 1.17549435e-38f;  // normal
  const float rs = fast ? 1.f / s : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(codes + r * cols);
  for (int64_t i = lane; i < n8; i += 32) {
    uint2 out = make_uint2(0u, 0u);
    if (!zero) {
      const uint4 v = __ldg(src + i);
      out.x = code_byte(bf16_lo(v.x), s, rs, fast) | code_byte(bf16_hi(v.x), s, rs, fast) << 8 |
              code_byte(bf16_lo(v.y), s, rs, fast) << 16 | code_byte(bf16_hi(v.y), s, rs, fast) << 24;
      out.y = code_byte(bf16_lo(v.z), s, rs, fast) | code_byte(bf16_hi(v.z), s, rs, fast) << 8 |
              code_byte(bf16_lo(v.w), s, rs, fast) << 16 | code_byte(bf16_hi(v.w), s, rs, fast) << 24;
    }
    dst[i] = out;
  }
  if (lane == 0) scales[r] = !finite ? __uint_as_float(0x7FC00000u) : (m16 == 0u ? 0.f : s);
}

// Per-row INT4 (the same rule with the 4-bit code range: s = max|w| / 7, codes w / s
// rounded to nearest with ties away from zero, clamped to +-7): one warp per row; the codes
// are two's-complement nibbles, element 2i in the low nibble of byte i.  The quotients are
// IEEE round-to-nearest divisions, as the rule takes its decision in f32.
__global__ void __launch_bounds__(kQuantWarps * 32) k_quantize_i4_rows(const uint16_t* __restrict__ w, int64_t rows,
                                                                       int64_t cols, uint8_t* __restrict__ codes,
                                                                       float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint16_t* wr = w + r * cols;
  uint32_t mbits = 0;  // largest |w| as bf16 magnitude bits (monotonic for finite values)
  bool finite = true;
  for (int64_t c = lane; c < cols; c += 32) {
    const uint32_t a = wr[c] & 0x7FFFu;
    finite = finite && a < 0x7F80u;
    mbits = max(mbits, a);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mbits = max(mbits, __shfl_xor_sync(0xffffffffu, mbits, off));
  finite = __all_sync(0xffffffffu, finite);
  uint8_t* qr = codes + r * (cols / 2);
  const float m = __uint_as_float(mbits << 16);
  if (!finite || m == 0.f) {
    for (int64_t c = lane; c < cols / 2; c += 32) qr[c] = 0;
    if (lane == 0) scales[r] = finite ? 0.f : __uint_as_float(0x7FC00000u);
    return;
  }
  const float sc = __fdiv_rn(m, 7.0f);
  for (int64_t c = lane; c < cols / 2; c += 32) {
    int q[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float v = __uint_as_float((uint32_t)wr[2 * c + k] << 16);
      q[k] = (int)fminf(fmaxf(roundf(__fdiv_rn(v, sc)), -7.0f), 7.0f);
    }
    qr[c] = (uint8_t)((q[0] & 0x0F) | ((q[1] & 0x0F) << 4));
  }
  if (lane == 0) scales[r] = sc;
}

}  // namespace
}  // namespace qd

using namespace qd;

extern "C" qd_status qd_quantize_i4_rows(const uint16_t* w_bf16, int64_t rows, int64_t cols, void* out,
                                         size_t out_bytes, qd_stream_t stream) {
  if (!w_bf16 || !out) return QD_ERR_INVALID_ARG;
  if (!shape_ok(QD_I4_ROW, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(out)) return QD_ERR_ALIGN;
  if (out_bytes < src_bytes(QD_I4_ROW, rows, cols)) return QD_ERR_NOMEM;
  uint8_t* codes = static_cast<uint8_t*>(out);
  float* scales = reinterpret_cast<float*>(codes + rows * (cols / 2));
  const int64_t grid = (rows + kQuantWarps - 1) / kQuantWarps;
  if (grid > 0x7FFFFFFF) return QD_ERR_SHAPE;
  k_quantize_i4_rows<<<(unsigned)grid, kQuantWarps * 32, 0, (cudaStream_t)stream>>>(w_bf16, rows, cols, codes,
                                                                                    scales);
  return launch_status();
}

extern "C" qd_status qd_quantize_i8_rows(const uint16_t* w_bf16, int64_t rows, int64_t cols, void* out,
                                         size_t out_bytes, qd_stream_t stream) {
  if (!w_bf16 || !out) return QD_ERR_INVALID_ARG;
  if (!shape_ok(QD_I8_ROW, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(w_bf16) || !aligned16(out)) return QD_ERR_ALIGN;
  if (out_bytes < src_bytes(QD_I8_ROW, rows, cols)) return QD_ERR_NOMEM;
  uint8_t* codes = static_cast<uint8_t*>(out);
  float* scales = reinterpret_cast<float*>(codes + rows * cols);
  const int64_t grid = (rows + kQuantWarps - 1) / kQuantWarps;
  if (grid > 0x7FFFFFFF) return QD_ERR_SHAPE;
  k_quantize_i8_rows<<<(unsigned)grid, kQuantWarps * 32, 0, (cudaStream_t)stream>>>(w_bf16, rows, cols, codes,
                                                                                    scales);
  return launch_status();
}
