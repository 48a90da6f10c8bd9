// Fused dequantise-and-dot GEMV over packed block-quantised weights.
//
// y[b][r] = sum_c deq(W)[r][c] * x[b][c]   (llmoxide blog, s1 "A neuron is a dot
// product" and s10's Q8_0 row dot; dasLLAMA 8.7.1.4 matmul).  As in the
// minillm-cpp README ("NEON kernels"), the weights are decoded in registers and
// never written out as f32.
//
// Work decomposition.  A warp owns R consecutive output rows.  Its lanes walk the
// row's "units" (32 weights for Q4_0/Q8_0/Q4_K, 16 for INT8) with stride 32, so a
// warp load instruction reads 32 consecutive units of one row: 512 contiguous
// bytes of Q4_0 codes, 1 KB of Q8_0 codes.  The codes of the next unit are loaded
// before the current one is computed.  For each unit the lane turns the codes
// into exact small-integer floats once per row (the byte lands in the mantissa of
// 2^23 and 2^23 is subtracted), then streams x once per batch column and applies
// the unit's scale to the unit's partial sum.  Block scales therefore multiply a
// 32-term partial sum rather than every weight; the per-row f32 sums are reduced
// across the warp with shuffles at the end.  (Per-row INT4 takes the same path with
// 32-weight units; Q4_1, Q5_0, Q5_K, Q6_K and F16 units are decoded to f32 values by
// k_gemv_deq.)
#include "qd_internal.cuh"

namespace qd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerCta = kThreads / kWarp;

template <int FMT>
struct Unit;  // raw codes + scale data of one unit of one row

// ----------------------------------------------------------------- Q4_0
template <>
struct Unit<QD_Q4_0> {
  static constexpr int kWeights = 32;
  uint4 q;
  uint32_t d;
  __device__ __forceinline__ void load(const PackedView& W, int64_t r, int64_t u) {
    q = ld_stream_v4(W.codes + r * W.row_code_bytes + u * 16);
    d = __ldg(reinterpret_cast<const unsigned short*>(W.scales + r * W.row_scale_bytes) + u);
  }
  // w[j] = q_j - 8 for element j of the block (exact).
  __device__ __forceinline__ void codes(float (&w)[32]) const {
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t lo = words[t] & 0x0F0F0F0Fu, hi = (words[t] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[4 * t + k] = byte_as_magic(lo, k) - (kMagic + 8.0f);
        w[16 + 4 * t + k] = byte_as_magic(hi, k) - (kMagic + 8.0f);
      }
    }
  }
  __device__ __forceinline__ float scale() const { return f16_bits_to_f32(d); }
  __device__ __forceinline__ static int64_t x_offset(int64_t u) { return u * 32; }
};

// ----------------------------------------------------------------- Q8_0
template <>
struct Unit<QD_Q8_0> {
  static constexpr int kWeights = 32;
  uint4 q0, q1;
  uint32_t d;
  __device__ __forceinline__ void load(const PackedView& W, int64_t r, int64_t u) {
    const uint8_t* p = W.codes + r * W.row_code_bytes + u * 32;
    q0 = ld_stream_v4(p);
    q1 = ld_stream_v4(p + 16);
    d = __ldg(reinterpret_cast<const unsigned short*>(W.scales + r * W.row_scale_bytes) + u);
  }
  __device__ __forceinline__ void codes(float (&w)[32]) const {
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t b = words[t] ^ 0x80808080u;  // int8 q -> unsigned q + 128
#pragma unroll
      for (int k = 0; k < 4; ++k) w[4 * t + k] = byte_as_magic(b, k) - (kMagic + 128.0f);
    }
  }
  __device__ __forceinline__ float scale() const { return f16_bits_to_f32(d); }
  __device__ __forceinline__ static int64_t x_offset(int64_t u) { return u * 32; }
};

// ----------------------------------------------------------------- INT8 rows
template <>
struct Unit<QD_I8_ROW> {
  static constexpr int kWeights = 16;
  uint4 q;
  __device__ __forceinline__ void load(const PackedView& W, int64_t r, int64_t u) {
    q = ld_stream_v4(W.codes + r * W.row_code_bytes + u * 16);
  }
  __device__ __forceinline__ void codes(float (&w)[16]) const {
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t b = words[t] ^ 0x80808080u;
#pragma unroll
      for (int k = 0; k < 4; ++k) w[4 * t + k] = byte_as_magic(b, k) - (kMagic + 128.0f);
    }
  }
  __device__ __forceinline__ static int64_t x_offset(int64_t u) { return u * 16; }
};

// ----------------------------------------------------------------- INT4 rows
template <>
struct Unit<QD_I4_ROW> {
  static constexpr int kWeights = 32;
  uint4 q;
  __device__ __forceinline__ void load(const PackedView& W, int64_t r, int64_t u) {
    q = ld_stream_v4(W.codes + r * W.row_code_bytes + u * 16);
  }
  // Packed as Q4_0 codes in offset binary: element j of the unit is the low nibble of
  // code byte j, element j + 16 its high nibble, each q + 8 (exact through the magic number).
  __device__ __forceinline__ void codes(float (&w)[32]) const {
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t lo = words[t] & 0x0F0F0F0Fu, hi = (words[t] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[4 * t + k] = byte_as_magic(lo, k) - (kMagic + 8.0f);
        w[16 + 4 * t + k] = byte_as_magic(hi, k) - (kMagic + 8.0f);
      }
    }
  }
  __device__ __forceinline__ static int64_t x_offset(int64_t u) { return u * 32; }
};

template <int N>
__device__ __forceinline__ float dot_x(const float (&w)[N], const float* __restrict__ xp) {
  const float4* x4 = reinterpret_cast<const float4*>(xp);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int t = 0; t < N / 4; ++t) {
    const float4 v = __ldg(x4 + t);
    s0 = fmaf(w[4 * t + 0], v.x, s0);
    s1 = fmaf(w[4 * t + 1], v.y, s1);
    s0 = fmaf(w[4 * t + 2], v.z, s0);
    s1 = fmaf(w[4 * t + 3], v.w, s1);
  }
  return s0 + s1;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// Epilogue shared by every format: reduce each (row, batch) sum across the warp
// and write it according to `mode`.
template <int R, int NB>
__device__ __forceinline__ void finish_rows(float (&acc)[R][NB], const float* row_scale, int64_t row0,
                                            int64_t rows, float* __restrict__ y, int batch, int mode, int lane) {
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[i][b] = warp_sum(acc[i][b]);
  if (lane != 0) return;
  if (mode == kGemvSwiGLU) {
    // rows (row0, row0+1) are (gate_i, up_i) with i = row0 / 2
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b < batch) {
        const float g = acc[0][b] * row_scale[0];
        const float u = acc[R - 1][b] * row_scale[R - 1];
        y[(int64_t)b * (rows / 2) + row0 / 2] = silu(g) * u;
      }
    return;
  }
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int64_t r = row0 + i;
    if (r >= rows) break;
#pragma unroll
    for (int b = 0; b < NB; ++b)
      if (b < batch) {
        const float v = acc[i][b] * row_scale[i];
        float* dst = y + (int64_t)b * rows + r;
        if (mode == kGemvAccumulate)
          *dst += v;
        else
          *dst = v;
      }
  }
}

// Q4_0 / Q8_0 / INT8: one scale per block (or per row) times an integer-code dot.
template <int FMT, int R, int NB>
__global__ void __launch_bounds__(kThreads) k_gemv_blocks(PackedView W, const float* __restrict__ x,
                                                           float* __restrict__ y, int batch, int mode) {
  using U = Unit<FMT>;
  constexpr int KW = U::kWeights;
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * R;
  if (row0 >= W.rows) return;
  const int64_t units = W.cols / KW;
  float acc[R][NB];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;

  U cur[R], nxt[R];
  int64_t u = lane;
  if (u < units) {
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i].load(W, row0 + i < W.rows ? row0 + i : row0, u);
  }
  for (; u < units; u += 32) {
    const int64_t un = u + 32;
    if (un < units) {
#pragma unroll
      for (int i = 0; i < R; ++i) nxt[i].load(W, row0 + i < W.rows ? row0 + i : row0, un);
    }
    float w[R][KW];
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i].codes(w[i]);
    const int64_t xo = U::x_offset(u);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < batch) {
        const float* xp = x + (int64_t)b * W.cols + xo;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float s = dot_x<KW>(w[i], xp);
          if constexpr (FMT == QD_I8_ROW || FMT == QD_I4_ROW)  // one scale per row, applied at the end
            acc[i][b] += s;
          else
            acc[i][b] = fmaf(cur[i].scale(), s, acc[i][b]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i] = nxt[i];
  }
  float row_scale[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    row_scale[i] = 1.0f;
    if constexpr (FMT == QD_I8_ROW || FMT == QD_I4_ROW) {
      const int64_t r = row0 + i < W.rows ? row0 + i : row0;
      row_scale[i] = __ldg(reinterpret_cast<const float*>(W.scales) + r);
    }
  }
  finish_rows<R, NB>(acc, row_scale, row0, W.rows, y, batch, mode, lane);
}

// Q4_K: a lane's unit is 16 code bytes of one 32-byte chunk c of a super-block:
// their low nibbles are 16 elements of sub-block 2c, their high nibbles 16
// elements of sub-block 2c+1.  With w = d*sc*q - dmin*m per sub-block,
//   sum w x = (d*sc) * sum q x - (dmin*m) * sum x,
// and sum x over each half is shared by the warp's rows.
template <int R, int NB>
__global__ void __launch_bounds__(kThreads) k_gemv_q4k(PackedView W, const float* __restrict__ x,
                                                       float* __restrict__ y, int batch, int mode) {
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * R;
  if (row0 >= W.rows) return;
  const int64_t units = W.cols / 32;  // 8 per super-block
  float acc[R][NB];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;

  for (int64_t u = lane; u < units; u += 32) {
    const int64_t s = u >> 3;
    const int c = (int)((u >> 1) & 3), h = (int)(u & 1);
    float wlo[R][16], whi[R][16], a_lo[R], b_lo[R], a_hi[R], b_hi[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int64_t r = row0 + i < W.rows ? row0 + i : row0;
      const uint4 q = ld_stream_v4(W.codes + r * W.row_code_bytes + s * 128 + 32 * c + 16 * h);
      const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(W.scales + r * W.row_scale_bytes + s * 16));
      uint8_t sb[12];
      const uint32_t hw[3] = {hdr.y, hdr.z, hdr.w};
#pragma unroll
      for (int k = 0; k < 12; ++k) sb[k] = (uint8_t)(hw[k >> 2] >> (8 * (k & 3)));
      int sc0, m0, sc1, m1;
      q4k_scale_min(2 * c, sb, sc0, m0);
      q4k_scale_min(2 * c + 1, sb, sc1, m1);
      const float d = f16_bits_to_f32(hdr.x & 0xFFFFu), dmin = f16_bits_to_f32(hdr.x >> 16);
      a_lo[i] = d * (float)sc0;
      b_lo[i] = dmin * (float)m0;
      a_hi[i] = d * (float)sc1;
      b_hi[i] = dmin * (float)m1;
      const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t lo = words[t] & 0x0F0F0F0Fu, hi = (words[t] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          wlo[i][4 * t + k] = byte_as_magic(lo, k) - kMagic;
          whi[i][4 * t + k] = byte_as_magic(hi, k) - kMagic;
        }
      }
    }
    const int64_t xo = s * 256 + 64 * c + 16 * h;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < batch) {
        const float* xp = x + (int64_t)b * W.cols + xo;
        const float4* xl = reinterpret_cast<const float4*>(xp);
        const float4* xh = reinterpret_cast<const float4*>(xp + 32);
        float sxl = 0.f, sxh = 0.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float4 vl = __ldg(xl + t), vh = __ldg(xh + t);
          sxl += (vl.x + vl.y) + (vl.z + vl.w);
          sxh += (vh.x + vh.y) + (vh.z + vh.w);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
          const float ql = dot_x<16>(wlo[i], xp);
          const float qh = dot_x<16>(whi[i], xp + 32);
          float v = fmaf(a_lo[i], ql, -b_lo[i] * sxl);
          v = fmaf(a_hi[i], qh, fmaf(-b_hi[i], sxh, v));
          acc[i][b] += v;
        }
      }
    }
  }
  float row_scale[R];
#pragma unroll
  for (int i = 0; i < R; ++i) row_scale[i] = 1.0f;
  finish_rows<R, NB>(acc, row_scale, row0, W.rows, y, batch, mode, lane);
}

// The formats a Q4_K_M-class file mixes in (Q4_1, Q5_0, Q5_K, Q6_K, F16): the 32
// dequantised f32 values of unit u (columns 32u .. 32u + 31) of row r, each rounded once
// (as the test dequantiser).
__device__ __forceinline__ float f16lo(uint32_t w) { return f16_bits_to_f32(w & 0xFFFFu); }
__device__ __forceinline__ float f16hi(uint32_t w) { return f16_bits_to_f32(w >> 16); }

// Raw bytes of unit u (columns 32u .. 32u + 31) of row r, loaded in one step so that the
// next unit's loads can be in flight while this one is decoded.
template <int FMT>
struct RawUnit {
  uint4 a[4];     // codes: F16 a[0..3]; Q4_1 / Q5_0 a[0]; Q5_K / Q6_K a[0..1] low nibbles, a[2..3] high bits
  uint4 hdr;      // Q5_K header (d, dmin, 12 scale bytes)
  uint32_t s0, s1;  // Q4_1 (d, m); Q5_0 d, qh; Q6_K d, the unit's two scale bytes
  __device__ __forceinline__ void load(const PackedView& W, int64_t r, int64_t u) {
    const uint8_t* cr = W.codes + r * W.row_code_bytes;
    const uint8_t* sr = W.scales + r * W.row_scale_bytes;
    if constexpr (FMT == QD_F16) {
#pragma unroll
      for (int t = 0; t < 4; ++t) a[t] = ld_stream_v4(cr + 64 * u + 16 * t);
    } else if constexpr (FMT == QD_Q4_1) {
      a[0] = ld_stream_v4(cr + 16 * u);
      s0 = __ldg(reinterpret_cast<const uint32_t*>(sr + 4 * u));
    } else if constexpr (FMT == QD_Q5_0) {
      a[0] = ld_stream_v4(cr + 16 * u);
      const unsigned short* h = reinterpret_cast<const unsigned short*>(sr + 6 * u);
      s0 = __ldg(h);
      s1 = (uint32_t)__ldg(h + 1) | ((uint32_t)__ldg(h + 2) << 16);
    } else {  // Q5_K, Q6_K: unit v = u % 8 of super-block u / 8
      const int64_t sb = u >> 3;
      const int v = (int)(u & 7);
      const uint8_t *lp, *hp;
      if constexpr (FMT == QD_Q5_K) {
        lp = cr + sb * 160 + 32 + 32 * (v >> 1);
        hp = cr + sb * 160;
        hdr = __ldg(reinterpret_cast<const uint4*>(sr + sb * 16));
      } else {
        lp = cr + sb * 192 + 64 * (v >> 2) + 32 * (v & 1);
        hp = cr + sb * 192 + 128 + 32 * (v >> 2);
        const uint8_t* h = sr + sb * 18;
        s0 = __ldg(reinterpret_cast<const unsigned short*>(h + 16));
        s1 = __ldg(reinterpret_cast<const unsigned short*>(h + 2 * v));  // scales 2k, 2k + 1 of half v / 4
      }
      a[0] = ld_stream_v4(lp);
      a[1] = ld_stream_v4(lp + 16);
      a[2] = ld_stream_v4(hp);
      a[3] = ld_stream_v4(hp + 16);
    }
  }
  // the 32 dequantised f32 values, each rounded once (as the test dequantiser)
  __device__ __forceinline__ void decode(int64_t u, float (&w)[32]) const {
    if constexpr (FMT == QD_F16) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t h[4] = {a[t].x, a[t].y, a[t].z, a[t].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          w[8 * t + 2 * k] = f16lo(h[k]);
          w[8 * t + 2 * k + 1] = f16hi(h[k]);
        }
      }
    } else if constexpr (FMT == QD_Q4_1 || FMT == QD_Q5_0) {
      const uint32_t q[4] = {a[0].x, a[0].y, a[0].z, a[0].w};
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint32_t byte = (q[j >> 2] >> (8 * (j & 3))) & 0xFFu;
        if constexpr (FMT == QD_Q4_1) {
          const float d = f16lo(s0), m = f16hi(s0);
          w[j] = fmaf(d, (float)(byte & 15u), m);
          w[j + 16] = fmaf(d, (float)(byte >> 4), m);
        } else {
          const float d = f16_bits_to_f32(s0);
          w[j] = (float)((int)((byte & 15u) | (((s1 >> j) & 1u) << 4)) - 16) * d;
          w[j + 16] = (float)((int)((byte >> 4) | (((s1 >> (j + 16)) & 1u) << 4)) - 16) * d;
        }
      }
    } else {
      const int v = (int)(u & 7);
      const uint32_t lw[8] = {a[0].x, a[0].y, a[0].z, a[0].w, a[1].x, a[1].y, a[1].z, a[1].w};
      const uint32_t hw[8] = {a[2].x, a[2].y, a[2].z, a[2].w, a[3].x, a[3].y, a[3].z, a[3].w};
      if constexpr (FMT == QD_Q5_K) {
        uint8_t sbytes[12];
        const uint32_t hs[3] = {hdr.y, hdr.z, hdr.w};
#pragma unroll
        for (int k = 0; k < 12; ++k) sbytes[k] = (uint8_t)(hs[k >> 2] >> (8 * (k & 3)));
        int sc, m;
        q4k_scale_min(v, sbytes, sc, m);  // sub-block v = 2 chunk + high
        const float ca = f16lo(hdr.x) * (float)sc, cb = -(f16hi(hdr.x) * (float)m);
        const int shift = (v & 1) ? 4 : 0;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
          const uint32_t lb = (lw[l >> 2] >> (8 * (l & 3))) & 0xFFu, hb = (hw[l >> 2] >> (8 * (l & 3))) & 0xFFu;
          const int q = (int)(((lb >> shift) & 15u) | (((hb >> v) & 1u) << 4));
          w[l] = fmaf(ca, (float)q, cb);
        }
      } else {
        const int k = v & 3;
        const float d = f16_bits_to_f32(s0);
        const float c0 = d * (float)(int8_t)(s1 & 0xFFu), c1 = d * (float)(int8_t)(s1 >> 8);
        const int shift = k < 2 ? 0 : 4;
#pragma unroll
        for (int l = 0; l < 32; ++l) {
          const uint32_t lb = (lw[l >> 2] >> (8 * (l & 3))) & 0xFFu, hb = (hw[l >> 2] >> (8 * (l & 3))) & 0xFFu;
          const int q = (int)(((lb >> shift) & 15u) | (((hb >> (2 * k)) & 3u) << 4));
          w[l] = (l < 16 ? c0 : c1) * (float)(q - 32);
        }
      }
    }
  }
};

// Q4_1, Q5_0, Q5_K, Q6_K, F16: each lane dequantises its 32-column units to f32 and dots
// them with x.
template <int FMT, int R, int NB>
__global__ void __launch_bounds__(kThreads) k_gemv_deq(PackedView W, const float* __restrict__ x,
                                                        float* __restrict__ y, int batch, int mode) {
  const int lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * R;
  if (row0 >= W.rows) return;
  const int64_t units = W.cols / 32;
  float acc[R][NB];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[i][b] = 0.f;
  RawUnit<FMT> cur[R], nxt[R];
  int64_t u = lane;
  if (u < units) {
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i].load(W, row0 + i < W.rows ? row0 + i : row0, u);
  }
  for (; u < units; u += 32) {
    if (u + 32 < units) {  // the next unit's loads, in flight during this one's arithmetic
#pragma unroll
      for (int i = 0; i < R; ++i) nxt[i].load(W, row0 + i < W.rows ? row0 + i : row0, u + 32);
    }
    float w[R][32];
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i].decode(u, w[i]);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < batch) {
        const float* xp = x + (int64_t)b * W.cols + u * 32;
#pragma unroll
        for (int i = 0; i < R; ++i) acc[i][b] += dot_x<32>(w[i], xp);
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) cur[i] = nxt[i];
  }
  float row_scale[R];
#pragma unroll
  for (int i = 0; i < R; ++i) row_scale[i] = 1.0f;
  finish_rows<R, NB>(acc, row_scale, row0, W.rows, y, batch, mode, lane);
}

template <int FMT, int R, int NB>
qd_status launch_t(const PackedView& W, const float* x, float* y, int batch, int mode, cudaStream_t stream) {
  const int64_t warps = (W.rows + R - 1) / R;
  const int64_t ctas = (warps + kWarpsPerCta - 1) / kWarpsPerCta;
  if constexpr (FMT == QD_Q4_K)
    k_gemv_q4k<R, NB><<<(unsigned)ctas, kThreads, 0, stream>>>(W, x, y, batch, mode);
  else if constexpr (FMT >= QD_Q4_1 && FMT != QD_I4_ROW)
    k_gemv_deq<FMT, R, NB><<<(unsigned)ctas, kThreads, 0, stream>>>(W, x, y, batch, mode);
  else
    k_gemv_blocks<FMT, R, NB><<<(unsigned)ctas, kThreads, 0, stream>>>(W, x, y, batch, mode);
  return launch_status();
}

template <int FMT>
qd_status launch_fmt(const PackedView& W, const float* x, float* y, int batch, int mode, cudaStream_t stream) {
  // The SwiGLU epilogue needs each (gate, up) row pair in one warp: R = 2.
  const bool pair = (mode == kGemvSwiGLU);
  if (batch <= 1) return pair ? launch_t<FMT, 2, 1>(W, x, y, batch, mode, stream)
                              : launch_t<FMT, 2, 1>(W, x, y, batch, mode, stream);
  if (batch <= 2) return launch_t<FMT, 2, 2>(W, x, y, batch, mode, stream);
  if (batch <= 4) return pair ? launch_t<FMT, 2, 4>(W, x, y, batch, mode, stream)
                              : launch_t<FMT, 1, 4>(W, x, y, batch, mode, stream);
  if (batch <= 8) return pair ? launch_t<FMT, 2, 8>(W, x, y, batch, mode, stream)
                              : launch_t<FMT, 1, 8>(W, x, y, batch, mode, stream);
  return pair ? launch_t<FMT, 2, 16>(W, x, y, batch, mode, stream)
              : launch_t<FMT, 1, 16>(W, x, y, batch, mode, stream);
}

}  // namespace

bool gemv_fuses_norm(const GemvArgs& a, const float* gains) {
  GemvArgs n = a;  // decided with the gains in place: they take shared memory too
  n.norm_g = gains;
  return gains && (gemv_mma_supported(n) || gemv_streams(n));
}

qd_status launch_q_gemv(const GemvArgs& a, cudaStream_t stream) {
  // Batch 3-16 (Q4_0, Q8_0, INT8 rows): the mma.sync tensor-core kernel.  Batch 1-8 and the shapes
  // it supports: the streaming kernel.  Both fuse RMSNorm.  Otherwise the register-path
  // kernel below (RMSNorm must then have been applied by the caller, see gemv_fuses_norm).
  {
    const qd_status st = launch_q_gemv_mma(a, stream);
    if (st != QD_ERR_UNSUPPORTED) return st;
  }
  {
    const qd_status st = launch_q_gemv_stream(a, stream);
    if (st != QD_ERR_UNSUPPORTED) return st;
  }
  // Batch 9-16 INT8 rows the mma kernel does not take (x too wide): tcgen05 tensor cores.
  {
    const qd_status st = launch_q_gemv_tc(a, stream);
    if (st != QD_ERR_UNSUPPORTED) return st;
  }
  if (a.norm_g) return QD_ERR_UNSUPPORTED;
  switch (a.fmt) {
    case QD_Q4_0: return launch_fmt<QD_Q4_0>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_Q8_0: return launch_fmt<QD_Q8_0>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_Q4_K: return launch_fmt<QD_Q4_K>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_I8_ROW: return launch_fmt<QD_I8_ROW>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_Q4_1: return launch_fmt<QD_Q4_1>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_Q5_0: return launch_fmt<QD_Q5_0>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_Q5_K: return launch_fmt<QD_Q5_K>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_Q6_K: return launch_fmt<QD_Q6_K>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_F16: return launch_fmt<QD_F16>(a.W, a.x, a.y, a.batch, a.mode, stream);
    case QD_I4_ROW: return launch_fmt<QD_I4_ROW>(a.W, a.x, a.y, a.batch, a.mode, stream);
    default: return QD_ERR_UNSUPPORTED;
  }
}

}  // namespace qd

using namespace qd;

namespace qd {
namespace calib {

// Roofline calibration: every 16-byte chunk of a buffer read once with streaming loads,
// eight in flight per thread, nothing computed; each CTA reads one contiguous run.  The
// sink word is written only by a CTA whose XOR of everything it read is a value that
// random data does not give, which keeps the loads alive.  With `pdl` the kernel lets its
// successor launch at once and waits for its predecessor only before that write, as a
// GEMV waits before it reads x.
__global__ void __launch_bounds__(512) k_read_ceiling(const uint4* __restrict__ p, int64_t n16, uint32_t* sink,
                                                     int pdl) {
  if (pdl) pdl_trigger();
  const int64_t per = (n16 + gridDim.x - 1) / gridDim.x;
  const int64_t b0 = (int64_t)blockIdx.x * per;
  const int64_t b1 = b0 + per < n16 ? b0 + per : n16;
  uint32_t acc = 0;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += 8 * (int64_t)blockDim.x) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int64_t j = i + (int64_t)k * blockDim.x;
      v[k] = j < b1 ? ld_stream_v4(p + j) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  if (pdl) pdl_wait();
  if (acc == 0x9E3779B9u) atomicOr(sink, 1u);
}

}  // namespace calib
}  // namespace qd

extern "C" {

qd_status qd_read_ceiling(const void* buf, size_t bytes, int ctas_per_sm, int threads, unsigned flags,
                          uint32_t* sink, qd_stream_t stream) {
  if (!buf || !sink || (flags & ~QD_GEMV_OVERLAP)) return QD_ERR_INVALID_ARG;
  if (!aligned16(buf) || bytes % 16) return QD_ERR_ALIGN;
  if (ctas_per_sm < 1 || ctas_per_sm > 8 || (threads != 128 && threads != 256 && threads != 512)) return QD_ERR_SHAPE;
  if (bytes == 0) return QD_OK;
  const int sms = attn_sm_count();
  return launch_k(calib::k_read_ceiling, dim3((unsigned)(sms * ctas_per_sm)), dim3((unsigned)threads), 0,
                  (cudaStream_t)stream, (flags & QD_GEMV_OVERLAP) != 0, static_cast<const uint4*>(buf),
                  (int64_t)(bytes / 16), sink, (int)((flags & QD_GEMV_OVERLAP) != 0));
}

size_t qd_q_gemv_workspace(qd_fmt fmt, int64_t rows, int64_t cols, int batch) {
  (void)fmt;
  (void)rows;
  (void)cols;
  (void)batch;
  return 0;
}

qd_status qd_q_gemv(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                    void* workspace, size_t workspace_bytes, qd_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  return qd_q_gemv_ex(fmt, W, rows, cols, x, y, batch, 0u, stream);
}

qd_status qd_q_gemv_ex(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                       unsigned int flags, qd_stream_t stream) {
  if (flags & ~QD_GEMV_OVERLAP) return QD_ERR_INVALID_ARG;
  if (!fmt_ok(fmt)) return QD_ERR_UNSUPPORTED;
  if (!W || !x || !y) return QD_ERR_INVALID_ARG;
  if (batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  if (!shape_ok(fmt, rows, cols)) return QD_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(x) || !aligned16(y)) return QD_ERR_ALIGN;
  GemvArgs a;
  a.fmt = fmt;
  a.W = packed_view(fmt, W, rows, cols);
  a.x = x;
  a.y = y;
  a.batch = batch;
  a.pdl = (flags & QD_GEMV_OVERLAP) != 0;
  return launch_q_gemv(a, (cudaStream_t)stream);
}

size_t qd_q_gemm_workspace(qd_fmt fmt, int64_t rows, int64_t cols, int t) {
  if ((fmt != QD_Q4_0 && fmt != QD_Q8_0 && fmt != QD_I8_ROW) || rows < 1 || cols < 64 || cols % 64 || t < 1 ||
      t > QD_MAX_GEMM_TOKENS)
    return 0;
  return gemm_workspace_bytes(cols, t);
}

qd_status qd_q_gemm(qd_fmt fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int t,
                    void* workspace, size_t workspace_bytes, qd_stream_t stream) {
  if (!fmt_ok(fmt)) return QD_ERR_UNSUPPORTED;
  if (fmt != QD_Q4_0 && fmt != QD_Q8_0 && fmt != QD_I8_ROW) return QD_ERR_UNSUPPORTED;
  if (!W || !x || !y || !workspace) return QD_ERR_INVALID_ARG;
  if (rows < 1 || rows > (int64_t)1 << 30 || cols < 64 || cols % 64 || cols > (int64_t)1 << 20 || t < 1 ||
      t > QD_MAX_GEMM_TOKENS)
    return QD_ERR_SHAPE;
  if (workspace_bytes < gemm_workspace_bytes(cols, t)) return QD_ERR_NOMEM;
  if (!aligned16(W) || !aligned16(x) || !aligned16(y) || !aligned16(workspace)) return QD_ERR_ALIGN;
  return launch_q_gemm(fmt, packed_view(fmt, W, rows, cols), x, y, t, workspace, nullptr, (cudaStream_t)stream);
}

}  // extern "C"
