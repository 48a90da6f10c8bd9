// Integer dot products of quantised weight codes with x held as 24-bit integer planes:
// the record layout, the unit builder and the plane dot products.
//
// Each 32-element unit of x is written as 24-bit integers xq with one power-of-two scale
// (2^-22 of the unit's largest |x| rounded down to a power of two: error at most half a
// step, about the rounding of an f32, exact for dyadic x), held as three byte planes
// (signed high, unsigned middle and low bytes) so that one dp4a multiplies four codes
// with four bytes of a plane: sum q x = s * (65536 sum q x2 + 256 sum q x1 + sum q x0),
// each plane's sum exact in int32.
#pragma once
#include "qd_internal.cuh"

namespace qd {
namespace intdot {

// Four-way byte dot products with an int32 accumulator (a: weight codes, b: x bytes).
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {  // a unsigned, b signed
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {  // both unsigned
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {  // both signed
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {  // a signed, b unsigned
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Element offsets (in x) of the two 16-element halves A, B of unit u:
//  Q4_0: A = [32u, 32u+16), B = [32u+16, 32u+32); code byte i: low nibble -> A[i], high -> B[i]
//  Q4_K, Q5_K: u = 8s + 2c + h, A = [256s+64c+16h, +16), B = A + 32; same nibble rule
//  Q8_0 / INT8: A <- code bytes 0..15, B <- bytes 16..31
template <int FMT>
__device__ __forceinline__ int unit_xa(int u) {
  if constexpr (FMT == QD_Q4_K || FMT == QD_Q5_K) return (u >> 3) * 256 + ((u >> 1) & 3) * 64 + (u & 1) * 16;
  return u * 32;
}
template <int FMT>
__device__ __forceinline__ int unit_xb(int u) {
  return unit_xa<FMT>(u) + ((FMT == QD_Q4_K || FMT == QD_Q5_K) ? 32 : 16);
}
template <int FMT>
constexpr int code_bytes() {
  return (FMT == QD_Q8_0 || FMT == QD_I8_ROW) ? 32 : 16;
}

// Shared-memory x records: per batch row and unit, 112 bytes in seven 16-byte chunks:
// 0/1 the high bytes of halves A/B, 2/3 the middle bytes, 4/5 the low bytes, 6 the
// unit's metadata: the scale s and, for Q4_0 (and INT4 rows, packed as Q4_0 codes), -8
// times each plane's element sum (the code offset, as int bits); for Q4_K and Q4_1, sum x
// over A and over B.  The 7-chunk stride puts 8 lanes reading one chunk of 8 consecutive units
// on 8 different bank groups.
constexpr int kRecBytes = 112;
__device__ __forceinline__ int rec_off(int u, int k) { return u * kRecBytes + 16 * k; }

// Q4_K (scale, min) of sub-block j (0..7) from the 12 scale bytes held as three
// little-endian words; the same bit layout as q4k_scale_min, read from registers.
__device__ __forceinline__ void q4k_sm_words(uint32_t w0, uint32_t w1, uint32_t w2, int j, int& sc, int& m) {
  const int sh = 8 * (j & 3);
  const uint32_t b0 = (w0 >> sh) & 0xFFu, b1 = (w1 >> sh) & 0xFFu, b2 = (w2 >> sh) & 0xFFu;
  const int lo_sc = (int)(b0 & 63u), lo_m = (int)(b1 & 63u);
  const int hi_sc = (int)((b2 & 15u) | ((b0 >> 6) << 4)), hi_m = (int)((b2 >> 4) | ((b1 >> 6) << 4));
  sc = j < 4 ? lo_sc : hi_sc;
  m = j < 4 ? lo_m : hi_m;
}

// Dot of 8 code words (half A: words 0-3, half B: words 4-7) with one byte plane of a
// unit record (chunks ca, ca + 1), starting from c.
template <bool CODES_SIGNED, bool PLANE_SIGNED>
__device__ __forceinline__ int plane_dot(const uint32_t (&w)[8], uint4 pa, uint4 pb, int c) {
  const uint32_t xv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    if constexpr (CODES_SIGNED && PLANE_SIGNED) c = dp4a_ss(w[t], xv[t], c);
    else if constexpr (CODES_SIGNED) c = dp4a_su(w[t], xv[t], c);
    else if constexpr (PLANE_SIGNED) c = dp4a_us(w[t], xv[t], c);
    else c = dp4a_uu(w[t], xv[t], c);
  }
  return c;
}
// Same over 4 code words against one 16-byte chunk.
template <bool PLANE_SIGNED>
__device__ __forceinline__ int half_dot(const uint32_t* w, uint4 p, int c) {
  const uint32_t xv[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) c = PLANE_SIGNED ? dp4a_us(w[t], xv[t], c) : dp4a_uu(w[t], xv[t], c);
  return c;
}
// Same over 4 signed code words (Q6_K's q - 32).
template <bool PLANE_SIGNED>
__device__ __forceinline__ int half_dot_s(const uint32_t* w, uint4 p, int c) {
  const uint32_t xv[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) c = PLANE_SIGNED ? dp4a_ss(w[t], xv[t], c) : dp4a_su(w[t], xv[t], c);
  return c;
}
// 65536 h + 256 m + l as a float (h exact; the rest rounded once).
__device__ __forceinline__ float planes_value(int h, int m, int l) {
  return fmaf((float)h, 65536.f, (float)(m * 256 + l));
}

// Build the record of unit u at `rec` from 8 lanes (k = lane & 7, 0-7) holding 4
// elements each: lane k < 4 the elements 4k..4k+3 of half A, k >= 4 those of half B.
// All 32 lanes of the warp take part (shuffles); lanes with ok == false store nothing.
template <int FMT>
__device__ __forceinline__ void write_record(uint8_t* rec, int k, bool ok, float4 v) {
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
  if (isnan(v.x) || isnan(v.y) || isnan(v.z) || isnan(v.w)) m = INFINITY;  // fmaxf drops NaN
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
  // Power-of-two scale s = 2^(F - 22) for a largest |value| m in [2^F, 2^(F+1)),
  // so |x / s| < 2^23 and x / s is exact for dyadic x (integers, the tests'
  // exact case).  Units with m below 2^-100 are stored as zeros.
  const int F = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  const bool live = F >= -100;
  const float r = live ? __uint_as_float((uint32_t)(127 + 22 - F) << 23) : 0.f;
  // a non-finite x (F = 128) gives a NaN scale, so the row sums become NaN
  const float sc = F == 128 ? __uint_as_float(0x7FC00000u)
                            : live ? __uint_as_float((uint32_t)(127 - 22 + F) << 23) : 0.f;
  // x / s may still round up to 2^23 (one fractional bit): clamp to 24 bits
  auto to_q = [&](float f) { return max(min(__float2int_rn(f * r), 8388607), -8388607); };
  const int q0 = to_q(v.x), q1 = to_q(v.y), q2 = to_q(v.z), q3 = to_q(v.w);
  // bytes 2, 1, 0 of a 24-bit two's-complement value: its signed high part and
  // two unsigned parts, q = 65536 * hi + 256 * mid + lo
  const uint32_t w2 = __byte_perm(__byte_perm(q0, q1, 0x0062u), __byte_perm(q2, q3, 0x0062u), 0x5410u);
  const uint32_t w1 = __byte_perm(__byte_perm(q0, q1, 0x0051u), __byte_perm(q2, q3, 0x0051u), 0x5410u);
  const uint32_t w0 = __byte_perm(__byte_perm(q0, q1, 0x0040u), __byte_perm(q2, q3, 0x0040u), 0x5410u);
  const int off = 16 * (k >> 2) + 4 * (k & 3);
  if (ok) {
    *reinterpret_cast<uint32_t*>(rec + off) = w2;
    *reinterpret_cast<uint32_t*>(rec + 32 + off) = w1;
    *reinterpret_cast<uint32_t*>(rec + 64 + off) = w0;
  }
  float4 meta = make_float4(sc, 0.f, 0.f, 0.f);
  if constexpr (FMT == QD_Q4_0 || FMT == QD_I4_ROW) {
    int s2 = (q0 >> 16) + (q1 >> 16) + (q2 >> 16) + (q3 >> 16);
    int s1 = ((q0 >> 8) & 255) + ((q1 >> 8) & 255) + ((q2 >> 8) & 255) + ((q3 >> 8) & 255);
    int s0 = (q0 & 255) + (q1 & 255) + (q2 & 255) + (q3 & 255);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s0 += __shfl_xor_sync(0xffffffffu, s0, o);
    }
    meta = make_float4(sc, __int_as_float(-8 * s2), __int_as_float(-8 * s1), __int_as_float(-8 * s0));
  } else if constexpr (FMT == QD_Q4_K || FMT == QD_Q5_K || FMT == QD_Q4_1) {
    float sv = (v.x + v.y) + (v.z + v.w);
    sv += __shfl_xor_sync(0xffffffffu, sv, 1);
    sv += __shfl_xor_sync(0xffffffffu, sv, 2);  // lanes 0-3: sum over A, 4-7: over B
    meta = make_float4(sc, sv, __shfl_xor_sync(0xffffffffu, sv, 4), 0.f);
  }
  if (ok && k == 0) *reinterpret_cast<float4*>(rec + 96) = meta;
}



}  // namespace intdot
}  // namespace qd
