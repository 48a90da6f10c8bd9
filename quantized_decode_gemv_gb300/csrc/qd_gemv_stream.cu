// Streaming q_gemv for batch 1-2 on the CUDA cores.
//
// y[b][r] = sum_c deq(W)[r][c] * x[b][c]  (llmoxide blog s1 and s10's row dot;
// dasLLAMA 8.7.1.4 matmul), the weights decoded in registers with no f32 copy
// (minillm-cpp README, "NEON kernels").  Decode reads every weight byte once per
// token (llmoxide s11); the kernel is shaped by measurements on GB300:
//
//  * Each warp owns groups of RW consecutive rows, taken round-robin over every warp
//    of the grid (global warp ids interleave the CTAs so left-over groups spread over
//    all SMs); RW is chosen per shape so the groups split evenly.  Lanes walk a group's
//    32-weight units with stride 32: one 16-byte chunk per lane, unit and row.
//  * Weights stream through a per-warp 4-stage ring in shared memory filled with
//    cp.async: each lane copies its own code chunks (and a few lanes the scale data),
//    so up to three unit steps per warp are in flight without holding registers and
//    without any CTA barrier.  The first copies are issued before
//    `griddepcontrol.wait`, so under programmatic dependent launch the weight fetch
//    overlaps the predecessor kernel.  (A TMA-staged variant with a producer warp and
//    an mbarrier ring reached the same DRAM rate but paid a CTA barrier per tile.)
//  * x * g is staged once per CTA in shared memory, padded to 9 float4 chunks per
//    32-float unit so 32 lanes (32 units) read it without bank conflicts.  With RMSNorm
//    fused, the factor 1/sqrt(mean(x^2) + eps) multiplies each finished row sum.
//  * A 4-bit code q becomes the float 1 + q/16 with one byte permute (q lands in
//    mantissa bits 19-22 of 1.0f); paired FFMA2s accumulate sum f*x, and
//    sum (q-8) x = 16 sum f x - 24 sum x.  8-bit codes land in the low mantissa of 2^23
//    and 2^23 + 128 is subtracted (exact).  Each block scale multiplies a 32-term sum.
//  * A warp reduces its RW x NB row sums with one reduce-scatter and writes them (or
//    feeds the fused epilogues: SwiGLU, RoPE + KV append, argmax).
#include "qd_internal.cuh"

namespace qd {

namespace stream_gemv {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;


// 4-bit code byte k of m (prepared as 0x80 | q<<3 per byte) -> the float 1 + q/16.
__device__ __forceinline__ float q4f(uint32_t m, int k) {
  return __uint_as_float(__byte_perm(m, 0x3F000000u, 0x7044u | ((uint32_t)k << 8)));
}
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// Sum of v[k] over the warp for V values at once: afterwards lanes
// [k*32/V, (k+1)*32/V) hold the total of value k.
template <int V>
__device__ __forceinline__ float reduce_scatter(float (&v)[V], int lane) {
#pragma unroll
  for (int n = V, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? v[k] : v[k + n / 2];
      const float keep = upper ? v[k + n / 2] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float t = v[0];
#pragma unroll
  for (int off = 16 / V; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
  return t;
}

// Shared-memory x: each 32-float unit occupies 9 float4 chunks (one of padding), so
// unit u starts at chunk 9u.  Lanes reading the same chunk of 8 consecutive units land
// on 8 different 16-byte bank groups, and a lane's 8 chunks sit at fixed immediate
// offsets from its unit base.
__device__ __forceinline__ int xchunk(int e) { return (e >> 5) * 9 + ((e & 31) >> 2); }

// Element offsets (in x) of the two 16-float halves A, B of unit u:
//  Q4_0: A = [32u, 32u+16), B = [32u+16, 32u+32); code byte i: low nibble -> A[i], high -> B[i]
//  Q4_K: u = 8s + 2c + h, A = [256s+64c+16h, +16), B = A + 32; same nibble rule
//  Q8_0 / INT8: A <- code bytes 0..15, B <- bytes 16..31
template <int FMT>
__device__ __forceinline__ int unit_xa(int u) {
  if constexpr (FMT == QD_Q4_K) return (u >> 3) * 256 + ((u >> 1) & 3) * 64 + (u & 1) * 16;
  return u * 32;
}
template <int FMT>
__device__ __forceinline__ int unit_xb(int u) {
  return unit_xa<FMT>(u) + ((FMT == QD_Q4_K) ? 32 : 16);
}
// Padded-layout chunk index of the first float4 of half A / B of unit u.
template <int FMT>
__device__ __forceinline__ int unit_ca(int u) {
  return xchunk(unit_xa<FMT>(u));
}
template <int FMT>
__device__ __forceinline__ int unit_cb(int u) {
  return xchunk(unit_xb<FMT>(u));
}
template <int FMT>
constexpr int code_bytes() {
  return (FMT == QD_Q8_0 || FMT == QD_I8_ROW) ? 32 : 16;
}

struct Params {
  PackedView W;
  const float* x;
  float* y;
  const float* norm_g;  // RMSNorm gains for the prologue, or null
  float eps;
  int batch;
  int mode;
  uint32_t* err;
  QkvEpilogue qkv;
  ArgmaxEpilogue am;
};

// kGemvQKV: rows r (even) and r+1 of batch b hold a RoPE pair (q or k) or two
// consecutive v values; rotate and scatter them (see QkvEpilogue).
__device__ __forceinline__ void qkv_pair_out(const Params& p, int64_t r, int b, float a, float bb) {
  const QkvEpilogue& e = p.qkv;
  const int pos = e.pos[b];
  if (pos < 0 || pos >= e.max_ctx) {
    if (p.err) atomicOr(p.err, kErrPosition);
    return;
  }
  const int hd = e.head_dim, half = hd / 2;
  if (r < e.q_rows + e.k_rows) {
    const bool isq = r < e.q_rows;
    const int64_t local = isq ? r : r - e.q_rows;
    const int64_t h = local / hd;
    const int pi = (int)(local % hd) / 2;
    const int d0 = e.pairing == QD_ROPE_HALF ? pi : 2 * pi;
    const int d1 = e.pairing == QD_ROPE_HALF ? pi + half : 2 * pi + 1;
    const float2 cs = *reinterpret_cast<const float2*>(e.rope + ((int64_t)pos * half + pi) * 2);
    const float o0 = a * cs.x - bb * cs.y, o1 = a * cs.y + bb * cs.x;
    float* dst = isq ? e.q_out + (int64_t)b * e.q_stride + h * hd
                     : e.kc + (int64_t)b * e.cache_batch_stride + (h * e.max_ctx + pos) * hd;
    dst[d0] = o0;
    dst[d1] = o1;
  } else {
    const int64_t local = r - e.q_rows - e.k_rows;
    const int64_t h = local / hd;
    const int d = (int)(local % hd);
    float* dst = e.vc + (int64_t)b * e.cache_batch_stride + (h * e.max_ctx + pos) * hd;
    dst[d] = a;
    dst[d + 1] = bb;
  }
}

// Row pointers (codes, scales) of the RW rows of a group; rows past the end repeat
// the last row (their sums are never written).
template <int RW>
struct RowPtrs {
  const uint8_t* c[RW];
  const uint8_t* s[RW];
};
template <int RW>
__device__ __forceinline__ void row_ptrs(RowPtrs<RW>& rp, const PackedView& W, int64_t row0) {
#pragma unroll
  for (int rr = 0; rr < RW; ++rr) {
    const int64_t r = min(row0 + rr, W.rows - 1);
    rp.c[rr] = W.codes + r * W.row_code_bytes;
    rp.s[rr] = W.scales + r * W.row_scale_bytes;
  }
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Per-warp staging ring in shared memory: kStages slots, one unit step each.  A slot
// holds, for the RW rows of the group, every lane's code chunk (lane-major, so each
// lane reads back only what it copied) and then 64 bytes of scale data per row:
// Q4_0/Q8_0 the 32 lanes' f16 scales, Q4_K the 4 super-block headers the 32 units
// span, INT8 the row scale.
constexpr int kStages = 4;
template <int FMT, int RW>
constexpr int slot_code_bytes() {
  return RW * 32 * code_bytes<FMT>();
}
template <int FMT, int RW>
constexpr int slot_bytes() {
  return slot_code_bytes<FMT, RW>() + RW * 64;
}

// Issue the copies of one unit step (unit u of the rows in rp) into the slot at `slot`.
template <int FMT, int RW>
__device__ __forceinline__ void stage_step(uint32_t slot, const RowPtrs<RW>& rp, int u, int lane) {
  constexpr int CB = code_bytes<FMT>();
#pragma unroll
  for (int rr = 0; rr < RW; ++rr) {
    const uint8_t* c = rp.c[rr] + (uint32_t)u * (uint32_t)CB;
    const uint32_t dst = slot + (uint32_t)(rr * 32 + lane) * CB;
#pragma unroll
    for (int k = 0; k < CB / 16; ++k) cp16(dst + 16 * k, c + 16 * k);
    const uint32_t sdst = slot + slot_code_bytes<FMT, RW>() + rr * 64;
    if constexpr (FMT == QD_Q4_0 || FMT == QD_Q8_0) {
      if ((lane & 1) == 0) cp4(sdst + 2 * lane, rp.s[rr] + 2 * (uint32_t)u);  // d of units u, u+1
    } else if constexpr (FMT == QD_Q4_K) {
      if ((lane & 7) == 0) cp16(sdst + 2 * lane, rp.s[rr] + (uint32_t)(u >> 3) * 16u);  // header
    } else {
      if (lane == 0) cp4(sdst, rp.s[rr]);  // row scale
    }
  }
}

template <int NB, int RW>
struct Acc {
  float v[RW][NB];
};

// Compute one unit step from a staged slot into acc.
template <int FMT, int NB, int RW>
__device__ __forceinline__ void compute_step(Acc<NB, RW>& acc, const uint8_t* slot, const float4* xs4, int xstride,
                                             int u, int lane) {
  constexpr int CB = code_bytes<FMT>();
  const uint8_t* sc = slot + slot_code_bytes<FMT, RW>();
  const int ca = unit_ca<FMT>(u), cb = unit_cb<FMT>(u);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float4* xb = xs4 + b * xstride;
    float4 xa4[4], xb4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      xa4[k] = xb[ca + k];
      xb4[k] = xb[cb + k];
    }
    if constexpr (FMT == QD_Q4_0 || FMT == QD_Q4_K) {
      // sums of the unit's two x halves (the 4-bit formats' block offsets)
      float sa = 0.f, sbb = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sa += (xa4[k].x + xa4[k].y) + (xa4[k].z + xa4[k].w);
        sbb += (xb4[k].x + xb4[k].y) + (xb4[k].z + xb4[k].w);
      }
#pragma unroll
      for (int rr = 0; rr < RW; ++rr) {
        const uint4 q = *reinterpret_cast<const uint4*>(slot + (rr * 32 + lane) * CB);
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
        float2 aa = f2(0.f, 0.f), ab = f2(0.f, 0.f), ac = f2(0.f, 0.f), ad = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t ml = ((wv[t] << 3) & 0x78787878u) | 0x80808080u;
          const uint32_t mh = ((wv[t] >> 1) & 0x78787878u) | 0x80808080u;
          aa = __ffma2_rn(f2(q4f(ml, 0), q4f(ml, 1)), f2(xa4[t].x, xa4[t].y), aa);
          ab = __ffma2_rn(f2(q4f(ml, 2), q4f(ml, 3)), f2(xa4[t].z, xa4[t].w), ab);
          ac = __ffma2_rn(f2(q4f(mh, 0), q4f(mh, 1)), f2(xb4[t].x, xb4[t].y), ac);
          ad = __ffma2_rn(f2(q4f(mh, 2), q4f(mh, 3)), f2(xb4[t].z, xb4[t].w), ad);
        }
        const float fa = (aa.x + aa.y) + (ab.x + ab.y);  // sum f x over A
        const float fb = (ac.x + ac.y) + (ad.x + ad.y);  // over B
        if constexpr (FMT == QD_Q4_0) {
          // sum (q-8) x = 16 (fa + fb) - 24 (sum A + sum B)
          const float d = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sc + rr * 64 + 2 * lane));
          acc.v[rr][b] = fmaf(d, fmaf(16.f, fa + fb, -24.f * (sa + sbb)), acc.v[rr][b]);
        } else {
          const uint4 hdr = *reinterpret_cast<const uint4*>(sc + rr * 64 + (lane >> 3) * 16);
          const int cc = (u >> 1) & 3;
          uint8_t sb8[12];
          const uint32_t hw[3] = {hdr.y, hdr.z, hdr.w};
#pragma unroll
          for (int k = 0; k < 12; ++k) sb8[k] = (uint8_t)(hw[k >> 2] >> (8 * (k & 3)));
          int sc0, m0, sc1, m1;
          q4k_scale_min(2 * cc, sb8, sc0, m0);
          q4k_scale_min(2 * cc + 1, sb8, sc1, m1);
          const float dd = f16_bits_to_f32(hdr.x & 0xFFFFu), dmin = f16_bits_to_f32(hdr.x >> 16);
          // sum q x_A = 16 (fa - sum A); value d sc q - dmin m
          float v = fmaf(dd * (float)sc0, 16.f * (fa - sa), -(dmin * (float)m0) * sa);
          v = fmaf(dd * (float)sc1, 16.f * (fb - sbb), fmaf(-(dmin * (float)m1), sbb, v));
          acc.v[rr][b] += v;
        }
      }
    } else {  // Q8_0, INT8: 32 signed bytes
      const float2 off = f2(-(kMagic + 128.f), -(kMagic + 128.f));
#pragma unroll
      for (int rr = 0; rr < RW; ++rr) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(slot + (rr * 32 + lane) * CB);
        const uint4 q1 = *reinterpret_cast<const uint4*>(slot + (rr * 32 + lane) * CB + 16);
        const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        float2 a0 = f2(0.f, 0.f), a1 = f2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint32_t w = wv[t] ^ 0x80808080u;
          const float4 xv = t < 4 ? xa4[t & 3] : xb4[t & 3];
          a0 = __ffma2_rn(__fadd2_rn(f2(byte_as_magic(w, 0), byte_as_magic(w, 1)), off), f2(xv.x, xv.y), a0);
          a1 = __ffma2_rn(__fadd2_rn(f2(byte_as_magic(w, 2), byte_as_magic(w, 3)), off), f2(xv.z, xv.w), a1);
        }
        const float s = (a0.x + a0.y) + (a1.x + a1.y);
        if constexpr (FMT == QD_Q8_0) {
          const float d = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sc + rr * 64 + 2 * lane));
          acc.v[rr][b] = fmaf(d, s, acc.v[rr][b]);
        } else {
          acc.v[rr][b] += s;
        }
      }
    }
  }
}

template <int FMT, int NB, int RW>
__global__ void __launch_bounds__(kThreads, 2) k_gemv_warp(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];  // [warps][kStages] slots, then x [NB][units][9 float4]
  __shared__ float red[kWarps][NB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PackedView& W = p.W;
  const int cols = (int)W.cols;
  const int units = cols / 32;
  const int iters = (units + 31) / 32;  // unit steps per row group
  const int64_t groups = (W.rows + RW - 1) / RW;
  // Global warp ids interleave the CTAs (warp-major), so the groups left over after
  // an even split land on warps spread over every CTA rather than on the first CTAs.
  const int64_t gw = (int64_t)warp * gridDim.x + blockIdx.x, nw = (int64_t)gridDim.x * kWarps;
  constexpr uint32_t SB = slot_bytes<FMT, RW>();
  uint8_t* ring = smem + (size_t)warp * kStages * SB;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  const int xstride = units * 9;  // float4 chunks per batch column
  float4* xs4 = reinterpret_cast<float4*>(smem + (size_t)kWarps * kStages * SB);

  // ---- start streaming the first steps (weights never depend on the previous kernel)
  int64_t lg = gw;  // group of the next copy
  int lj = 0;       // its unit step
  RowPtrs<RW> lrp;
  if (lg < groups) row_ptrs<RW>(lrp, W, lg * RW);
  auto issue = [&](int slot_idx) {
    if (lg < groups) {
      const int u = lane + 32 * lj;
      if (u < units) stage_step<FMT, RW>(ring_s + (uint32_t)slot_idx * SB, lrp, u, lane);
      if (++lj == iters) {
        lj = 0;
        lg += nw;
        if (lg < groups) row_ptrs<RW>(lrp, W, lg * RW);
      }
    }
    cp_commit();
  };
#pragma unroll
  for (int k = 0; k < kStages - 1; ++k) issue(k);

  pdl_wait();  // x is the previous kernel's output

  // ---- stage x * g (x itself without norm) in shared memory.  RMSNorm is
  // x * g / sqrt(mean(x^2) + eps): the scalar 1/sqrt(...) multiplies each finished row
  // sum instead, so one barrier suffices.
  float inv[NB];
  {
    const int chunks = cols / 4;
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.f;
      float4* dst = xs4 + b * xstride;
      const float4* xr = reinterpret_cast<const float4*>(p.x + (int64_t)(b < p.batch ? b : 0) * cols);
      const float4* gr = reinterpret_cast<const float4*>(p.norm_g);
      for (int i = threadIdx.x; i < chunks; i += kThreads) {
        float4 v = __ldcg(xr + i);
        if (b >= p.batch) v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.norm_g) {
          ss[b] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[b]))));
          const float4 g = __ldg(gr + i);
          v = make_float4(v.x * g.x, v.y * g.y, v.z * g.z, v.w * g.w);
        }
        dst[(i >> 3) * 9 + (i & 7)] = v;
      }
      if (p.norm_g) {
        ss[b] = warp_sum(ss[b]);
        if (lane == 0) red[warp][b] = ss[b];
      }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      inv[b] = 1.f;
      if (p.norm_g) {
        float t = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kWarps; ++w2) t += red[w2][b];
        inv[b] = 1.0f / sqrtf(t / (float)cols + p.eps);
      }
    }
  }

  // ---- main loop over this warp's (group, unit step) sequence
  pdl_trigger();  // the next kernel may start its own weight prefetch now
  unsigned long long best0 = 0, best1 = 0;  // kGemvArgmax: best (value, index) keys per batch row
  Acc<NB, RW> acc;
  int cs = 0;  // slot of the step being computed
  int j = 0;
  for (int64_t g = gw; g < groups;) {
    __syncwarp();  // every lane is done with the slot about to be refilled
    issue(cs == 0 ? kStages - 1 : cs - 1);
    cp_wait<kStages - 1>();  // this step's group of copies has landed
    __syncwarp();            // ...for every lane (scales are shared across lanes)
    if (j == 0) {
#pragma unroll
      for (int rr = 0; rr < RW; ++rr)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc.v[rr][b] = 0.f;
    }
    const int u = lane + 32 * j;
    const uint8_t* slot = ring + (size_t)cs * SB;
    if (u < units) compute_step<FMT, NB, RW>(acc, slot, xs4, xstride, u, lane);
    float rsc[RW];  // INT8 row scales (staged with every step)
    if constexpr (FMT == QD_I8_ROW) {
#pragma unroll
      for (int rr = 0; rr < RW; ++rr) rsc[rr] = *reinterpret_cast<const float*>(slot + slot_code_bytes<FMT, RW>() + rr * 64);
    }
    cs = (cs + 1 == kStages) ? 0 : cs + 1;
    if (++j < iters) continue;
    j = 0;

    // ---- end of a group: reduce and write its RW rows
    const int64_t row0 = g * RW;
    if constexpr (FMT == QD_I8_ROW) {
#pragma unroll
      for (int rr = 0; rr < RW; ++rr)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc.v[rr][b] *= rsc[rr];
    }
    constexpr int V = RW * NB, GRP = 32 / V;
    float v[V];
#pragma unroll
    for (int rr = 0; rr < RW; ++rr)
#pragma unroll
      for (int b = 0; b < NB; ++b) v[rr * NB + b] = acc.v[rr][b];
    const int kb_ = (lane / GRP) % NB;  // batch row of this lane's reduced value
    const float tot = reduce_scatter<V>(v, lane) * (kb_ == 0 ? inv[0] : inv[NB - 1]);
    const float partner = __shfl_down_sync(0xffffffffu, tot, (NB * GRP) & 31);  // row +1, same batch
    if ((lane % GRP) == 0) {
      const int k = lane / GRP, rr = k / NB, b = k % NB;
      const int64_t r = row0 + rr;
      if (b < p.batch && r < W.rows) {
        if (p.mode == kGemvSwiGLU) {
          if ((rr & 1) == 0 && r + 1 < W.rows)
            p.y[(int64_t)b * (W.rows / 2) + r / 2] = tot / (1.0f + expf(-tot)) * partner;
        } else if (p.mode == kGemvQKV) {
          if ((rr & 1) == 0 && r + 1 < W.rows) qkv_pair_out(p, r, b, tot, partner);
        } else {
          if (p.mode == kGemvArgmax) {
            const unsigned long long key = argmax_key(tot, (uint32_t)r);
            if (b == 0)
              best0 = key > best0 ? key : best0;
            else
              best1 = key > best1 ? key : best1;
          }
          float* dst = p.y + (int64_t)b * W.rows + r;
          if (p.mode == kGemvAccumulate)
            *dst += tot;
          else
            *dst = tot;
        }
      }
    }
    g += nw;
  }
  cp_wait<0>();  // no copy may still target this CTA's shared memory at exit
  if (p.mode == kGemvArgmax) {
    // warp max of the keys, one atomicMax per warp, then the last CTA finalises
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      unsigned long long k = b == 0 ? best0 : best1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, off);
        k = o > k ? o : k;
      }
      if (lane == 0 && k != 0 && b < p.batch) atomicMax(p.am.key + b, k);
    }
    __threadfence();
    __syncthreads();
    __shared__ bool last;
    if (threadIdx.x == 0) {
      last = atomicAdd(p.am.counter, 1u) == gridDim.x - 1;
      if (last) {
        __threadfence();
        for (int b = 0; b < p.batch; ++b) {
          const unsigned long long k = atomicExch(p.am.key + b, 0ull);
          p.am.tok_out[b] = (int32_t)argmax_key_index(k);
          p.am.pos[b] += 1;
        }
        *p.am.counter = 0u;
        __threadfence();
      }
    }
  }
}

int sm_count() {
  static int n[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (!n[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 152;
    n[dev] = v;
  }
  return n[dev];
}

// Resident CTAs per SM for a kernel at a dynamic shared-memory size (cached).
template <typename K>
int resident_ctas(K kern, size_t smem) {
  static size_t keys[32] = {};
  static int vals[32] = {};
  static int dev_of[32] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < 32; ++i)
    if (keys[i] == smem + 1 && dev_of[i] == dev) return vals[i];
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kThreads, smem) != cudaSuccess || o < 1) o = 1;
  for (int i = 0; i < 32; ++i)
    if (keys[i] == 0) {
      keys[i] = smem + 1;
      vals[i] = o;
      dev_of[i] = dev;
      break;
    }
  return o;
}

template <int FMT, int NB, int RW>
size_t smem_bytes_t(int64_t cols) {
  const size_t units = (size_t)cols / 32;
  const bool q4 = FMT == QD_Q4_0 || FMT == QD_Q4_K;
  (void)q4;
  return (size_t)kWarps * kStages * slot_bytes<FMT, RW>() + (size_t)NB * units * 9 * 16;
}

// Largest shared-memory need over the RW choices (for the support check).
size_t smem_bytes(int fmt, int64_t cols, int nb) {
  switch (fmt) {
    case QD_Q4_0: return nb == 1 ? smem_bytes_t<QD_Q4_0, 1, 4>(cols) : smem_bytes_t<QD_Q4_0, 2, 2>(cols);
    case QD_Q8_0: return nb == 1 ? smem_bytes_t<QD_Q8_0, 1, 4>(cols) : smem_bytes_t<QD_Q8_0, 2, 2>(cols);
    case QD_Q4_K: return nb == 1 ? smem_bytes_t<QD_Q4_K, 1, 4>(cols) : smem_bytes_t<QD_Q4_K, 2, 1>(cols);
    default: return nb == 1 ? smem_bytes_t<QD_I8_ROW, 1, 4>(cols) : smem_bytes_t<QD_I8_ROW, 2, 2>(cols);
  }
}

template <int FMT, int NB, int RW>
qd_status launch_rw(const Params& p, bool pdl, cudaStream_t stream, int64_t ctas) {
  auto kern = k_gemv_warp<FMT, NB, RW>;
  const size_t smem = smem_bytes_t<FMT, NB, RW>(p.W.cols);
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
      return QD_ERR_CUDA;
    attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return QD_ERR_CUDA;
  return QD_OK;
}

// CTAs for RW rows per group: one wave of resident CTAs at most.
template <int FMT, int NB, int RW>
int64_t ctas_for(int64_t rows, int64_t cols) {
  const int64_t groups = (rows + RW - 1) / RW;
  const int64_t want = (groups + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)sm_count() * resident_ctas(k_gemv_warp<FMT, NB, RW>, smem_bytes_t<FMT, NB, RW>(cols));
  return want < cap ? want : cap;
}

// Rows per group: the choice whose groups split most evenly over the warps (the kernel
// lasts as long as its busiest warp), preferring more rows (more reuse of staged x).
template <int FMT, int NB>
qd_status launch_inst(const Params& p, bool pdl, cudaStream_t stream) {
  const int64_t rows = p.W.rows, cols = p.W.cols;
  double best = -1.0;
  int brw = 2;
  int64_t bctas = 1;
  // batch 2 keeps at most 2 rows per group (4 would spill registers), Q4_K batch 2 one;
  // the paired epilogues need an even number of rows per group
  constexpr int kMaxRW = NB == 1 ? 4 : (FMT == QD_Q4_K ? 1 : 2);
  const bool pairs = p.mode == kGemvSwiGLU || p.mode == kGemvQKV;
  for (int rw : {4, 2, 1}) {
    if (rw > kMaxRW || (pairs && rw == 1)) continue;
    int64_t ctas = 1;
    if constexpr (kMaxRW >= 4) {
      if (rw == 4) ctas = ctas_for<FMT, NB, 4>(rows, cols);
    }
    if constexpr (kMaxRW >= 2) {
      if (rw == 2) ctas = ctas_for<FMT, NB, 2>(rows, cols);
    }
    if (rw == 1) ctas = ctas_for<FMT, NB, 1>(rows, cols);
    const int64_t groups = (rows + rw - 1) / rw;
    const int64_t slots = ctas * kWarps;
    const int64_t rounds = (groups + slots - 1) / slots;
    double score;
    if (rounds <= 1) {
      // every group runs at once: the kernel lasts one group, so fewer rows per group
      // (more warps, shorter dependent chains) is faster
      score = 1e6 / rw;
    } else {
      // time ~ rounds * rw rows; useful rows per unit time, small bonus for reuse of x
      score = (double)rows / ((double)rounds * rw * slots) * (1.0 + 0.03 * rw);
    }
    if (score > best) {
      best = score;
      brw = rw;
      bctas = ctas;
    }
  }
  if constexpr (kMaxRW >= 4) {
    if (brw == 4) return launch_rw<FMT, NB, 4>(p, pdl, stream, bctas);
  }
  if constexpr (kMaxRW >= 2) {
    if (brw == 2) return launch_rw<FMT, NB, 2>(p, pdl, stream, bctas);
  }
  return launch_rw<FMT, NB, 1>(p, pdl, stream, bctas);
}

bool supported(const GemvArgs& a) {
  if (a.batch > 2 || a.W.cols % 32) return false;
  if ((a.mode == kGemvSwiGLU || a.mode == kGemvQKV) && a.batch == 2 && a.fmt == QD_Q4_K) return false;
  if (a.W.cols > (1 << 24)) return false;
  if (smem_bytes(a.fmt, a.W.cols, a.batch <= 1 ? 1 : 2) > 200 * 1024) return false;
  // 4-byte scale copies need an even number of blocks per row
  if ((a.fmt == QD_Q4_0 || a.fmt == QD_Q8_0) && ((a.W.cols / 32) & 1)) return false;
  return true;
}

}  // namespace stream_gemv

bool gemv_streams(const GemvArgs& a) { return stream_gemv::supported(a); }

// Returns QD_ERR_UNSUPPORTED when the shape/batch is not handled by the streaming
// kernel (the caller then uses the register-path kernel).
qd_status launch_q_gemv_stream(const GemvArgs& a, cudaStream_t stream) {
  using namespace stream_gemv;
  if (!supported(a)) return QD_ERR_UNSUPPORTED;
  Params p;
  p.W = a.W;
  p.x = a.x;
  p.y = a.y;
  p.norm_g = a.norm_g;
  p.eps = a.eps;
  p.batch = a.batch;
  p.mode = a.mode;
  p.err = a.err;
  p.qkv = a.qkv;
  p.am = a.am;
  const bool nb1 = a.batch <= 1;
  switch (a.fmt) {
    case QD_Q4_0: return nb1 ? launch_inst<QD_Q4_0, 1>(p, a.pdl, stream) : launch_inst<QD_Q4_0, 2>(p, a.pdl, stream);
    case QD_Q8_0: return nb1 ? launch_inst<QD_Q8_0, 1>(p, a.pdl, stream) : launch_inst<QD_Q8_0, 2>(p, a.pdl, stream);
    case QD_Q4_K: return nb1 ? launch_inst<QD_Q4_K, 1>(p, a.pdl, stream) : launch_inst<QD_Q4_K, 2>(p, a.pdl, stream);
    case QD_I8_ROW:
      return nb1 ? launch_inst<QD_I8_ROW, 1>(p, a.pdl, stream) : launch_inst<QD_I8_ROW, 2>(p, a.pdl, stream);
    default: return QD_ERR_UNSUPPORTED;
  }
}

}  // namespace qd

