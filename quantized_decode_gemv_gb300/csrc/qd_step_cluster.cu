// The decode step's layers as one thread-block cluster per sequence.
//
// Same step as the kernel chain of qd_model.cu (llmoxide blog s7 "The block, and the
// residual stream"; dasLLAMA 8.7.1.6 forward): per layer RMSNorm, the fused QKV product
// with RoPE and the cache append, GQA attention over positions 0..pos, the Wo product
// with the residual add, RMSNorm, the gate/up product with SwiGLU, the down product with
// the residual add.  For small models every one of those five steps is a few
// microseconds of work spread over the GPU, and a dependent kernel boundary per step costs
// about as much as the work.  Here the C CTAs of one cluster (C = 16, or 8) run all layers
// of one sequence:
//
//  * Each CTA owns a fixed slice of the rows of every product (row pairs for the RoPE and
//    SwiGLU pairs) and of the attention positions.  A step's outputs stay in the producing
//    CTA's shared memory; one cluster barrier later, every CTA pulls the whole vector it
//    needs from its owners' shared memory (distributed shared memory).  Measured on GB300:
//    the cluster barrier ~0.34 us at any size up to 16, a pull ~0.25 us, against ~1 us for a
//    kernel boundary and ~1.8 us for a handoff through global memory across the grid.
//  * The CTA's weight slice of the next product but one is fetched by 1-D bulk copies
//    (cp.async.bulk, completion counted in bytes on an mbarrier) into one of two shared
//    buffers while the current products run; the cached K/V rows of the CTA's attention
//    positions are fetched the same way at the start of each layer.
//  * Products use the streaming GEMV's integer arithmetic (x as 24-bit integer planes,
//    dp4a against the codes, see qd_intdot.cuh), the RMSNorm scale applied to the finished
//    row sums.
//  * Attention: each CTA takes one (kv head, position chunk) unit, computes its G query
//    heads' (max, sum, weighted values) over the chunk, and the Wo step merges the chunks
//    of every head after the pull (log-sum-exp merge in chunk order).
//
// The output head (tied embedding, with the final RMSNorm and the greedy argmax) stays a
// separate GEMV over all SMs, launched as a programmatic dependent of this kernel.
// No spin on global memory: the only waits are cluster barriers (hardware) and bounded
// mbarrier waits on the CTA's own bulk copies (a timeout sets kErrTimeout).
#include <cooperative_groups.h>

#include <algorithm>

#include "qd_intdot.cuh"
#include "qd_tc.cuh"

namespace qd {
namespace cstep {

namespace cg = cooperative_groups;
using namespace intdot;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kHd = 64;                 // head width
constexpr int kPart = kHd + 2;          // one attention partial: m, l, o[64]
constexpr float kQScale = 0.18033688011112042f;  // log2(e) / sqrt(64)

// One weight matrix of a layer: byte offsets from the layer's base, and its row bytes.
struct Mat {
  int64_t codes, scales;
  int32_t rcb, rsb;  // code / scale bytes per row
};

struct Params {
  const uint8_t* w;                 // weight memory
  int64_t layer0, layer_stride;     // first layer's offset, bytes between layers
  int64_t off_attn_norm, off_ffn_norm;
  Mat qkv, wo, gu, wd;
  PackedView emb;
  int emb_fmt;
  int layers, D, F, QD, KD, G, n_kv, max_ctx, pairing, vocab;
  float eps;
  const int32_t* tok;
  const int32_t* pos;
  float* kc;
  float* vc;
  int64_t cache_layer_stride, cache_batch_stride;  // elements
  const float* rope;                               // [max_ctx][32][2]
  float* x_out;                                    // [batch][D]
  uint32_t* err;
  // work split and shared-memory layout (host-computed)
  int S;                // attention chunks per kv head (units = n_kv * S <= C)
  int kvp;              // largest chunk, positions
  int nmax;             // floats per output slot
  uint32_t wbuf_bytes;  // one weight buffer (a product's slice, then the norm gains it takes)
  uint32_t off_wbuf, off_kv, off_slot, off_x, off_v, off_rec, off_sc, off_misc, off_bar;
  uint32_t smem_bytes;
};

__device__ __forceinline__ int64_t lo_of(int r, int64_t n, int c) { return (int64_t)r * n / c; }
// Owner of item i when n items are split evenly over c CTAs (CTA r takes [r n/c, (r+1) n/c)).
__device__ __forceinline__ int owner_of(int64_t i, int64_t n, int c) { return (int)(((i + 1) * c - 1) / n); }

// Position of natural dim d of a RoPE'd head in the packed (pair-adjacent) row order.
__device__ __forceinline__ int packed_dim(int d, int pairing) {
  if (pairing != QD_ROPE_HALF) return d;
  return d < kHd / 2 ? 2 * d : 2 * (d - kHd / 2) + 1;
}

// Byte offset, inside a weight buffer, of the scale data and of the norm gains that follow
// a slice of rows [r0, r1).
__host__ __device__ __forceinline__ int64_t slice_scale_off(int64_t r0, int64_t r1, int64_t rcb) {
  return ((r1 - r0) * rcb + 15) & ~(int64_t)15;
}
__host__ __device__ __forceinline__ int64_t slice_gain_off(int64_t r0, int64_t r1, int64_t rcb, int64_t rsb) {
  const int64_t s0 = (r0 * rsb) & ~(int64_t)15, s1 = (r1 * rsb + 15) & ~(int64_t)15;
  return slice_scale_off(r0, r1, rcb) + (s1 - s0);
}

// Bulk-copy the slice of rows [r0, r1) of matrix m (layer base lw) into buffer dst:
// codes at 0, scales from slice_scale_off (the scale range widened to 16-byte boundaries,
// so the first row's scales start at byte (r0 * rsb) % 16 of it), then, when gains is
// set, n_gain f32 norm gains at slice_gain_off.  Issued by one thread.
__device__ __forceinline__ void fetch_rows(const uint8_t* lw, const Mat& m, int64_t r0, int64_t r1, uint32_t dst,
                                           uint32_t mbar, const float* gains, int n_gain) {
  const uint32_t cb = (uint32_t)((r1 - r0) * m.rcb);
  const int64_t s0 = (r0 * m.rsb) & ~(int64_t)15, s1 = (r1 * m.rsb + 15) & ~(int64_t)15;
  const uint32_t sb = (uint32_t)(s1 - s0);
  const uint32_t gb = gains ? (uint32_t)n_gain * 4u : 0u;
  tc::mbar_arrive_expect_tx(mbar, cb + sb + gb);
  if (cb) tc::bulk_copy_g2s(dst, lw + m.codes + r0 * m.rcb, cb, mbar);
  if (sb) tc::bulk_copy_g2s(dst + (uint32_t)slice_scale_off(r0, r1, m.rcb), lw + m.scales + s0, sb, mbar);
  if (gb) tc::bulk_copy_g2s(dst + (uint32_t)slice_gain_off(r0, r1, m.rcb, m.rsb), gains, gb, mbar);
}

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

// 24-bit plane records of v (n values, n % 32 == 0) times g (optional) into rec; 8 threads
// per unit.
template <int FMT>
__device__ __forceinline__ void build_records(const float* v, const float* g, int n, uint8_t* rec) {
  const int units = n / 32;
  for (int base = 0; base < units * 8; base += kThreads) {  // uniform loop
    const int idx = base + (int)threadIdx.x;
    const int u = idx >> 3, k = idx & 7;
    const bool ok = u < units;
    float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
    if (ok) {
      const int e = k < 4 ? unit_xa<FMT>(u) + 4 * k : unit_xb<FMT>(u) + 4 * (k - 4);
      x4 = *reinterpret_cast<const float4*>(v + e);
      if (g) {
        const float4 g4 = *reinterpret_cast<const float4*>(g + e);
        x4 = make_float4(x4.x * g4.x, x4.y * g4.y, x4.z * g4.z, x4.w * g4.w);
      }
    }
    // every lane of the warp takes part in the record's shuffles
    write_record<FMT>(rec + (size_t)(ok ? u : 0) * kRecBytes, k, ok, x4);
  }
}

// A unit record held in registers.
struct Rec {
  uint4 hA, hB, mA, mB, lA, lB;
  float4 mt;
};
__device__ __forceinline__ Rec load_rec(const uint8_t* r) {
  Rec q;
  q.hA = *reinterpret_cast<const uint4*>(r + 0);
  q.hB = *reinterpret_cast<const uint4*>(r + 16);
  q.mA = *reinterpret_cast<const uint4*>(r + 32);
  q.mB = *reinterpret_cast<const uint4*>(r + 48);
  q.lA = *reinterpret_cast<const uint4*>(r + 64);
  q.lB = *reinterpret_cast<const uint4*>(r + 80);
  q.mt = *reinterpret_cast<const float4*>(r + 96);
  return q;
}

// One unit of one row: d * s * sum(codes x) (Q4_0 / Q8_0).
template <int FMT>
__device__ __forceinline__ float unit_dot(const uint8_t* cp, const uint8_t* sp, int u, const Rec& q) {
  uint32_t w[8];
  if constexpr (FMT == QD_Q4_0) {
    const uint4 c = *reinterpret_cast<const uint4*>(cp + 16 * u);
    const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      w[t] = wv[t] & 0x0F0F0F0Fu;
      w[t + 4] = (wv[t] >> 4) & 0x0F0F0F0Fu;
    }
  } else {
    const uint4 c0 = *reinterpret_cast<const uint4*>(cp + 32 * u), c1 = *reinterpret_cast<const uint4*>(cp + 32 * u + 16);
    w[0] = c0.x; w[1] = c0.y; w[2] = c0.z; w[3] = c0.w;
    w[4] = c1.x; w[5] = c1.y; w[6] = c1.z; w[7] = c1.w;
  }
  const float d = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sp + 2 * u));
  float pv;
  if constexpr (FMT == QD_Q4_0) {
    pv = planes_value(plane_dot<false, true>(w, q.hA, q.hB, __float_as_int(q.mt.y)),
                      plane_dot<false, false>(w, q.mA, q.mB, __float_as_int(q.mt.z)),
                      plane_dot<false, false>(w, q.lA, q.lB, __float_as_int(q.mt.w)));
  } else {
    pv = planes_value(plane_dot<true, true>(w, q.hA, q.hB, 0), plane_dot<true, false>(w, q.mA, q.mB, 0),
                      plane_dot<true, false>(w, q.lA, q.lB, 0));
  }
  return d * q.mt.x * pv;
}

constexpr int kRW = 4;  // rows per warp step

// The CTA's rows of one product: groups of kRW consecutive rows go round-robin to the
// warps; lane l holds the records of units l and l + 32 (the input has at most 64 units),
// so a row costs each lane one or two unit dots and the group one reduce-scatter.
// `epi(row, value, partner)` runs in one lane per row with the row's total (and the next
// row's, for pairs).
template <int FMT, int NU, typename Epi>
__device__ __forceinline__ void rows_product_nu(const uint8_t* buf, const uint8_t* sbuf, int64_t rcb, int64_t rsb,
                                                int64_t nrows, const uint8_t* rec, int units, Epi epi) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool has0 = lane < units, has1 = NU > 1 && lane + 32 < units;
  Rec q0{}, q1{};
  if (has0) q0 = load_rec(rec + (size_t)lane * kRecBytes);
  if constexpr (NU > 1) {
    if (has1) q1 = load_rec(rec + (size_t)(lane + 32) * kRecBytes);
  }
  constexpr int GRP = 32 / kRW;
  for (int64_t g = (int64_t)warp * kRW; g < nrows; g += (int64_t)kWarps * kRW) {  // uniform per warp
    float acc[kRW];
#pragma unroll
    for (int rr = 0; rr < kRW; ++rr) {
      acc[rr] = 0.f;
      const int64_t i = min(g + rr, nrows - 1);
      const uint8_t* cp = buf + i * rcb;
      const uint8_t* sp = sbuf + i * rsb;
      if (has0) acc[rr] += unit_dot<FMT>(cp, sp, lane, q0);
      if constexpr (NU > 1) {
        if (has1) acc[rr] += unit_dot<FMT>(cp, sp, lane + 32, q1);
      }
    }
    const float tot = reduce_scatter<kRW>(acc, lane);
    const float partner = __shfl_down_sync(0xffffffffu, tot, GRP);
    if ((lane % GRP) == 0) {
      const int64_t i = g + lane / GRP;
      if (i < nrows) epi(i, tot, partner);
    }
  }
}
template <int FMT, typename Epi>
__device__ __forceinline__ void rows_product(const uint8_t* buf, const uint8_t* sbuf, int64_t rcb, int64_t rsb,
                                             int64_t nrows, const uint8_t* rec, int units, Epi epi) {
  if (units <= 32)
    rows_product_nu<FMT, 1>(buf, sbuf, rcb, rsb, nrows, rec, units, epi);
  else
    rows_product_nu<FMT, 2>(buf, sbuf, rcb, rsb, nrows, rec, units, epi);
}

// Pull elements [0, n) of the vector held slice by slice in the CTAs' output slots (same
// offset `slot` in every CTA) into dst, owner(i) naming the CTA of element i.  Loads go
// out eight at a time per thread before any is stored.  Returns this thread's sum of
// squares of what it pulled.
template <typename Owner>
__device__ __forceinline__ float pull(cg::cluster_group& cl, float* slot, float* dst, int n, Owner owner) {
  float ss = 0.f;
  for (int base = 0; base < n; base += 8 * kThreads) {
    float v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = base + k * kThreads + (int)threadIdx.x;
      v[k] = i < n ? *cl.map_shared_rank(slot + i, owner(i)) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = base + k * kThreads + (int)threadIdx.x;
      if (i < n) dst[i] = v[k];
      ss = fmaf(v[k], v[k], ss);
    }
  }
  return ss;
}

// Sum over the CTA of one value per thread (every thread gets the total); one barrier.
__device__ __forceinline__ float cta_sum(float v, float* red, int parity) {
  v = warp_sum(v);
  float* r = red + 32 * parity;  // alternate halves so back-to-back calls need no second barrier
  if ((threadIdx.x & 31) == 0) r[threadIdx.x >> 5] = v;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) tot += r[w];
  return tot;
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_step_cluster(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int b = (int)(blockIdx.x / (unsigned)C);  // sequence
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;

  uint8_t* wbuf0 = smem + p.off_wbuf;
  float* kvbuf = reinterpret_cast<float*>(smem + p.off_kv);  // K rows, then V rows
  float* slot0 = reinterpret_cast<float*>(smem + p.off_slot);
  float* x = reinterpret_cast<float*>(smem + p.off_x);       // residual stream [D]
  float* v = reinterpret_cast<float*>(smem + p.off_v);       // a product's input / QKV [nmax]
  uint8_t* rec = smem + p.off_rec;
  float* sc = reinterpret_cast<float*>(smem + p.off_sc);     // attention weights [G][kvp]
  float* misc = reinterpret_cast<float*>(smem + p.off_misc);  // [0, 64) RoPE row, [64, 128) reductions
  float* rope_s = misc;
  float* red = misc + 64;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);  // [0], [1] weights, [2] K/V
  const uint32_t wbar[2] = {tc::smem_u32(&bars[0]), tc::smem_u32(&bars[1])};
  const uint32_t kvbar = tc::smem_u32(&bars[2]);

  pdl_trigger();  // the head GEMV may launch and stream its weights meanwhile

  const int D = p.D, F = p.F, QD = p.QD, KD = p.KD, G = p.G;
  const int R = QD + 2 * KD;  // packed QKV rows
  const int P = R / 2;        // QKV row pairs
  const int pos = __ldcg(p.pos + b);
  const int tok = __ldcg(p.tok + b);
  const bool pos_ok = pos >= 0 && pos < p.max_ctx;
  const bool tok_ok = tok >= 0 && tok < p.vocab;
  if (t == 0 && rank == 0 && p.err) {
    if (!pos_ok) atomicOr(p.err, kErrPosition);
    if (!tok_ok) atomicOr(p.err, kErrToken);
  }
  const bool live = pos_ok && tok_ok;  // uniform over the cluster

  // this CTA's rows of each product
  const int64_t q0 = lo_of(rank, P, C), q1 = lo_of(rank + 1, P, C);  // QKV pairs
  const int64_t o0 = lo_of(rank, D, C), o1 = lo_of(rank + 1, D, C);  // Wo / down rows
  const int64_t g0 = lo_of(rank, F, C), g1 = lo_of(rank + 1, F, C);  // gate/up pairs
  // this CTA's attention unit: kv head h, chunk s of positions [0, pos]
  const bool has_unit = rank < p.n_kv * p.S;
  const int uh = has_unit ? rank / p.S : 0, us = has_unit ? rank % p.S : 0;
  const int npos = pos + 1;
  const int c0 = (int)((int64_t)us * npos / p.S), c1 = (int)((int64_t)(us + 1) * npos / p.S);
  const int cached_end = min(c1, pos);  // rows from the cache: [c0, cached_end); pos from QKV
  const int nch = live && has_unit ? max(0, c1 - c0) : 0;  // this chunk's positions

  if (t == 0) {
    tc::mbar_init(wbar[0], 1);
    tc::mbar_init(wbar[1], 1);
    tc::mbar_init(kvbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (t < kHd) rope_s[t] = live ? __ldg(p.rope + (int64_t)pos * kHd + t) : (t & 1 ? 0.f : 1.f);
  __syncthreads();

  auto layer_base = [&](int l) { return p.w + p.layer0 + (int64_t)l * p.layer_stride; };
  // weight phase j = 4l + k (k: 0 QKV, 1 Wo, 2 gate/up, 3 down) -> buffer j & 1; the QKV
  // and gate/up slices bring their norm gains
  auto issue_w = [&](int j) {
    if (t != 0 || j >= 4 * p.layers) return;
    const uint8_t* lw = layer_base(j >> 2);
    const uint32_t dst = tc::smem_u32(wbuf0 + (size_t)(j & 1) * p.wbuf_bytes);
    switch (j & 3) {
      case 0:
        fetch_rows(lw, p.qkv, 2 * q0, 2 * q1, dst, wbar[j & 1], reinterpret_cast<const float*>(lw + p.off_attn_norm), D);
        break;
      case 1: fetch_rows(lw, p.wo, o0, o1, dst, wbar[j & 1], nullptr, 0); break;
      case 2:
        fetch_rows(lw, p.gu, 2 * g0, 2 * g1, dst, wbar[j & 1], reinterpret_cast<const float*>(lw + p.off_ffn_norm), D);
        break;
      default: fetch_rows(lw, p.wd, o0, o1, dst, wbar[j & 1], nullptr, 0); break;
    }
  };
  bool timed_out = false;
  auto wait_w = [&](int j) {
    if (!tc::mbar_wait_sleep(wbar[j & 1], (uint32_t)((j >> 1) & 1))) timed_out = true;
  };
  issue_w(0);
  issue_w(1);

  // ---- embedding: every CTA decodes the whole row of its sequence's token
  float ss = 0.f;
  for (int i = t; i < D; i += kThreads) {
    const float e = tok_ok ? dequant_elem(p.emb_fmt, p.emb, tok, i) : 0.f;
    x[i] = e;
    ss = fmaf(e, e, ss);
  }
  int rp = 0;  // alternating half of `red`
  float sumsq = cta_sum(ss, red, rp ^= 1);

  int ph = 0;  // cluster phase counter: output slot ph & 1
  for (int l = 0; l < p.layers; ++l) {
    const int64_t cl_off = (int64_t)l * p.cache_layer_stride + (int64_t)b * p.cache_batch_stride;
    // ---- K/V rows of this CTA's attention chunk (positions before pos are final)
    if (t == 0) {
      const int nrow = nch > 0 ? max(0, cached_end - c0) : 0;
      const uint32_t bytes = (uint32_t)nrow * kHd * 4;
      tc::mbar_arrive_expect_tx(kvbar, 2 * bytes);
      if (bytes) {
        const int64_t e = cl_off + ((int64_t)uh * p.max_ctx + c0) * kHd;
        tc::bulk_copy_g2s(tc::smem_u32(kvbuf), p.kc + e, bytes, kvbar);
        tc::bulk_copy_g2s(tc::smem_u32(kvbuf + (size_t)p.kvp * kHd), p.vc + e, bytes, kvbar);
      }
    }

    // ================= QKV (weight phase 4l): RMSNorm, product, RoPE, cache append
    {
      const float inv = 1.0f / sqrtf(sumsq / (float)D + p.eps);
      wait_w(4 * l);
      const uint8_t* buf = wbuf0 + (size_t)((4 * l) & 1) * p.wbuf_bytes;
      const int64_t r0 = 2 * q0, r1 = 2 * q1;
      const float* gains = reinterpret_cast<const float*>(buf + slice_gain_off(r0, r1, p.qkv.rcb, p.qkv.rsb));
      build_records<FMT>(x, gains, D, rec);
      __syncthreads();
      float* slot = slot0 + (size_t)(ph & 1) * p.nmax;
      const uint8_t* sbuf = buf + slice_scale_off(r0, r1, p.qkv.rcb) + ((r0 * p.qkv.rsb) & 15);
      rows_product<FMT>(buf, sbuf, p.qkv.rcb, p.qkv.rsb, r1 - r0, rec, D / 32, [&](int64_t i, float a, float bb) {
        if (i & 1) return;  // the pair's first row writes both
        const int64_t row = r0 + i;
        a *= inv;
        bb *= inv;
        if (row < QD + KD) {  // a RoPE pair of q or k
          const bool isq = row < QD;
          const int64_t local = isq ? row : row - QD;
          const int pi = (int)(local % kHd) / 2;
          const float cs = rope_s[2 * pi], sn = rope_s[2 * pi + 1];
          const float r0v = a * cs - bb * sn, r1v = a * sn + bb * cs;
          a = r0v;
          bb = r1v;
          if (!isq && live) {
            const int64_t h = local / kHd;
            const int d0 = p.pairing == QD_ROPE_HALF ? pi : 2 * pi;
            const int d1 = p.pairing == QD_ROPE_HALF ? pi + kHd / 2 : 2 * pi + 1;
            const int64_t e = cl_off + (h * p.max_ctx + pos) * kHd;
            p.kc[e + d0] = a;
            p.kc[e + d1] = bb;
          }
        } else if (live) {  // two consecutive v values
          const int64_t local = row - QD - KD;
          const int64_t e = cl_off + ((local / kHd) * p.max_ctx + pos) * kHd + local % kHd;
          p.vc[e] = a;
          p.vc[e + 1] = bb;
        }
        slot[row] = a;
        slot[row + 1] = bb;
      });
      cl.sync();
      issue_w(4 * l + 2);  // into the buffer the QKV slice used
      pull(cl, slot, v, R, [&](int i) { return owner_of(i / 2, P, C); });
      ++ph;
      __syncthreads();
    }

    // ================= attention: this CTA's (kv head, chunk) unit for its G query heads
    {
      float* slot = slot0 + (size_t)(ph & 1) * p.nmax;
      if (!tc::mbar_wait_sleep(kvbar, (uint32_t)(l & 1))) timed_out = true;
      if (has_unit) {  // uniform per CTA
        const float* Kn = v + QD + uh * kHd;       // the new key (packed order)
        const float* Vn = v + QD + KD + uh * kHd;  // the new value
        // scores: thread (g, position), a full 64-dim dot with four partial sums
        for (int gp = t; gp < G * nch; gp += kThreads) {
          const int g = gp / nch, pp = gp % nch;
          const float* qh = v + (uh * G + g) * kHd;
          const bool fresh = c0 + pp == pos;
          const float* kr = kvbuf + (size_t)pp * kHd;
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 16
          for (int d = 0; d < kHd; ++d) {
            const int pd = packed_dim(d, p.pairing);
            s4[d & 3] = fmaf(qh[pd], fresh ? Kn[pd] : kr[d], s4[d & 3]);
          }
          sc[g * p.kvp + pp] = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * kQScale;
        }
        __syncthreads();
        // per head (warp g): max, weights 2^(s - m), sum
        if (warp < G) {
          float m = -INFINITY;
          for (int pp = lane; pp < nch; pp += 32) m = fmaxf(m, sc[warp * p.kvp + pp]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
          float sw = 0.f;
          for (int pp = lane; pp < nch; pp += 32) {
            const float w = exp2f(sc[warp * p.kvp + pp] - m);
            sc[warp * p.kvp + pp] = w;
            sw += w;
          }
          sw = warp_sum(sw);
          if (lane == 0) {
            float* part = slot + (size_t)(rank * G + warp) * kPart;
            part[0] = nch > 0 ? m : -INFINITY;
            part[1] = sw;
          }
        }
        __syncthreads();
        // weighted values: thread (g, d), four partial sums over the positions
        for (int gd = t; gd < G * kHd; gd += kThreads) {
          const int g = gd / kHd, d = gd % kHd;
          float o4[4] = {0.f, 0.f, 0.f, 0.f};
          const float* wg = sc + g * p.kvp;
          for (int pp = 0; pp < nch; ++pp) {
            const float vv = c0 + pp == pos ? Vn[d] : kvbuf[(size_t)(p.kvp + pp) * kHd + d];
            o4[pp & 3] = fmaf(wg[pp], vv, o4[pp & 3]);
          }
          slot[(size_t)(rank * G + g) * kPart + 2 + d] = (o4[0] + o4[1]) + (o4[2] + o4[3]);
        }
      }
      cl.sync();
      // merge every query head's chunks straight from their owners (log-sum-exp, chunk
      // order) into v (natural order)
      for (int hd = t; hd < QD; hd += kThreads) {
        const int hq = hd / kHd, d = hd % kHd;
        const int h = hq / G, g = hq % G;
        float M = -INFINITY;
#pragma unroll 4
        for (int s = 0; s < p.S; ++s) {
          const int u = h * p.S + s;
          M = fmaxf(M, *cl.map_shared_rank(slot + (size_t)(u * G + g) * kPart, u));
        }
        float num = 0.f, den = 0.f;
#pragma unroll 4
        for (int s = 0; s < p.S; ++s) {
          const int u = h * p.S + s;
          const float* part = cl.map_shared_rank(slot + (size_t)(u * G + g) * kPart, u);
          const float m = part[0];
          const float w = m == -INFINITY ? 0.f : exp2f(m - M);
          num = fmaf(w, part[2 + d], num);
          den = fmaf(w, part[1], den);
        }
        v[hd] = den > 0.f ? num / den : 0.f;
      }
      ++ph;
      __syncthreads();
    }

    // ================= Wo (weight phase 4l + 1) + residual
    {
      build_records<FMT>(v, nullptr, QD, rec);
      wait_w(4 * l + 1);
      __syncthreads();
      float* slot = slot0 + (size_t)(ph & 1) * p.nmax;
      const uint8_t* buf = wbuf0 + (size_t)((4 * l + 1) & 1) * p.wbuf_bytes;
      const uint8_t* sbuf = buf + slice_scale_off(o0, o1, p.wo.rcb) + ((o0 * p.wo.rsb) & 15);
      rows_product<FMT>(buf, sbuf, p.wo.rcb, p.wo.rsb, o1 - o0, rec, QD / 32, [&](int64_t i, float a, float) {
        slot[o0 + i] = x[o0 + i] + a;
      });
      cl.sync();
      issue_w(4 * l + 3);
      sumsq = cta_sum(pull(cl, slot, x, D, [&](int i) { return owner_of(i, D, C); }), red, rp ^= 1);
      ++ph;
    }

    // ================= gate/up (weight phase 4l + 2): RMSNorm, product, SwiGLU
    {
      const float inv = 1.0f / sqrtf(sumsq / (float)D + p.eps);
      wait_w(4 * l + 2);
      const uint8_t* buf = wbuf0 + (size_t)((4 * l + 2) & 1) * p.wbuf_bytes;
      const int64_t r0 = 2 * g0, r1 = 2 * g1;
      const float* gains = reinterpret_cast<const float*>(buf + slice_gain_off(r0, r1, p.gu.rcb, p.gu.rsb));
      build_records<FMT>(x, gains, D, rec);
      __syncthreads();
      float* slot = slot0 + (size_t)(ph & 1) * p.nmax;
      const uint8_t* sbuf = buf + slice_scale_off(r0, r1, p.gu.rcb) + ((r0 * p.gu.rsb) & 15);
      rows_product<FMT>(buf, sbuf, p.gu.rcb, p.gu.rsb, r1 - r0, rec, D / 32, [&](int64_t i, float a, float bb) {
        if (i & 1) return;
        const float gt = a * inv, up = bb * inv;
        slot[g0 + i / 2] = gt / (1.0f + expf(-gt)) * up;
      });
      cl.sync();
      issue_w(4 * l + 4);  // next layer's QKV
      pull(cl, slot, v, F, [&](int i) { return owner_of(i, F, C); });
      ++ph;
      __syncthreads();
    }

    // ================= down (weight phase 4l + 3) + residual
    {
      build_records<FMT>(v, nullptr, F, rec);
      wait_w(4 * l + 3);
      __syncthreads();
      float* slot = slot0 + (size_t)(ph & 1) * p.nmax;
      const uint8_t* buf = wbuf0 + (size_t)((4 * l + 3) & 1) * p.wbuf_bytes;
      const uint8_t* sbuf = buf + slice_scale_off(o0, o1, p.wd.rcb) + ((o0 * p.wd.rsb) & 15);
      rows_product<FMT>(buf, sbuf, p.wd.rcb, p.wd.rsb, o1 - o0, rec, F / 32, [&](int64_t i, float a, float) {
        slot[o0 + i] = x[o0 + i] + a;
      });
      cl.sync();
      issue_w(4 * l + 5);  // next layer's Wo
      sumsq = cta_sum(pull(cl, slot, x, D, [&](int i) { return owner_of(i, D, C); }), red, rp ^= 1);
      ++ph;
    }
  }
  // the residual stream after the last layer, for the head GEMV
  if (rank == 0)
    for (int i = t; i < D; i += kThreads) p.x_out[(int64_t)b * D + i] = live ? x[i] : 0.f;
  if (timed_out && p.err) atomicOr(p.err, kErrTimeout);
  cl.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace cstep
}  // namespace qd

// ---------------------------------------------------------------------------------------
// Host side: plan (cluster size, work split, shared-memory layout) and launch.
// ---------------------------------------------------------------------------------------
namespace qd {

namespace {

// Largest bytes of one CTA's slice (codes, 16-aligned, then the 16-widened scale range)
// of rows [r0, r1) over the C CTAs, rows taken `pair` at a time.
uint32_t max_slice_bytes(int64_t units_total, int pair, int C, int64_t rcb, int64_t rsb) {
  uint32_t best = 0;
  for (int r = 0; r < C; ++r) {
    const int64_t a = (int64_t)r * units_total / C * pair, b = (int64_t)(r + 1) * units_total / C * pair;
    const int64_t cb = align16u((b - a) * rcb);
    const int64_t s0 = (a * rsb) & ~(int64_t)15, s1 = (b * rsb + 15) & ~(int64_t)15;
    const int64_t tot = cb + (s1 - s0);
    if (tot > (int64_t)best) best = (uint32_t)tot;
  }
  return best;
}

uint32_t up128(size_t v) { return (uint32_t)((v + 127) & ~(size_t)127); }

// The kernel's dynamic shared-memory limit is raised to the device's opt-in maximum (not
// to one model's need, so models planned later never lower it under an earlier model's
// captured launches).
template <int FMT>
bool cluster_fits(int C, size_t smem, int optin) {
  auto kern = cstep::k_step_cluster<FMT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C);
  cfg.blockDim = dim3(cstep::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = (unsigned)C;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return n >= 1;
}

}  // namespace

bool step_cluster_plan(const StepClusterModel& m, StepClusterPlan* plan) {
  using cstep::kHd;
  if (m.fmt != QD_Q4_0 && m.fmt != QD_Q8_0) return false;
  if (m.n_heads % m.n_kv || m.n_heads / m.n_kv > 8) return false;
  const int QD = m.n_heads * kHd, KD = m.n_kv * kHd, G = m.n_heads / m.n_kv;
  if (m.D % 32 || m.F % 32 || m.D < 32 || m.F < 32) return false;
  // a lane holds the records of at most two units of a product's input
  if (m.D > 64 * 32 || m.F > 64 * 32 || QD > 64 * 32) return false;
  if ((QD + 2 * KD) % 2) return false;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  const int64_t rcb_d = row_code_bytes(m.fmt, m.D), rsb_d = row_scale_bytes(m.fmt, m.D);
  const int64_t rcb_q = row_code_bytes(m.fmt, QD), rsb_q = row_scale_bytes(m.fmt, QD);
  const int64_t rcb_f = row_code_bytes(m.fmt, m.F), rsb_f = row_scale_bytes(m.fmt, m.F);
  for (int C : {16, 8}) {
    if (m.n_kv > C) continue;
    const int S = C / m.n_kv;
    const int kvp = (m.max_ctx + S - 1) / S;
    const int U = m.n_kv * S;
    const int R = QD + 2 * KD;
    int nmax = std::max(std::max(R, m.F), std::max(m.D, U * G * cstep::kPart));
    nmax = std::max(nmax, QD);
    uint32_t wb = 0;
    const uint32_t gains = (uint32_t)m.D * 4;  // the QKV and gate/up slices bring their norm gains
    wb = std::max(wb, max_slice_bytes(R / 2, 2, C, rcb_d, rsb_d) + gains);  // QKV pairs
    wb = std::max(wb, max_slice_bytes(m.D, 1, C, rcb_q, rsb_q));            // Wo rows
    wb = std::max(wb, max_slice_bytes(m.F, 2, C, rcb_d, rsb_d) + gains);    // gate/up pairs
    wb = std::max(wb, max_slice_bytes(m.D, 1, C, rcb_f, rsb_f));            // down rows
    wb = up128(wb);
    StepClusterPlan pl{};
    pl.C = C;
    pl.S = S;
    pl.kvp = kvp;
    pl.nmax = nmax;
    pl.wbuf_bytes = wb;
    uint32_t off = 0;
    pl.off_wbuf = off;  off += 2 * wb;
    pl.off_kv = off;    off += up128((size_t)2 * kvp * kHd * 4);
    pl.off_slot = off;  off += up128((size_t)2 * nmax * 4);
    pl.off_x = off;     off += up128((size_t)m.D * 4);
    pl.off_v = off;     off += up128((size_t)nmax * 4);
    pl.off_rec = off;   off += up128((size_t)(std::max(std::max(m.D, QD), m.F) / 32) * intdot::kRecBytes);
    pl.off_sc = off;    off += up128((size_t)G * kvp * 4);
    pl.off_misc = off;  off += 128 * 4;  // RoPE row, reductions
    pl.off_bar = off;   off += 128;
    pl.smem = off;
    if ((int)off > optin) continue;
    const bool ok = m.fmt == QD_Q4_0 ? cluster_fits<QD_Q4_0>(C, off, optin) : cluster_fits<QD_Q8_0>(C, off, optin);
    if (!ok) continue;
    *plan = pl;
    return true;
  }
  return false;
}

qd_status launch_step_cluster(const StepClusterModel& m, const StepClusterPlan& pl, const int32_t* tok,
                              const int32_t* pos, float* x_out, uint32_t* err, int batch, cudaStream_t stream) {
  using cstep::kHd;
  cstep::Params p{};
  const int QD = m.n_heads * kHd, KD = m.n_kv * kHd;
  auto mat = [&](int64_t off, int64_t rows, int64_t cols) {
    cstep::Mat r;
    r.codes = off;
    r.scales = off + (int64_t)packed_code_region(m.fmt, rows, cols);
    r.rcb = (int32_t)row_code_bytes(m.fmt, cols);
    r.rsb = (int32_t)row_scale_bytes(m.fmt, cols);
    return r;
  };
  p.w = m.w;
  p.layer0 = m.layer0;
  p.layer_stride = m.layer_stride;
  p.off_attn_norm = m.off_attn_norm;
  p.off_ffn_norm = m.off_ffn_norm;
  p.qkv = mat(m.off_qkv, QD + 2 * KD, m.D);
  p.wo = mat(m.off_wo, m.D, QD);
  p.gu = mat(m.off_gu, 2 * (int64_t)m.F, m.D);
  p.wd = mat(m.off_wd, m.D, m.F);
  p.emb = m.emb;
  p.emb_fmt = m.emb_fmt;
  p.layers = m.layers;
  p.D = m.D;
  p.F = m.F;
  p.QD = QD;
  p.KD = KD;
  p.G = m.n_heads / m.n_kv;
  p.n_kv = m.n_kv;
  p.max_ctx = m.max_ctx;
  p.pairing = m.pairing;
  p.vocab = m.vocab;
  p.eps = m.eps;
  p.tok = tok;
  p.pos = pos;
  p.kc = m.kc;
  p.vc = m.vc;
  p.cache_layer_stride = m.cache_layer_stride;
  p.cache_batch_stride = m.cache_batch_stride;
  p.rope = m.rope;
  p.x_out = x_out;
  p.err = err;
  p.S = pl.S;
  p.kvp = pl.kvp;
  p.nmax = pl.nmax;
  p.wbuf_bytes = pl.wbuf_bytes;
  p.off_wbuf = pl.off_wbuf;
  p.off_kv = pl.off_kv;
  p.off_slot = pl.off_slot;
  p.off_x = pl.off_x;
  p.off_v = pl.off_v;
  p.off_rec = pl.off_rec;
  p.off_sc = pl.off_sc;
  p.off_misc = pl.off_misc;
  p.off_bar = pl.off_bar;
  p.smem_bytes = pl.smem;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(batch * pl.C));
  cfg.blockDim = dim3(cstep::kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = (unsigned)pl.C;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (m.fmt == QD_Q4_0)
    e = cudaLaunchKernelEx(&cfg, cstep::k_step_cluster<QD_Q4_0>, p);
  else
    e = cudaLaunchKernelEx(&cfg, cstep::k_step_cluster<QD_Q8_0>, p);
  return e == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

}  // namespace qd
