// Streaming q_gemv for batch 1-8 on the CUDA cores.
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
//  * The dot products run on the integer pipe.  Once per CTA, each 32-element unit of
//    x * g is written as 24-bit integers xq with one power-of-two scale s, 2^-22 of the
//    unit's largest |x| rounded down to a power of two (error at most s/2 per element,
//    about the rounding of an f32; exact for dyadic x), held as three byte
//    planes (signed high, unsigned middle and low bytes) so that one dp4a multiplies
//    four codes with four bytes of a plane: sum q x = s * (65536 sum q x2 +
//    256 sum q x1 + sum q x0), each plane's sum exact in int32.  A 4-bit code word
//    needs one LOP3 (and a shift) per four codes, so a Q4_0 weight costs under 1.5
//    instructions instead of a float decode plus an FMA.  (Two planes, 16 bits, lost
//    up to 2e-5 of a unit's largest |x| per element: too much where a short row sum
//    cancels.)  With RMSNorm fused, 1/sqrt(mean(x^2) + eps) multiplies each finished
//    row sum.
//  * A warp reduces its RW x NB row sums with one reduce-scatter and writes them (or
//    feeds the fused epilogues: SwiGLU, RoPE + KV append, argmax).
#include "qd_intdot.cuh"

namespace qd {

namespace stream_gemv {

using namespace intdot;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

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
  int ksplit;  // CTAs per cluster sharing each row group, each over its own unit steps
  int maxk;    // row groups per warp at most (the partial-sum slots, ksplit > 1)
};

// Distributed shared memory (thread-block clusters): store v at this CTA's shared address
// `addr` as mapped into CTA `rank` of the cluster; and the cluster-wide barrier.
__device__ __forceinline__ void st_cluster(uint32_t addr, int rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// kGemvQKV: rows r (even) and r+1 of batch b hold a RoPE pair (q or k) or two
// consecutive v values; rotate and scatter them (see QkvEpilogue).
// The epilogue's own inputs for one writer lane of a group, loaded right after the
// dependency wait (or when the previous group ends) so their latency overlaps the
// prologue and the main loop: the old y (accumulate), the position and the RoPE
// (cos, sin) of the row pair (QKV).
struct EpiPrefetch {
  float y_old = 0.f;
  int pos = -1;
  float2 cs = make_float2(1.f, 0.f);
};

__device__ __forceinline__ void qkv_pair_out(const Params& p, int64_t r, int b, float a, float bb,
                                             const EpiPrefetch& pf) {
  const QkvEpilogue& e = p.qkv;
  const int pos = pf.pos;
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
    const float2 cs = pf.cs;
    const float o0 = a * cs.x - bb * cs.y, o1 = a * cs.y + bb * cs.x;
    if (isq) {
      float* dst = e.q_out + (int64_t)b * e.q_stride + h * hd;
      dst[d0] = o0;
      dst[d1] = o1;
    } else {
      const int64_t row = (int64_t)b * e.cache_batch_stride + (h * e.max_ctx + pos) * hd;
      cache_store(e.kc, e.kv_f16, row + d0, o0);
      cache_store(e.kc, e.kv_f16, row + d1, o1);
    }
  } else {
    const int64_t local = r - e.q_rows - e.k_rows;
    const int64_t h = local / hd;
    const int d = (int)(local % hd);
    const int64_t row = (int64_t)b * e.cache_batch_stride + (h * e.max_ctx + pos) * hd;
    cache_store(e.vc, e.kv_f16, row + d, a);
    cache_store(e.vc, e.kv_f16, row + d + 1, bb);
  }
}

// Prefetch for the writer lane of group g (lanes with lane % grp == 0 write value
// k = lane / grp: row g * RW + k / NB, batch row k % NB).
template <int NB, int RW>
__device__ __forceinline__ EpiPrefetch epi_prefetch(const Params& p, int64_t g, int lane) {
  constexpr int V = RW * NB, GRP = 32 / V;
  EpiPrefetch pf;
  const int kk = lane / GRP, rr = kk / NB, b = kk % NB;
  const int64_t r = g * RW + rr;
  if ((lane % GRP) != 0 || b >= p.batch || r >= p.W.rows) return pf;
  if (p.mode == kGemvAccumulate) {
    pf.y_old = __ldcg(p.y + (int64_t)b * p.W.rows + r);
  } else if (p.mode == kGemvQKV) {
    const QkvEpilogue& e = p.qkv;
    pf.pos = __ldcg(e.pos + b);
    if ((rr & 1) == 0 && r < e.q_rows + e.k_rows && pf.pos >= 0 && pf.pos < e.max_ctx) {
      const int64_t local = r < e.q_rows ? r : r - e.q_rows;
      const int pi = (int)(local % e.head_dim) / 2;
      pf.cs = __ldg(reinterpret_cast<const float2*>(e.rope + ((int64_t)pf.pos * (e.head_dim / 2) + pi) * 2));
    }
  }
  return pf;
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

// Per-warp staging ring in shared memory: stages<FMT, RW>() slots, one unit step each.
// A slot holds, for the RW rows of the group, every lane's code chunk (lane-major, so
// each lane reads back only what it copied) and then the scale data of each row: 64
// bytes (Q4_0/Q8_0 the 32 lanes' f16 scales, Q4_K the 4 super-block headers the 32 units
// span, INT8 / INT4 the row scale) or, for Q4_1, 128 (the 32 lanes' (d, m) pairs).
// Q6_K and Q5_K take their step's four super-blocks whole instead (Q6_K 768 bytes of ql
// and qh per row and 72 bytes of scale records; Q5_K 640 bytes of fifth bits and nibbles
// and 64 bytes of headers), the lanes of a super-block reading the bytes they share.
constexpr int kQ6Step = 4 * 192, kQ5KStep = 4 * 160;
template <int FMT>
constexpr bool whole_blocks() {
  return FMT == QD_Q6_K || FMT == QD_Q5_K;
}
template <int FMT, int RW>
constexpr int slot_code_bytes() {
  return FMT == QD_Q6_K ? RW * kQ6Step : FMT == QD_Q5_K ? RW * kQ5KStep : RW * 32 * code_bytes<FMT>();
}
// scale bytes per row of a slot: Q4_1 one (d, m) pair per lane's unit, Q5_0 one (d, qh)
// record (6 bytes) per lane's unit, Q6_K its 4 super-blocks' 18-byte records, the others 64
template <int FMT>
constexpr int slot_scale_bytes() {
  return FMT == QD_Q4_1 ? 128 : FMT == QD_Q5_0 ? 192 : FMT == QD_Q6_K ? 80 : 64;
}
template <int FMT, int RW>
constexpr int slot_bytes() {
  return slot_code_bytes<FMT, RW>() + RW * slot_scale_bytes<FMT>();
}
// Ring depth: every warp keeps about kInFlight bytes of codes in flight whatever the
// rows per group (HBM latency times bandwidth over the SMs' warps wants several KB per
// warp: a 4-stage ring of 512-byte single-row steps left the DRAM pipe half empty).
#ifndef QD_GEMV_INFLIGHT
#define QD_GEMV_INFLIGHT 8192
#endif
constexpr int kInFlight = QD_GEMV_INFLIGHT;
template <int FMT, int RW>
constexpr int stages() {
  constexpr int s = kInFlight / slot_code_bytes<FMT, RW>() + 1;
  return s < 4 ? 4 : (s > 16 ? 16 : s);
}

// Issue the copies of one unit step (unit u of the rows in rp) into the slot at `slot`.
template <int FMT, int RW>
__device__ __forceinline__ void stage_step(uint32_t slot, const RowPtrs<RW>& rp, int u, int lane, int units) {
  constexpr int CB = code_bytes<FMT>();
  if constexpr (whole_blocks<FMT>()) {
    // the step's super-blocks, chunk c of their codes by lane c and c - 32; Q6_K's scale
    // records (an even number of super-blocks a row: whole words) word w by lane w, Q5_K's
    // 16-byte headers header k by lane k
    constexpr int kBlk = FMT == QD_Q6_K ? 192 : 160, kStep = 4 * kBlk;
    const int sb0 = (u - lane) >> 3, nsb = min(4, units / 8 - sb0);
#pragma unroll
    for (int rr = 0; rr < RW; ++rr) {
      const uint8_t* c = rp.c[rr] + (uint32_t)sb0 * (uint32_t)kBlk;
      const uint32_t dst = slot + (uint32_t)(rr * kStep);
      const int chunks = nsb * kBlk / 16;
      if (lane < chunks) cp16(dst + 16 * lane, c + 16 * lane);
      if (lane + 32 < chunks) cp16(dst + 16 * (lane + 32), c + 16 * (lane + 32));
      const uint32_t sdst = slot + slot_code_bytes<FMT, RW>() + rr * slot_scale_bytes<FMT>();
      if constexpr (FMT == QD_Q6_K) {
        if (lane < nsb * 18 / 4) cp4(sdst + 4 * lane, rp.s[rr] + (uint32_t)sb0 * 18u + 4 * lane);
      } else {
        if (lane < nsb) cp16(sdst + 16 * lane, rp.s[rr] + (uint32_t)(sb0 + lane) * 16u);
      }
    }
  } else {
#pragma unroll
    for (int rr = 0; rr < RW; ++rr) {
      const uint32_t dst = slot + (uint32_t)(rr * 32 + lane) * CB;
      const uint8_t* c = rp.c[rr] + (uint32_t)u * (uint32_t)CB;
#pragma unroll
      for (int k = 0; k < CB / 16; ++k) cp16(dst + 16 * k, c + 16 * k);
      const uint32_t sdst = slot + slot_code_bytes<FMT, RW>() + rr * slot_scale_bytes<FMT>();
      if constexpr (FMT == QD_Q4_1) {
        cp4(sdst + 4 * lane, rp.s[rr] + 4 * (uint32_t)u);  // (d, m) of this lane's unit
      } else if constexpr (FMT == QD_Q4_0 || FMT == QD_Q8_0) {
        if ((lane & 1) == 0) cp4(sdst + 2 * lane, rp.s[rr] + 2 * (uint32_t)u);  // d of units u, u+1
      } else if constexpr (FMT == QD_Q5_0) {
        if ((lane & 1) == 0) {  // (d, qh) of units u, u+1: 12 bytes
#pragma unroll
          for (int k = 0; k < 3; ++k) cp4(sdst + 6 * lane + 4 * k, rp.s[rr] + 6 * (uint32_t)u + 4 * k);
        }
      } else if constexpr (FMT == QD_Q4_K) {
        if ((lane & 7) == 0) cp16(sdst + 2 * lane, rp.s[rr] + (uint32_t)(u >> 3) * 16u);  // header
      } else {
        if (lane == 0) cp4(sdst, rp.s[rr]);  // row scale
      }
    }
  }
}

template <int NB, int RW>
struct Acc {
  float v[RW][NB];
};

// Compute one unit step (unit u of the RW rows staged in `slot`) into acc.
template <int FMT, int NB, int RW>
__device__ __forceinline__ void compute_step(Acc<NB, RW>& acc, const uint8_t* slot, const uint8_t* xq, int units,
                                             int u, int lane, int batch) {
  constexpr int CB = code_bytes<FMT>();
  const uint8_t* sc = slot + slot_code_bytes<FMT, RW>();
  if constexpr (FMT == QD_Q6_K) {
    // unit v = u % 8 of super-block u / 8 (the step's lsb-th): elements 32v..32v+31 take the
    // low (k < 2) or high nibbles of ql bytes 64h + 32(k & 1) + l and bits 2k, 2k+1 of qh
    // bytes 128 + 32h + l (h = v / 4, k = v % 4), as signed q - 32 (bytes: (q | 0x80) - 0x20
    // cannot borrow, then ^ 0x80); halves A, B are sub-blocks 8h + 2k and 8h + 2k + 1
    const int v = u & 7, h = v >> 2, k = v & 3, lsb = (u & 31) >> 3;
    const int sh = (k >> 1) * 4, hs = 2 * k;
    uint32_t w[RW][8];
    float c0[RW], c1[RW];
#pragma unroll
    for (int rr = 0; rr < RW; ++rr) {
      const uint8_t* blk = slot + rr * kQ6Step + lsb * 192;
      const uint4 l0 = *reinterpret_cast<const uint4*>(blk + 64 * h + 32 * (k & 1));
      const uint4 l1 = *reinterpret_cast<const uint4*>(blk + 64 * h + 32 * (k & 1) + 16);
      const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 128 + 32 * h);
      const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 128 + 32 * h + 16);
      const uint32_t lw[8] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w};
      const uint32_t hw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t q = ((lw[t] >> sh) & 0x0F0F0F0Fu) | (((hw[t] >> hs) & 0x03030303u) << 4);
        w[rr][t] = ((q | 0x80808080u) - 0x20202020u) ^ 0x80808080u;
      }
      const uint8_t* sr = sc + rr * slot_scale_bytes<FMT>() + lsb * 18;
      const float d = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sr + 16));
      c0[rr] = d * (float)(int8_t)sr[8 * h + 2 * k];
      c1[rr] = d * (float)(int8_t)sr[8 * h + 2 * k + 1];
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (NB > 1 && b >= batch) break;
      const uint8_t* rec = xq + ((size_t)b * units + u) * kRecBytes;
      const uint4 hA = *reinterpret_cast<const uint4*>(rec + 0), hB = *reinterpret_cast<const uint4*>(rec + 16);
      const uint4 mA = *reinterpret_cast<const uint4*>(rec + 32), mB = *reinterpret_cast<const uint4*>(rec + 48);
      const uint4 lA = *reinterpret_cast<const uint4*>(rec + 64), lB = *reinterpret_cast<const uint4*>(rec + 80);
      const float xs = *reinterpret_cast<const float*>(rec + 96);
#pragma unroll
      for (int rr = 0; rr < RW; ++rr) {
        const float va = planes_value(half_dot_s<true>(w[rr], hA, 0), half_dot_s<false>(w[rr], mA, 0),
                                      half_dot_s<false>(w[rr], lA, 0));
        const float vb = planes_value(half_dot_s<true>(w[rr] + 4, hB, 0), half_dot_s<false>(w[rr] + 4, mB, 0),
                                      half_dot_s<false>(w[rr] + 4, lB, 0));
        acc.v[rr][b] = fmaf(xs, fmaf(c0[rr], va, c1[rr] * vb), acc.v[rr][b]);
      }
    }
  } else {
    // codes: Q4_0 / Q4_K word t < 4 = low nibbles of code bytes 4t..4t+3 (half A),
    // t >= 4 = their high nibbles (half B); Q8_0 / INT8 the 32 code bytes in order
    uint32_t w[RW][8];
    float dq[RW], dm[RW];
    int s0[RW], s1[RW], m0[RW], m1[RW];
#pragma unroll
    for (int rr = 0; rr < RW; ++rr) {
      const uint8_t* cp = slot + (rr * 32 + lane) * CB;
      if constexpr (FMT == QD_Q4_0 || FMT == QD_Q4_K || FMT == QD_I4_ROW || FMT == QD_Q4_1) {
        const uint4 q = *reinterpret_cast<const uint4*>(cp);
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          w[rr][t] = wv[t] & 0x0F0F0F0Fu;
          w[rr][t + 4] = (wv[t] >> 4) & 0x0F0F0F0Fu;
        }
      } else if constexpr (FMT == QD_Q5_0) {
        // Q4_0's nibbles plus fifth bit j of qh for element j, spread to bit 4 of each byte
        // (x * 0x00204081 moves bit i of a 4-bit x to bit 8i, no carries), as signed q - 16
        const uint4 q = *reinterpret_cast<const uint4*>(cp);
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
        const unsigned short* rec = reinterpret_cast<const unsigned short*>(sc + rr * slot_scale_bytes<FMT>() + 6 * lane);
        const uint32_t qh = (uint32_t)rec[1] | ((uint32_t)rec[2] << 16);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t fa = (((qh >> (4 * t)) & 15u) * 0x00204081u) & 0x01010101u;
          const uint32_t fb = (((qh >> (16 + 4 * t)) & 15u) * 0x00204081u) & 0x01010101u;
          const uint32_t qa = (wv[t] & 0x0F0F0F0Fu) | (fa << 4), qb = ((wv[t] >> 4) & 0x0F0F0F0Fu) | (fb << 4);
          w[rr][t] = ((qa | 0x80808080u) - 0x10101010u) ^ 0x80808080u;
          w[rr][t + 4] = ((qb | 0x80808080u) - 0x10101010u) ^ 0x80808080u;
        }
      } else if constexpr (FMT == QD_Q5_K) {
        // Q4_K's nibbles plus the fifth bit: unsigned 5-bit codes through Q4_K's dot.  Unit
        // u = 8s + 2c + h of its 160-byte super-block (the step's lane / 8-th): nibbles at
        // 32 + 32c + 16h, fifth bits at 16h (bit 2c for the low nibbles, 2c + 1 the high)
        const uint8_t* blk = slot + rr * kQ5KStep + (lane >> 3) * 160;
        const uint4 q = *reinterpret_cast<const uint4*>(blk + 32 + 32 * ((u >> 1) & 3) + 16 * (u & 1));
        const uint4 hq = *reinterpret_cast<const uint4*>(blk + 16 * (u & 1));
        const uint32_t wv[4] = {q.x, q.y, q.z, q.w}, hv[4] = {hq.x, hq.y, hq.z, hq.w};
        const int b0 = 2 * ((u >> 1) & 3);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          w[rr][t] = (wv[t] & 0x0F0F0F0Fu) | (((hv[t] >> b0) & 0x01010101u) << 4);
          w[rr][t + 4] = ((wv[t] >> 4) & 0x0F0F0F0Fu) | (((hv[t] >> (b0 + 1)) & 0x01010101u) << 4);
        }
      } else {
        const uint4 q0 = *reinterpret_cast<const uint4*>(cp);
        const uint4 q1 = *reinterpret_cast<const uint4*>(cp + 16);
        w[rr][0] = q0.x; w[rr][1] = q0.y; w[rr][2] = q0.z; w[rr][3] = q0.w;
        w[rr][4] = q1.x; w[rr][5] = q1.y; w[rr][6] = q1.z; w[rr][7] = q1.w;
      }
      dm[rr] = 0.f;
      s0[rr] = s1[rr] = m0[rr] = m1[rr] = 0;
      if constexpr (FMT == QD_Q4_1) {
        const uint32_t dmv = *reinterpret_cast<const uint32_t*>(sc + rr * slot_scale_bytes<FMT>() + 4 * lane);
        dq[rr] = f16_bits_to_f32(dmv & 0xFFFFu);
        dm[rr] = f16_bits_to_f32(dmv >> 16);
      } else if constexpr (FMT == QD_Q4_0 || FMT == QD_Q8_0) {
        dq[rr] = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sc + rr * 64 + 2 * lane));
      } else if constexpr (FMT == QD_Q5_0) {
        dq[rr] = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sc + rr * slot_scale_bytes<FMT>() + 6 * lane));
      } else if constexpr (FMT == QD_Q4_K || FMT == QD_Q5_K) {
        const uint4 hdr = *reinterpret_cast<const uint4*>(sc + rr * 64 + (lane >> 3) * 16);
        const int j0 = 2 * ((u >> 1) & 3);
        q4k_sm_words(hdr.y, hdr.z, hdr.w, j0, s0[rr], m0[rr]);
        q4k_sm_words(hdr.y, hdr.z, hdr.w, j0 + 1, s1[rr], m1[rr]);
        dq[rr] = f16_bits_to_f32(hdr.x & 0xFFFFu);
        dm[rr] = f16_bits_to_f32(hdr.x >> 16);
      } else {
        dq[rr] = 1.f;  // INT8 / INT4 rows: the row scale multiplies the finished row sum
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (NB > 1 && b >= batch) break;
      const uint8_t* rec = xq + ((size_t)b * units + u) * kRecBytes;
      const uint4 hA = *reinterpret_cast<const uint4*>(rec + 0), hB = *reinterpret_cast<const uint4*>(rec + 16);
      const uint4 mA = *reinterpret_cast<const uint4*>(rec + 32), mB = *reinterpret_cast<const uint4*>(rec + 48);
      const uint4 lA = *reinterpret_cast<const uint4*>(rec + 64), lB = *reinterpret_cast<const uint4*>(rec + 80);
      const float4 mt = *reinterpret_cast<const float4*>(rec + 96);
#pragma unroll
      for (int rr = 0; rr < RW; ++rr) {
        if constexpr (FMT == QD_Q4_0 || FMT == QD_I4_ROW) {
          // planes start at -8 * their element sums: sum (q - 8) xq, plane by plane (INT4
          // rows are packed as Q4_0 codes in offset binary, q + 8)
          const int h = plane_dot<false, true>(w[rr], hA, hB, __float_as_int(mt.y));
          const int m = plane_dot<false, false>(w[rr], mA, mB, __float_as_int(mt.z));
          const int l = plane_dot<false, false>(w[rr], lA, lB, __float_as_int(mt.w));
          acc.v[rr][b] = fmaf(dq[rr] * mt.x, planes_value(h, m, l), acc.v[rr][b]);
        } else if constexpr (FMT == QD_Q4_1) {
          // value d q + m: d sum q xq (plane by plane) + m sum x (the record's half sums)
          const int h = plane_dot<false, true>(w[rr], hA, hB, 0);
          const int m = plane_dot<false, false>(w[rr], mA, mB, 0);
          const int l = plane_dot<false, false>(w[rr], lA, lB, 0);
          acc.v[rr][b] = fmaf(dq[rr] * mt.x, planes_value(h, m, l), fmaf(dm[rr], mt.y + mt.z, acc.v[rr][b]));
        } else if constexpr (FMT == QD_Q4_K || FMT == QD_Q5_K) {
          // value d sc q - dmin m, summed over halves A (sub-block 2c) and B (2c + 1)
          const float va = planes_value(half_dot<true>(w[rr], hA, 0), half_dot<false>(w[rr], mA, 0),
                                        half_dot<false>(w[rr], lA, 0));
          const float vb = planes_value(half_dot<true>(w[rr] + 4, hB, 0), half_dot<false>(w[rr] + 4, mB, 0),
                                        half_dot<false>(w[rr] + 4, lB, 0));
          const float q = fmaf((float)s0[rr], va, (float)s1[rr] * vb);
          const float mins = fmaf((float)m0[rr], mt.y, (float)m1[rr] * mt.z);
          acc.v[rr][b] = fmaf(dq[rr] * mt.x, q, fmaf(-dm[rr], mins, acc.v[rr][b]));
        } else {
          const int h = plane_dot<true, true>(w[rr], hA, hB, 0);
          const int m = plane_dot<true, false>(w[rr], mA, mB, 0);
          const int l = plane_dot<true, false>(w[rr], lA, lB, 0);
          acc.v[rr][b] = fmaf(dq[rr] * mt.x, planes_value(h, m, l), acc.v[rr][b]);
        }
      }
    }
  }
}

template <int FMT, int NB, int RW, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1) k_gemv_warp(const Params p) {
  // dynamic shared memory: [warps][stages] ring slots, then the x records [NB][units]
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float red[kWarps][NB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PackedView& W = p.W;
  const int cols = (int)W.cols;
  const int units = cols / 32;
  const int64_t groups = (W.rows + RW - 1) / RW;
  // Split-K over a cluster of C CTAs: each takes the same row groups over its own
  // contiguous unit steps [j0, j1) (and builds only those units' x records); the partial
  // row sums meet in the first CTA, which adds them in CTA order and writes the rows.
  // (a kernel that can split carries cluster instructions, which measured ~0.3 us slower to
  // launch even at C = 1: the split is a separate instantiation)
  const int C = SPLIT ? p.ksplit : 1;
  const int rank = C > 1 ? (int)(blockIdx.x % C) : 0;
  const int64_t ncl = gridDim.x / C, cid = blockIdx.x / C;
  const int steps_all = (units + 31) / 32;  // unit steps per row group
  const int j0 = rank * steps_all / C, j1 = (rank + 1) * steps_all / C;
  const int ua = 32 * j0, ub = min(32 * j1, units);  // this CTA's units
  if constexpr (SPLIT) cluster_arrive_relaxed();  // every CTA of the cluster has started (waited below)
  // Global warp ids interleave the clusters (warp-major), so the groups left over after
  // an even split land on warps spread over every SM rather than on the first ones.
  const int64_t gw = (int64_t)warp * ncl + cid, nw = ncl * kWarps;
  constexpr uint32_t SB = slot_bytes<FMT, RW>();
  constexpr int kStages = stages<FMT, RW>();
  uint8_t* ring = smem + (size_t)warp * kStages * SB;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  uint8_t* xq = smem + (size_t)kWarps * kStages * SB;

  // ---- start streaming the first steps (weights never depend on the previous kernel)
  int64_t lg = gw;  // group of the next copy
  int lj = j0;      // its unit step
  RowPtrs<RW> lrp;
  if (lg < groups) row_ptrs<RW>(lrp, W, lg * RW);
  auto issue = [&](int slot_idx) {
    if (lg < groups) {
      const int u = lane + 32 * lj;
      // (Q6_K: copies by chunk, not by unit, so every lane takes part in a short last step)
      if (u < units || whole_blocks<FMT>()) stage_step<FMT, RW>(ring_s + (uint32_t)slot_idx * SB, lrp, u, lane, units);
      if (++lj == j1) {
        lj = j0;
        lg += nw;
        if (lg < groups) row_ptrs<RW>(lrp, W, lg * RW);
      }
    }
    cp_commit();
  };
  // One stage before the dependency wait (for the decode step's small products that is
  // all of a warp's weights); the rest after x's first loads, which would otherwise queue
  // behind the whole ring's copies (measured: ~2.5 us of prologue at 14336x4096 Q8_0).
  issue(0);

  pdl_wait();  // x is the previous kernel's output
  EpiPrefetch pf;
  if (gw < groups) pf = epi_prefetch<NB, RW>(p, gw, lane);

  // ---- x * g as 24-bit integer records (see the header comment).  Eight lanes build
  // one unit: lane k < 4 takes elements 4k..4k+3 of half A, lane k >= 4 those of half
  // B.  RMSNorm's 1/sqrt(mean(x^2) + eps) multiplies the finished row sums instead, so
  // one barrier suffices.
  float inv[NB];
  {
    const int k = lane & 7;
    constexpr int kPass = kWarps * 4;  // units per pass of the CTA
    constexpr int kBatch = 4;          // passes of a warp whose loads are issued together
    auto load = [&](int b, int u, float4& v, float4& g) {
      const bool ok = u < ub;
      const int e = k < 4 ? unit_xa<FMT>(u) + 4 * k : unit_xb<FMT>(u) + 4 * (k - 4);
      const float* xr = p.x + (int64_t)b * cols;
      v = ok ? __ldcg(reinterpret_cast<const float4*>(xr + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
      g = ok && p.norm_g ? __ldg(reinterpret_cast<const float4*>(p.norm_g + e)) : make_float4(1.f, 1.f, 1.f, 1.f);
    };
    // this warp's first passes of batch row 0, loaded before the rest of the ring is issued
    float4 v0[kBatch], g0[kBatch];
#pragma unroll
    for (int t = 0; t < kBatch; ++t) load(0, ua + warp * 4 + t * kPass + (lane >> 3), v0[t], g0[t]);
#pragma unroll
    for (int s = 1; s < kStages - 1; ++s) issue(s);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float ss = 0.f;
      if (b < p.batch) {
        // one unit record from this lane's 4 elements v (gains g)
        auto record = [&](int u, bool ok, float4 v, float4 g) {
          if (p.norm_g) {
            ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
            v = make_float4(v.x * g.x, v.y * g.y, v.z * g.z, v.w * g.w);
          }
          intdot::write_record<FMT>(xq + ((size_t)b * units + u) * kRecBytes, k, ok, v);
        };
        for (int ub0 = ua + warp * 4; ub0 < ub; ub0 += kBatch * kPass) {  // uniform per warp
          float4 vv[kBatch], gg[kBatch];
          if (b == 0 && ub0 == ua + warp * 4) {
#pragma unroll
            for (int t = 0; t < kBatch; ++t) {
              vv[t] = v0[t];
              gg[t] = g0[t];
            }
          } else {
#pragma unroll
            for (int t = 0; t < kBatch; ++t) load(b, ub0 + t * kPass + (lane >> 3), vv[t], gg[t]);
          }
#pragma unroll
          for (int t = 0; t < kBatch; ++t) {
            if (ub0 + t * kPass >= ub) break;  // uniform per warp
            const int u = ub0 + t * kPass + (lane >> 3);
            record(u, u < ub, vv[t], gg[t]);
          }
        }
      }
      if (p.norm_g) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp][b] = ss;
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
  unsigned long long best[NB];  // kGemvArgmax: best (value, index) key per batch row
#pragma unroll
  for (int b = 0; b < NB; ++b) best[b] = 0ull;
  Acc<NB, RW> acc;
  constexpr int V = RW * NB, GRP = 32 / V;
  static_assert(V <= 32, "one reduce-scatter per group");
  // split-K partial sums, in the first CTA of the cluster: [rank][warp][maxk][V]
  float* part = reinterpret_cast<float*>(xq + (size_t)NB * units * kRecBytes);
  const uint32_t part_s = (uint32_t)__cvta_generic_to_shared(part);
  // Write (or, split, hand over) the V row sums of a finished group: lanes with
  // lane % GRP == 0 write value kk = lane / GRP (row row0 + kk / NB, batch row kk % NB);
  // `partner` is the next row's value (same batch row) for the pair epilogues.
  auto emit = [&](int64_t row0, float tot, float partner, const EpiPrefetch& pf_) {
    if ((lane % GRP) != 0) return;
    const int kk = lane / GRP, rr = kk / NB, b = kk % NB;
    const int64_t r = row0 + rr;
    if (b >= p.batch || r >= W.rows) return;
    if (p.mode == kGemvSwiGLU) {
      if ((rr & 1) == 0 && r + 1 < W.rows) p.y[(int64_t)b * (W.rows / 2) + r / 2] = tot / (1.0f + expf(-tot)) * partner;
    } else if (p.mode == kGemvQKV) {
      if ((rr & 1) == 0 && r + 1 < W.rows) qkv_pair_out(p, r, b, tot, partner, pf_);
    } else {
      if (p.mode == kGemvArgmax) {
        const unsigned long long key = argmax_key(tot, (uint32_t)r);
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
          if (bb == b) best[bb] = key > best[bb] ? key : best[bb];
      }
      float* dst = p.y + (int64_t)b * W.rows + r;
      *dst = p.mode == kGemvAccumulate ? pf_.y_old + tot : tot;
    }
  };
  if constexpr (SPLIT) cluster_wait();  // the partial-sum slots of the first CTA exist from here on
  int cs = 0;  // slot of the step being computed
  int j = j0;
  int kg = 0;  // this warp's finished groups
  for (int64_t g = gw; g < groups;) {
    __syncwarp();  // every lane is done with the slot about to be refilled
    issue(cs == 0 ? kStages - 1 : cs - 1);
    cp_wait<kStages - 1>();  // this step's group of copies has landed
    __syncwarp();            // ...for every lane (scales are shared across lanes)
    if (j == j0) {
#pragma unroll
      for (int rr = 0; rr < RW; ++rr)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc.v[rr][b] = 0.f;
    }
    const int u = lane + 32 * j;
    const uint8_t* slot = ring + (size_t)cs * SB;
    if (u < units) compute_step<FMT, NB, RW>(acc, slot, xq, units, u, lane, p.batch);
    float rsc[RW];  // INT8 / INT4 row scales (staged with every step)
    if constexpr (FMT == QD_I8_ROW || FMT == QD_I4_ROW) {
#pragma unroll
      for (int rr = 0; rr < RW; ++rr) rsc[rr] = *reinterpret_cast<const float*>(slot + slot_code_bytes<FMT, RW>() + rr * 64);
    }
    cs = (cs + 1 == kStages) ? 0 : cs + 1;
    if (++j < j1) continue;
    j = j0;

    // ---- end of a group: reduce and write its RW rows
    const int64_t row0 = g * RW;
    if constexpr (FMT == QD_I8_ROW || FMT == QD_I4_ROW) {
#pragma unroll
      for (int rr = 0; rr < RW; ++rr)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc.v[rr][b] *= rsc[rr];
    }
    float v[V];
#pragma unroll
    for (int rr = 0; rr < RW; ++rr)
#pragma unroll
      for (int b = 0; b < NB; ++b) v[rr * NB + b] = acc.v[rr][b];
    const int kb = (lane / GRP) % NB;  // batch row of this lane's reduced value
    float iv = inv[0];
#pragma unroll
    for (int b = 1; b < NB; ++b) iv = kb == b ? inv[b] : iv;
    const float tot = reduce_scatter<V>(v, lane) * iv;
    if constexpr (SPLIT) {
      // this CTA's part of the group, to slot [rank][warp][kg] of the first CTA
      if ((lane % GRP) == 0)
        st_cluster(part_s + 4u * (uint32_t)(((rank * kWarps + warp) * p.maxk + kg) * V + lane / GRP), 0, tot);
      ++kg;
      g += nw;
      continue;
    }
    const float partner = __shfl_down_sync(0xffffffffu, tot, (NB * GRP) & 31);  // row +1, same batch
    emit(row0, tot, partner, pf);
    g += nw;
    if (g < groups) pf = epi_prefetch<NB, RW>(p, g, lane);
  }
  if constexpr (SPLIT) {
    // every part has landed in the first CTA, which adds them in CTA order and writes
    cp_wait<0>();
    cluster_arrive();
    cluster_wait();
    if (rank == 0) {
      int k = 0;
      for (int64_t g = gw; g < groups; g += nw, ++k) {
        const EpiPrefetch pf2 = epi_prefetch<NB, RW>(p, g, lane);
        float tot = 0.f;
        for (int r = 0; r < C; ++r) tot += part[((r * kWarps + warp) * p.maxk + k) * V + lane / GRP];
        const float partner = __shfl_down_sync(0xffffffffu, tot, (NB * GRP) & 31);
        emit(g * RW, tot, partner, pf2);
      }
    }
  }
  cp_wait<0>();  // no copy may still target this CTA's shared memory at exit
  if (p.mode == kGemvArgmax) {
    // warp max of the keys, one atomicMax per warp; after a CTA barrier one thread
    // publishes the CTA's arrival (release) and the last CTA to arrive (acquire)
    // finalises the tokens and re-arms the keys and the counter
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      unsigned long long k = best[b];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, off);
        k = o > k ? o : k;
      }
      if (lane == 0 && k != 0 && b < p.batch) atomicMax(p.am.key + b, k);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int old;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.am.counter) : "memory");
      if (old == gridDim.x - 1) {
        for (int b = 0; b < p.batch; ++b) {
          const unsigned long long k = atomicExch(p.am.key + b, 0ull);
          p.am.tok_out[b] = (int32_t)argmax_key_index(k);
          p.am.pos[b] += 1;
        }
        *p.am.counter = 0u;
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

// Resident CTAs per SM for a kernel at a dynamic shared-memory size (cached per
// kernel, size and device).
template <typename K>
int resident_ctas(K kern, size_t smem) {
  struct Entry {
    const void* fn;
    size_t smem;
    int dev, ctas;
  };
  static Entry cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const void* fn = reinterpret_cast<const void*>(kern);
  for (const Entry& e : cache)
    if (e.fn == fn && e.smem == smem && e.dev == dev) return e.ctas;
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kThreads, smem) != cudaSuccess || o < 1) o = 1;
  for (Entry& e : cache)
    if (!e.fn) {
      e = Entry{fn, smem, dev, o};
      break;
    }
  return o;
}

template <int FMT, int NB, int RW>
size_t smem_bytes_t(int64_t cols, int ksplit = 1, int maxk = 0) {
  const size_t units = (size_t)cols / 32;
  const size_t part = ksplit > 1 ? (size_t)ksplit * kWarps * maxk * RW * NB * 4 : 0;
  return (size_t)kWarps * stages<FMT, RW>() * slot_bytes<FMT, RW>() + (size_t)NB * units * kRecBytes + part;
}

// Rows per group available for NB batch rows (more rows would spill registers).
template <int NB>
constexpr int max_rw() {
  return 4;
}
template <int NB>
constexpr int min_rw() {
  return NB == 1 ? 1 : 2;
}

// Shared-memory need of the smallest-footprint RW for NB batch rows.
size_t smem_bytes(int fmt, int64_t cols, int nb) {
  switch (fmt) {
#define QD_SMEM_CASE(F)                                      \
  case F:                                                    \
    switch (nb) {                                            \
      case 1: return smem_bytes_t<F, 1, min_rw<1>()>(cols);  \
      case 2: return smem_bytes_t<F, 2, min_rw<2>()>(cols);  \
      case 4: return smem_bytes_t<F, 4, min_rw<4>()>(cols);  \
      default: return smem_bytes_t<F, 8, min_rw<8>()>(cols); \
    }
    QD_SMEM_CASE(QD_Q4_0)
    QD_SMEM_CASE(QD_Q8_0)
    QD_SMEM_CASE(QD_Q4_K)
    QD_SMEM_CASE(QD_I8_ROW)
    QD_SMEM_CASE(QD_I4_ROW)
    QD_SMEM_CASE(QD_Q4_1)
    QD_SMEM_CASE(QD_Q5_0)
    QD_SMEM_CASE(QD_Q5_K)
    QD_SMEM_CASE(QD_Q6_K)
#undef QD_SMEM_CASE
    default: return ~(size_t)0;
  }
}

constexpr size_t kSmemCap = 200 * 1024;

// The formats and batch widths that have a split-K instantiation (the split runs where it
// measured faster: batch 1-2; the tensor-core kernel takes these formats at batch 3-16).
template <int FMT, int NB>
constexpr bool split_built() {
  return NB <= 2 && (FMT == QD_Q4_0 || FMT == QD_Q8_0 || FMT == QD_I8_ROW || FMT == QD_Q4_K);
}

// Raise the kernel's dynamic shared-memory limit to kSmemCap once per device; the
// occupancy query and the launch both depend on it.
template <int FMT, int NB, int RW, bool SPLIT = false>
bool smem_attr_set() {
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(k_gemv_warp<FMT, NB, RW, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemCap) != cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

template <int FMT, int NB, int RW>
qd_status launch_rw(const Params& p, bool pdl, cudaStream_t stream, int64_t ctas) {
  auto kern = k_gemv_warp<FMT, NB, RW, false>;
  if constexpr (split_built<FMT, NB>()) {
    if (p.ksplit > 1) {
      if (!smem_attr_set<FMT, NB, RW, true>()) return QD_ERR_CUDA;
      kern = k_gemv_warp<FMT, NB, RW, true>;
    }
  }
  if (p.ksplit > 1 && !split_built<FMT, NB>()) return QD_ERR_UNSUPPORTED;
  const size_t smem = smem_bytes_t<FMT, NB, RW>(p.W.cols, p.ksplit, p.maxk);
  if (smem > kSmemCap) return QD_ERR_UNSUPPORTED;
  if (!smem_attr_set<FMT, NB, RW>()) return QD_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.ksplit > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)p.ksplit;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();
    return QD_ERR_CUDA;
  }
  return QD_OK;
}

// At most kCtasPerSm CTAs per SM, one wave.  One CTA (8 warps) per SM measured as fast as
// two on the large shapes and faster on several (the streams already fill the DRAM
// queues), and it leaves room for the next kernel's CTAs to start their weight copies early.
#ifndef QD_GEMV_CTAS_PER_SM
#define QD_GEMV_CTAS_PER_SM 1
#endif
constexpr int kCtasPerSm = QD_GEMV_CTAS_PER_SM;

// Launch geometry of one candidate: rows per group, CTAs per cluster (split-K), CTAs and
// the partial-sum slots per warp.
struct Geometry {
  int rw = 0, ksplit = 1, maxk = 0;
  int64_t ctas = 0;
};

// CTAs for RW rows per group split over `ksplit` CTAs per cluster: one warp per group up to
// one wave of at most kCtasPerSm CTAs per SM, whole clusters (ctas 0 when the shared memory
// does not fit).
template <int FMT, int NB, int RW>
Geometry geometry_for(int64_t rows, int64_t cols, int ksplit) {
  Geometry gm;
  gm.rw = RW;
  gm.ksplit = ksplit;
  if (smem_bytes_t<FMT, NB, RW>(cols) > kSmemCap || !smem_attr_set<FMT, NB, RW>()) return gm;
  const int64_t groups = (rows + RW - 1) / RW;
  int per_sm = resident_ctas(k_gemv_warp<FMT, NB, RW, false>, smem_bytes_t<FMT, NB, RW>(cols));
  if (per_sm > kCtasPerSm) per_sm = kCtasPerSm;
  const int64_t cap_cl = (int64_t)sm_count() * per_sm / ksplit;
  int64_t cl = (groups + kWarps - 1) / kWarps;
  if (cl > cap_cl) cl = cap_cl;
  if (cl < 1) return gm;
  gm.maxk = ksplit > 1 ? (int)((groups + cl * kWarps - 1) / (cl * kWarps)) : 0;
  if (smem_bytes_t<FMT, NB, RW>(cols, ksplit, gm.maxk) > kSmemCap) return gm;
  gm.ctas = cl * ksplit;
  return gm;
}

// Split-K across CTAs (a cluster of two sharing each row group) for the tall-and-thin
// products where it measured faster: store and accumulate without the fused norm (whose
// sum of squares spans all columns), 1024 rows or more and at least twice as many
// columns, at batch 2 or more (4096x11008 Q4_0 at batch 2: 17.7 -> 16.5 us; 2048x8192
// INT8: 10.0 -> 9.1 us) or with 8-bit weights (Q8_0 4096x11008: 12.8 -> 12.5 us).  At
// batch 1 with 4-bit weights, on the small decode shapes (576x1536: 3.1 -> 3.3 us), and
// with clusters of four it measured slower: clusters wait for groups of free SMs while
// the previous kernel still holds them.
int choose_ksplit(const Params& p, int fmt, int nb) {
  if (p.norm_g || (p.mode != kGemvStore && p.mode != kGemvAccumulate)) return 1;
  const int64_t rows = p.W.rows, cols = p.W.cols;
  if (rows < 1024 || cols < 2 * rows) return 1;
  if (nb >= 2 || fmt == QD_Q8_0 || fmt == QD_I8_ROW) return 2;
  return 1;
}

// Rows per group: the choice whose groups split most evenly over the warps (the kernel
// lasts as long as its busiest warp), preferring more rows (more reuse of staged x); then
// the split over a cluster (choose_ksplit).
template <int FMT, int NB>
qd_status launch_inst(Params p, bool pdl, cudaStream_t stream) {
  const int64_t rows = p.W.rows, cols = p.W.cols;
  constexpr int kMax = max_rw<NB>(), kMin = min_rw<NB>();
  const bool pairs = p.mode == kGemvSwiGLU || p.mode == kGemvQKV;  // need even rows per group
  auto geo = [&](int rw, int ks) {
    Geometry g;
    if constexpr (kMax >= 4) {
      if (rw == 4) g = geometry_for<FMT, NB, 4>(rows, cols, ks);
    }
    if (rw == 2) g = geometry_for<FMT, NB, 2>(rows, cols, ks);
    if constexpr (kMin <= 1) {
      if (rw == 1) g = geometry_for<FMT, NB, 1>(rows, cols, ks);
    }
    return g;
  };
  double best = -1.0;
  Geometry bg;
  for (int rw : {4, 2, 1}) {
    if (rw > kMax || rw < kMin || (pairs && rw == 1)) continue;
    const Geometry g = geo(rw, 1);
    if (g.ctas <= 0) continue;
    const int64_t groups = (rows + rw - 1) / rw;
    const int64_t slots = g.ctas * kWarps;
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
      bg = g;
    }
  }
  if (bg.ctas <= 0) return QD_ERR_UNSUPPORTED;
  const int steps_all = (int)((cols / 32 + 31) / 32);
  const int ks = split_built<FMT, NB>() ? choose_ksplit(p, FMT, NB) : 1;
  if (ks > 1 && ks <= steps_all) {
    const Geometry g = geo(bg.rw, ks);
    if (g.ctas > 0) bg = g;
  }
  p.ksplit = bg.ksplit;
  p.maxk = bg.maxk;
  if constexpr (kMax >= 4) {
    if (bg.rw == 4) return launch_rw<FMT, NB, 4>(p, pdl, stream, bg.ctas);
  }
  if (bg.rw == 2) return launch_rw<FMT, NB, 2>(p, pdl, stream, bg.ctas);
  if constexpr (kMin <= 1) {
    if (bg.rw == 1) return launch_rw<FMT, NB, 1>(p, pdl, stream, bg.ctas);
  }
  return QD_ERR_UNSUPPORTED;
}

int nb_for(int batch) { return batch <= 1 ? 1 : batch <= 2 ? 2 : batch <= 4 ? 4 : 8; }

bool supported(const GemvArgs& a) {
  // + INT4 rows, Q4_1, Q5_0, Q5_K, Q6_K (an even number of super-blocks per row: 4-byte
  // scale copies)
  if (!model_fmt_ok(a.fmt) && a.fmt != QD_I4_ROW && a.fmt != QD_Q4_1 && a.fmt != QD_Q5_0 && a.fmt != QD_Q5_K &&
      a.fmt != QD_Q6_K)
    return false;
  if (a.fmt == QD_Q6_K && a.W.cols % 512) return false;
  if (a.batch < 1 || a.batch > 8 || a.W.cols % 32) return false;
  if (a.W.cols > (1 << 24)) return false;
  if (smem_bytes(a.fmt, a.W.cols, nb_for(a.batch)) > kSmemCap) return false;
  // 4-byte scale copies need an even number of blocks per row
  if ((a.fmt == QD_Q4_0 || a.fmt == QD_Q8_0 || a.fmt == QD_Q5_0) && ((a.W.cols / 32) & 1)) return false;
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
  p.ksplit = 1;
  p.maxk = 0;
  const int nb = nb_for(a.batch);
#define QD_NB_SWITCH(F)                                      \
  switch (nb) {                                              \
    case 1: return launch_inst<F, 1>(p, a.pdl, stream);      \
    case 2: return launch_inst<F, 2>(p, a.pdl, stream);      \
    case 4: return launch_inst<F, 4>(p, a.pdl, stream);      \
    default: return launch_inst<F, 8>(p, a.pdl, stream);     \
  }
  switch (a.fmt) {
    case QD_Q4_0: QD_NB_SWITCH(QD_Q4_0)
    case QD_Q8_0: QD_NB_SWITCH(QD_Q8_0)
    case QD_Q4_K: QD_NB_SWITCH(QD_Q4_K)
    case QD_I8_ROW: QD_NB_SWITCH(QD_I8_ROW)
    case QD_I4_ROW: QD_NB_SWITCH(QD_I4_ROW)
    case QD_Q4_1: QD_NB_SWITCH(QD_Q4_1)
    case QD_Q5_0: QD_NB_SWITCH(QD_Q5_0)
    case QD_Q5_K: QD_NB_SWITCH(QD_Q5_K)
    case QD_Q6_K: QD_NB_SWITCH(QD_Q6_K)
    default: return QD_ERR_UNSUPPORTED;
  }
#undef QD_NB_SWITCH
}

}  // namespace qd
