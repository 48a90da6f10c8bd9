// q_gemv for batch 3-16 on the tensor cores (mma.sync, f16 inputs, f32 accumulate).
//
// y[b][r] = sum_c deq(W)[r][c] * x[b][c] (llmoxide blog s1, s10; dasLLAMA 8.7.1.4 matmul)
// for a few batch rows is a skinny dense contraction, and on the CUDA cores its cost grows
// with every batch row (the streaming kernel spends 24 dp4a per 32 weights per batch row:
// 14336x4096 Q4_0 took 11 / 24 / 48 us at batch 1 / 4 / 8).  Here it runs on the tensor
// cores without giving up the f32-activation contract:
//
//  * Weight codes are exact in binary16 (Q4_0 q - 8 in [-8, 7], Q8_0 / INT8 codes in
//    [-127, 127]), turned into f16 pairs in registers with the exponent-bias trick (the
//    code in the mantissa of 1024, then a subtraction).
//  * x reaches shared memory by bulk copies (one per batch row, counted on an mbarrier),
//    off the load path that the weight ring fills.  Each stage of 256 elements of every
//    batch row is then scaled by a power of two s (its largest |x| rounded down to a power
//    of two, so |x / s| < 2) and split in place into two binary16 parts, hi = f16(x / s)
//    and lo = f16(x / s - hi): about 22 bits of x, relative error ~2^-22 of the stage's
//    largest value (the batch-16 tensor-core GEMV uses the same split).  Products of f16
//    values are exact and sum in f32.
//  * mma.sync.m16n8k16 multiplies a 16-row tile of one unit's codes by the hi and lo parts
//    of 8 batch columns, two K halves: four instructions per unit and block of 8 columns
//    (batch 9-16: two blocks sharing the unit's A fragments).  The order of the 32 elements along K is free as long as A and B agree:
//    lane t takes its A values from code word t (bytes 4t..4t+3) of each row, pairing
//    bytes (0, 2) and (1, 3), so one 32-bit load and a few bit operations make its
//    fragments, and x is staged in the same order.  A unit is one quantisation block, so
//    the block scale d multiplies its f32 sums into a stage accumulator, and the stage's
//    x scale multiplies that into the tile's (INT8 rows, one scale a row, need neither
//    until the epilogue).  (GB300's int8 tensor path is ~4x slower than f16 here: 150
//    against 590 TOPS measured for mma.sync.)
//  * Weights stream as in the streaming kernel: every warp owns 16-row tiles taken round-
//    robin over the grid's warps, and copies its stages (16 rows x 8 or 4 units of codes
//    and scales, rows padded so that the fragment loads hit distinct banks) with per-lane
//    cp.async into a ring in shared memory, no CTA barrier in the main loop; the ring's
//    first stages are issued before the dependency wait.  A CTA has 16 warps with 4-unit
//    stages where x leaves room for a ring three stages deep (more warps hide more of the
//    fragment-building latency), otherwise 8 warps with 8-unit stages.
//  * Rows of x wider than the shared memory holds (store and accumulate only) split over
//    a thread-block cluster of 2 or 4 CTAs where every warp group of the grid then takes
//    one tile: each CTA stages, converts and multiplies only its share of the columns,
//    the others store their tile sums into the first CTA's shared memory (distributed
//    shared memory), and after one cluster barrier the first CTA adds them in CTA order
//    and runs the epilogue.  Otherwise they run as several launches over column ranges,
//    the first storing and the rest accumulating.  Either way the sums follow one fixed
//    order.
//  * Epilogues: store, accumulate, SwiGLU over interleaved (gate, up) rows, the QKV
//    epilogue (RoPE pairs, cache append) and the fused argmax, as the streaming kernel.
#include "qd_intdot.cuh"
#include "qd_tc.cuh"

namespace qd {
namespace mma_gemv {

constexpr int kTileRows = 16;
constexpr int kXUnits = 8;  // units per x scale (one power of two per 256 columns and batch row)
constexpr int kXCols = kXUnits * 32;
// units (32 columns each) per ring stage of a CTA of W warps
template <int W>
__host__ __device__ constexpr int stage_units() {
  return W == 16 ? 4 : 8;
}
constexpr int kXPad = 64;  // bytes after each staged x row: rows 2j, 2j + 1 on disjoint banks

struct Params {
  PackedView W;  // the column range's codes and scales start at unit u0
  const float* x;
  float* y;
  const float* norm_g;
  float eps;
  int batch;
  int mode;
  uint32_t* err;
  QkvEpilogue qkv;
  ArgmaxEpilogue am;
  int64_t x_stride;  // floats between batch rows of x
  int u0;            // first unit (32 columns) of the range
  int units;         // units in the range
  int stages;        // ring depth (slots per warp), sized to the shared memory left
  int ks;            // warps that share one tile, each over a contiguous part of its columns
  int ksplit;        // CTAs per cluster splitting the columns (split launches; 1 otherwise)
  int pdepth;        // buffers of warp partial sums: 0 (ks = 1), 1 (every warp group takes
                     // one tile at most) or 2
  bool accumulate;   // a later column range: y += partial product (store mode's chunks)
};

template <int FMT>
constexpr int code_bytes() {
  return FMT == QD_Q4_0 ? 16 : 32;
}
// a ring slot: codes [16 rows][row stride] (SU units a row, padded by 16 bytes so that the
// 8 rows a fragment load touches fall on different banks), then f16 scales [16][SU]
template <int FMT, int SU>
constexpr int row_stride() {
  return SU * code_bytes<FMT>() + 16;
}
template <int FMT, int SU>
constexpr int scale_bytes() {
  return FMT == QD_I8_ROW ? 0 : kTileRows * SU * 2;
}
template <int FMT, int SU>
constexpr int slot_bytes() {
  return kTileRows * row_stride<FMT, SU>() + scale_bytes<FMT, SU>();
}
// batch columns: one or two blocks of 8 (the MMA's N); scale and norm arrays keep 16 a stage
constexpr int kMaxCols = 16;
__host__ __device__ constexpr int col_blocks(int batch) { return batch > 8 ? 2 : 1; }
// per-warp partial accumulators for the warps sharing a tile: `depth` tiles deep (two; one
// where every warp group takes one tile at most; none where warps do not share tiles)
__host__ __device__ constexpr size_t partial_bytes(int nc, int warps, int depth) {
  return (size_t)depth * warps * 32 * 4 * nc * 4;
}

// Shared-memory layout of one launch (byte offsets; every part 16-byte aligned).
struct Layout {
  size_t ring, xs, gs, sx, ssq, partial, bar, spl, total;
  int64_t x_row;  // bytes between staged batch rows
};
template <int FMT, int W>
__host__ __device__ inline Layout layout(int units, int batch, bool norm, int stages, size_t split_bytes = 0,
                                         int depth = 2) {
  Layout L;
  const int nxg = (units + kXUnits - 1) / kXUnits;
  L.x_row = (int64_t)units * 128 + kXPad;
  L.ring = 0;
  L.xs = L.ring + (size_t)W * stages * slot_bytes<FMT, stage_units<W>()>();
  L.gs = L.xs + (size_t)batch * L.x_row;
  L.sx = L.gs + (norm ? (size_t)units * 128 : 0);
  L.ssq = L.sx + (size_t)nxg * kMaxCols * 4;
  L.partial = L.ssq + (size_t)nxg * kMaxCols * 4;
  L.bar = L.partial + partial_bytes(col_blocks(batch), W, depth);
  L.spl = L.bar + 16;
  L.total = L.spl + split_bytes;
  return L;
}

// Split launches: a cluster of C CTAs shares each tile, CTA r over the 256-column x groups
// [r G / C, (r + 1) G / C) of the G in the range, so each stages and converts only its
// share of x.  The widest share in units (the shared-memory layout is sized for it):
__host__ __device__ inline int split_units_cap(int units, int c) {
  const int nxg = (units + kXUnits - 1) / kXUnits;
  const int cap = (nxg + c - 1) / c * kXUnits;
  return cap < units ? cap : units;
}
// the first CTA's slots for the other CTAs' tile sums: [C - 1][groups][32 lanes][NC][4]
__host__ __device__ constexpr size_t split_slot_bytes(int c, int groups, int nc) {
  return (size_t)(c - 1) * groups * 32 * nc * 16;
}

template <int N>
__device__ __forceinline__ void cp_wait_n() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// cp.async.wait_group with a run-time count (the ring depth minus one, 1..7)
__device__ __forceinline__ void cp_wait_dyn(int n) {
  switch (n) {
    case 1: cp_wait_n<1>(); break;
    case 2: cp_wait_n<2>(); break;
    case 3: cp_wait_n<3>(); break;
    case 4: cp_wait_n<4>(); break;
    case 5: cp_wait_n<5>(); break;
    case 6: cp_wait_n<6>(); break;
    default: cp_wait_n<7>(); break;
  }
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Thread-block clusters: store four floats at this CTA's shared address `addr` as mapped
// into CTA `rank` of the cluster, and the cluster-wide barrier's arrive / wait.
__device__ __forceinline__ void st_cluster4(uint32_t addr, int rank, float a, float b, float c, float d) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// D = A (16x16, row) * B (16x8, col) + D over binary16 into f32.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t w) { return *reinterpret_cast<const __half2*>(&w); }

// One Q4_0 code word (bytes 4t..4t+3 of a block: low nibbles are elements 4t..4t+3, high
// nibbles elements 16 + 4t..) as f16 pairs q - 8: k0 = elements (4t, 4t + 2), k0b =
// (4t + 1, 4t + 3); k1, k1b the same for the high nibbles.  A nibble in the low bits of
// 1024's mantissa gives 1024 + n; one in bits 4-7 gives 1024 + 16n, scaled by 1/16.
__device__ __forceinline__ void q4_word(uint32_t w, uint32_t& k0, uint32_t& k0b, uint32_t& k1, uint32_t& k1b) {
  const __half2 c1032 = __floats2half2_rn(1032.f, 1032.f);
  const __half2 s16 = __floats2half2_rn(0.0625f, 0.0625f), c72 = __floats2half2_rn(-72.f, -72.f);
  const uint32_t w8 = w >> 8;
  k0 = h2_bits(__hsub2(bits_h2((w & 0x000F000Fu) | 0x64006400u), c1032));
  k0b = h2_bits(__hsub2(bits_h2((w8 & 0x000F000Fu) | 0x64006400u), c1032));
  k1 = h2_bits(__hfma2(bits_h2((w & 0x00F000F0u) | 0x64006400u), s16, c72));
  k1b = h2_bits(__hfma2(bits_h2((w8 & 0x00F000F0u) | 0x64006400u), s16, c72));
}
// One word of signed byte codes (elements 4t..4t+3) as f16 pairs: k = (4t, 4t + 2), kb =
// (4t + 1, 4t + 3).  q ^ 0x80 is q + 128 in 0..255: 1024 + q + 128, minus 1152.
__device__ __forceinline__ void i8_word(uint32_t w, uint32_t& k, uint32_t& kb) {
  const __half2 c1152 = __floats2half2_rn(1152.f, 1152.f);
  const uint32_t u = w ^ 0x80808080u;
  k = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4240u)), c1152));
  kb = h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4341u)), c1152));
}

// 2^e for e in [-127, 127] (2^-127 is subnormal)
__device__ __forceinline__ float pow2i(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// The QKV epilogue for one (even row r, row r + 1) pair of batch row b: a RoPE pair of q
// or k (rotated; q to q_out, k to the cache at pos[b]) or two consecutive v values.
__device__ __forceinline__ void qkv_pair(const Params& p, int64_t r, int b, float a, float bb) {
  const QkvEpilogue& e = p.qkv;
  const int pos = __ldcg(e.pos + b);
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
    const float2 cs = __ldg(reinterpret_cast<const float2*>(e.rope + ((int64_t)pos * half + pi) * 2));
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

// One unit's A fragments: rows g, g + 8 of the 16-row tile (codes at `row0` and `row8` in
// the ring slot; a0 = K half 0, a1 = K half 1, each rows (g, g + 8) x pairs
// ((4t, 4t+2), (4t+1, 4t+3))).
template <int FMT>
__device__ __forceinline__ void unit_a(const uint8_t* row0, const uint8_t* row8, int t, uint32_t (&a0)[4],
                                       uint32_t (&a1)[4]) {
  if constexpr (FMT == QD_Q4_0) {
    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(row0 + 4 * t);
    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(row8 + 4 * t);
    q4_word(w0, a0[0], a0[2], a1[0], a1[2]);
    q4_word(w1, a0[1], a0[3], a1[1], a1[3]);
  } else {
    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(row0 + 4 * t);
    const uint32_t w1 = *reinterpret_cast<const uint32_t*>(row8 + 4 * t);
    const uint32_t x0 = *reinterpret_cast<const uint32_t*>(row0 + 16 + 4 * t);
    const uint32_t x1 = *reinterpret_cast<const uint32_t*>(row8 + 16 + 4 * t);
    i8_word(w0, a0[0], a0[2]);
    i8_word(w1, a0[1], a0[3]);
    i8_word(x0, a1[0], a1[2]);
    i8_word(x1, a1[1], a1[3]);
  }
}
// One unit's B fragments for column g of a block (x at `xu`): v0, v1 = the two K halves'
// (hi b0, hi b1, lo b0, lo b1).
__device__ __forceinline__ void unit_b(const uint8_t* xu, int t, uint4& v0, uint4& v1) {
  v0 = *reinterpret_cast<const uint4*>(xu + 16 * t);
  v1 = *reinterpret_cast<const uint4*>(xu + 64 + 16 * t);
}
// d += A x B over the unit's two K halves, two chains of two MMAs (lo parts first), added.
__device__ __forceinline__ void unit_mma(float (&d)[4], const uint32_t (&a0)[4], const uint32_t (&a1)[4], uint4 v0,
                                         uint4 v1) {
  float e[4] = {0.f, 0.f, 0.f, 0.f};
  mma_f16(d, a0, v0.z, v0.w);
  mma_f16(e, a1, v1.z, v1.w);
  mma_f16(d, a0, v0.x, v0.y);
  mma_f16(e, a1, v1.x, v1.y);
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] += e[i];
}

// The f16 block scale of unit uu (0..2N-1) from a row's 2N scales held as N words.
template <int N>
__device__ __forceinline__ float scale_of(const uint32_t (&s)[N], int uu) {
  uint32_t w = s[0];
#pragma unroll
  for (int i = 1; i < N; ++i) w = (uu >> 1) == i ? s[i] : w;
  const float2 f = __half22float2(bits_h2(w));
  return (uu & 1) ? f.y : f.x;
}

// One ring stage of `NU` units (NU = SU, or 0: `nu` units known at run time) for NC blocks of
// 8 batch columns (x of block c at xst[c]) into the stage accumulators as[c]: block-scaled
// formats scale each unit's sums by the rows' block scales d; INT8 rows keep unit-
// interleaved MMA chains and add them at the end.  Each unit's A fragments serve every
// block.  Full stages run as groups of units: fragments first, then the MMAs round-robin
// over the group's units, so independent accumulator chains are in flight.
template <int FMT, int SU, int NU, int NC>
__device__ __forceinline__ void stage_mma(float (&as)[NC][4], const uint8_t* slot, const uint8_t* const (&xst)[NC],
                                          int g, int t, int nu) {
  constexpr int CB = code_bytes<FMT>();
  constexpr int RS = row_stride<FMT, SU>();
  constexpr int G = NC == 1 ? 4 : 2;  // units per group
  const uint8_t* row0 = slot + g * RS;
  const uint8_t* row8 = row0 + 8 * RS;
  if constexpr (FMT == QD_I8_ROW) {
    float c[NC][2][4];
#pragma unroll
    for (int b = 0; b < NC; ++b)
#pragma unroll
      for (int j = 0; j < 2; ++j) c[b][j][0] = c[b][j][1] = c[b][j][2] = c[b][j][3] = 0.f;
    auto one = [&](int uu, int j) {
      uint32_t a0[4], a1[4];
      unit_a<FMT>(row0 + uu * CB, row8 + uu * CB, t, a0, a1);
#pragma unroll
      for (int b = 0; b < NC; ++b) {
        uint4 v0, v1;
        unit_b(xst[b] + uu * 128, t, v0, v1);
        unit_mma(c[b][j], a0, a1, v0, v1);
      }
    };
    if constexpr (NU > 0) {
#pragma unroll
      for (int uu = 0; uu < NU; ++uu) one(uu, uu & 1);
    } else {
      for (int uu = 0; uu < nu; ++uu) one(uu, 0);
    }
#pragma unroll
    for (int b = 0; b < NC; ++b)
#pragma unroll
      for (int i = 0; i < 4; ++i) as[b][i] = c[b][0][i] + c[b][1][i];
  } else {
    // the block scales of rows g and g + 8 for the stage's SU units (f16, 2 SU bytes a row)
    const uint8_t* scs = slot + kTileRows * RS;
    uint32_t s0[SU / 2], s8[SU / 2];
    if constexpr (SU == 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(scs + g * 16);
      const uint4 b = *reinterpret_cast<const uint4*>(scs + (g + 8) * 16);
      s0[0] = a.x, s0[1] = a.y, s0[2] = a.z, s0[3] = a.w;
      s8[0] = b.x, s8[1] = b.y, s8[2] = b.z, s8[3] = b.w;
    } else {
      const uint2 a = *reinterpret_cast<const uint2*>(scs + g * 8);
      const uint2 b = *reinterpret_cast<const uint2*>(scs + (g + 8) * 8);
      s0[0] = a.x, s0[1] = a.y;
      s8[0] = b.x, s8[1] = b.y;
    }
    if constexpr (NU > 0) {
#pragma unroll
      for (int q = 0; q < NU / G; ++q) {
        uint32_t A0[G][4], A1[G][4];
        uint4 V0[NC][G], V1[NC][G];
        float D[NC][G][4];
#pragma unroll
        for (int u = 0; u < G; ++u) {
          unit_a<FMT>(row0 + (G * q + u) * CB, row8 + (G * q + u) * CB, t, A0[u], A1[u]);
#pragma unroll
          for (int b = 0; b < NC; ++b) {
            unit_b(xst[b] + (G * q + u) * 128, t, V0[b][u], V1[b][u]);
            D[b][u][0] = D[b][u][1] = D[b][u][2] = D[b][u][3] = 0.f;
          }
        }
#pragma unroll
        for (int b = 0; b < NC; ++b)
#pragma unroll
          for (int u = 0; u < G; ++u) unit_mma(D[b][u], A0[u], A1[u], V0[b][u], V1[b][u]);
#pragma unroll
        for (int u = 0; u < G; ++u) {
          const float d0 = scale_of(s0, G * q + u), d8 = scale_of(s8, G * q + u);
#pragma unroll
          for (int b = 0; b < NC; ++b) {
            as[b][0] = fmaf(d0, D[b][u][0], as[b][0]);
            as[b][1] = fmaf(d0, D[b][u][1], as[b][1]);
            as[b][2] = fmaf(d8, D[b][u][2], as[b][2]);
            as[b][3] = fmaf(d8, D[b][u][3], as[b][3]);
          }
        }
      }
    } else {
      for (int uu = 0; uu < nu; ++uu) {  // block formats: nu is even
        uint32_t a0[4], a1[4];
        unit_a<FMT>(row0 + uu * CB, row8 + uu * CB, t, a0, a1);
        const float d0 = scale_of(s0, uu), d8 = scale_of(s8, uu);
#pragma unroll
        for (int b = 0; b < NC; ++b) {
          uint4 v0, v1;
          unit_b(xst[b] + uu * 128, t, v0, v1);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          unit_mma(d, a0, a1, v0, v1);
          as[b][0] = fmaf(d0, d[0], as[b][0]);
          as[b][1] = fmaf(d0, d[1], as[b][1]);
          as[b][2] = fmaf(d8, d[2], as[b][2]);
          as[b][3] = fmaf(d8, d[3], as[b][3]);
        }
      }
    }
  }
}

// x in place: warp w converts the 256-column scale groups w, w + W, ... for R batch rows
// at once (R = 4 or 8), as straight-line code (rows past the batch convert zeros and store
// nothing), so the rows' loads and dependency chains overlap.  Lane l holds elements
// 8l..8l+7 of the group (unit l / 4, K half (l % 4) / 2): two 16-byte halves, each the four elements of one
// fragment thread (2 (l % 2) and 2 (l % 2) + 1), rewritten in place as that thread's
// (hi b0, hi b1, lo b0, lo b1).  Lanes 4-7 of each quarter take their second half
// first: the eight lanes of a 128-bit access then cover all 32 banks once.
template <int R, int W>
__device__ __forceinline__ void convert_x(uint8_t* xs, int64_t x_row, const float* gs, float* sxs, float* ssq, int units,
                                          int nxg, int batch, bool norm, int warp, int lane) {
  const int h = (lane >> 2) & 1;
  for (int s = warp; s < nxg; s += W) {
    const int e0 = s * kXCols + 8 * lane;
    const bool in = e0 < units * 32;
    uint8_t* sbase = xs + (int64_t)s * kXCols * 4 + 32 * lane;
    float v[R][8];  // [row][half h's 4 elements, then the other half's]
#pragma unroll
    for (int b = 0; b < R; ++b) {
      float4 q0 = make_float4(0.f, 0.f, 0.f, 0.f), q1 = q0;
      if (b < batch && in) {
        const float4* px = reinterpret_cast<const float4*>(sbase + b * x_row);
        q0 = px[h];
        q1 = px[h ^ 1];
      }
      v[b][0] = q0.x, v[b][1] = q0.y, v[b][2] = q0.z, v[b][3] = q0.w;
      v[b][4] = q1.x, v[b][5] = q1.y, v[b][6] = q1.z, v[b][7] = q1.w;
    }
    float ss[R];
#pragma unroll
    for (int b = 0; b < R; ++b) ss[b] = 0.f;
    if (norm) {
      float gv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (in) {
        const float4 g0 = *reinterpret_cast<const float4*>(gs + e0 + 4 * h);
        const float4 g1 = *reinterpret_cast<const float4*>(gs + e0 + 4 * (h ^ 1));
        gv[0] = g0.x, gv[1] = g0.y, gv[2] = g0.z, gv[3] = g0.w, gv[4] = g1.x, gv[5] = g1.y, gv[6] = g1.z, gv[7] = g1.w;
      }
#pragma unroll
      for (int b = 0; b < R; ++b) {
#pragma unroll
        for (int j2 = 0; j2 < 8; ++j2) {
          ss[b] = fmaf(v[b][j2], v[b][j2], ss[b]);
          v[b][j2] *= gv[j2];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int b = 0; b < R; ++b) ss[b] += __shfl_xor_sync(0xffffffffu, ss[b], o);
      }
    }
#pragma unroll
    for (int b = 0; b < R; ++b) {
      // the group's scale: 2^e with the largest |x| in [2^e, 2^(e+1)); magnitude bits
      // order like the values, and inf / NaN sit above every finite one
      uint32_t mb = 0;
#pragma unroll
      for (int j2 = 0; j2 < 8; ++j2) mb = max(mb, __float_as_uint(v[b][j2]) & 0x7FFFFFFFu);
      mb = __reduce_max_sync(0xffffffffu, mb);
      const bool bad = mb >= 0x7F800000u, live = mb != 0u;
      const int e = (int)(mb >> 23) - 127;
      const float rs = live && !bad ? pow2i(-e) : 0.f;
      float4 fr[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {  // the two halves, each one fragment thread's elements
        const float y0 = v[b][4 * k] * rs, y1 = v[b][4 * k + 1] * rs;
        const float y2 = v[b][4 * k + 2] * rs, y3 = v[b][4 * k + 3] * rs;
        const __half2 h0 = __floats2half2_rn(y0, y2), h1 = __floats2half2_rn(y1, y3);
        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
        const __half2 l0 = __floats2half2_rn(y0 - f0.x, y2 - f0.y), l1 = __floats2half2_rn(y1 - f1.x, y3 - f1.y);
        fr[k] = make_float4(__uint_as_float(h2_bits(h0)), __uint_as_float(h2_bits(h1)), __uint_as_float(h2_bits(l0)),
                            __uint_as_float(h2_bits(l1)));
      }
      if (b < batch) {
        if (in) {
          float4* px = reinterpret_cast<float4*>(sbase + b * x_row);
          px[h] = fr[0];
          px[h ^ 1] = fr[1];
        }
        if (lane == 0) {
          sxs[s * kMaxCols + b] = bad ? __uint_as_float(0x7FC00000u) : live ? pow2i(e) : 0.f;
          ssq[s * kMaxCols + b] = ss[b];
        }
      }
    }
  }
}

template <int FMT, int NC, int W, bool SPLIT>
__global__ void __launch_bounds__(W * 32, 1) k_gemv_mma(const Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int CB = code_bytes<FMT>();
  constexpr int SU = stage_units<W>();  // units per ring stage
  constexpr int RS = row_stride<FMT, SU>();
  constexpr int kSlot = slot_bytes<FMT, SU>();
  const int kStages = p.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;  // mma fragment: row group, thread in group
  const PackedView& Wm = p.W;
  // split launches: CTA `rank` of each cluster of C takes its share [ua, ub) of the range's
  // units (whole x groups); the clusters take tiles as CTAs do otherwise
  const int C = SPLIT ? p.ksplit : 1;
  const int rank = SPLIT ? (int)(blockIdx.x % C) : 0;
  const int64_t ncl = gridDim.x / C, cid = blockIdx.x / C;
  const int nxg_all = (p.units + kXUnits - 1) / kXUnits;
  const int ua = SPLIT ? rank * nxg_all / C * kXUnits : 0;
  const int ub = SPLIT ? min((rank + 1) * nxg_all / C * kXUnits, p.units) : p.units;
  const int units = ub - ua;             // this CTA's units
  const int64_t uoff = (int64_t)p.u0 + ua;  // the first of them in a row
  if constexpr (SPLIT) cluster_arrive_relaxed();  // every CTA of the cluster has started (waited below)
  const int nst = (units + SU - 1) / SU;                     // stages per tile
  const int nxg = (units + kXUnits - 1) / kXUnits;           // x scale groups
  const bool norm = p.norm_g != nullptr;
  const int KS = p.ks, grp = warp / KS, ks = warp % KS;
  const Layout L = layout<FMT, W>(SPLIT ? split_units_cap(p.units, C) : units, p.batch, norm, kStages,
                                  SPLIT ? split_slot_bytes(C, W / KS, NC) : 0, p.pdepth);
  const int64_t tiles = (Wm.rows + kTileRows - 1) / kTileRows;
  // the KS warps of a group share each of the group's tiles; warp ks of the group takes
  // the tile's stages [st0, st1); groups take tiles round-robin over the grid (a split
  // launch gives every group one tile at most)
  const int st0 = ks * nst / KS, st1 = (ks + 1) * nst / KS;
  const int64_t gslot = (int64_t)grp * ncl + cid, ngs = ncl * (W / KS);
  const int64_t tiles_end = SPLIT ? min(tiles, gslot + 1) : tiles;
  uint8_t* ring = smem + L.ring + (size_t)warp * kStages * kSlot;
  const uint32_t ring_s = tc::smem_u32(ring);
  uint8_t* xs = smem + L.xs;
  const float* gs = reinterpret_cast<const float*>(smem + L.gs);
  float* sxs = reinterpret_cast<float*>(smem + L.sx);   // [x group][16] x scales
  float* ssq = reinterpret_cast<float*>(smem + L.ssq);  // [x group][16] sums of squares
  float* partial = reinterpret_cast<float*>(smem + L.partial);  // [pdepth][warps][32][NC][4]
  const uint32_t bar = tc::smem_u32(smem + L.bar);

  if (threadIdx.x == 0) {
    tc::mbar_init(bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---- ring: stage s of a tile = units [SU s, SU s + SU) of its 16 rows.  Lane l copies
  // the 16-byte code chunk l % kPerRow of rows l / kPerRow + i * kRowsPerPass and the
  // 4-byte scale words l + 32 j (unit pair l % (SU / 2) of rows l / (SU / 2) + j 64 / SU);
  // the source rows of a tile are set up once per tile (clamped to the last row for a
  // ragged tile)
  constexpr int kPerRow = SU * CB / 16;  // 16-byte chunks per row and stage
  constexpr int kRowsPerPass = 32 / kPerRow;
  constexpr int kChunks = kTileRows / kRowsPerPass;  // code chunks per lane and stage
  const int crow = lane / kPerRow, crem = lane % kPerRow, cunit = crem / (CB / 16);
  constexpr int kScaleWords = SU / 4;  // scale words per lane and stage
  const int srow = lane / (SU / 2), spr = lane % (SU / 2);
  int64_t lt = gslot;  // tile of the next copy
  int ls = st0;        // its stage
  const uint8_t* cptr[kChunks];
  const uint8_t* sptr[kScaleWords];
  auto tile_ptrs = [&]() {
#pragma unroll
    for (int i = 0; i < kChunks; ++i) {
      const int64_t r = min(lt * kTileRows + crow + i * kRowsPerPass, Wm.rows - 1);
      cptr[i] = Wm.codes + r * Wm.row_code_bytes + uoff * CB + 16 * crem;
    }
    if constexpr (scale_bytes<FMT, SU>() > 0) {
#pragma unroll
      for (int j = 0; j < kScaleWords; ++j) {
        const int64_t r = min(lt * kTileRows + srow + j * (64 / SU), Wm.rows - 1);
        sptr[j] = Wm.scales + r * Wm.row_scale_bytes + (uoff + 2 * spr) * 2;
      }
    }
  };
  if (lt < tiles_end) tile_ptrs();
  auto issue = [&](int slot_idx) {
    if (lt < tiles_end && st1 > st0) {
      const uint32_t slot = ring_s + (uint32_t)slot_idx * kSlot;
      const int u0 = ls * SU;
      if (u0 + cunit < units) {
#pragma unroll
        for (int i = 0; i < kChunks; ++i)
          cp16(slot + (uint32_t)((crow + i * kRowsPerPass) * RS + 16 * crem), cptr[i] + (int64_t)u0 * CB);
      }
      if constexpr (scale_bytes<FMT, SU>() > 0) {
        // units come in pairs (even unit counts)
        if (u0 + 2 * spr < units) {
#pragma unroll
          for (int j = 0; j < kScaleWords; ++j)
            cp4(slot + (uint32_t)(kTileRows * RS + ((srow + j * (64 / SU)) * SU + 2 * spr) * 2), sptr[j] + u0 * 2);
        }
      }
      if (++ls == st1) {
        ls = st0;
        lt += ngs;
        if (lt < tiles_end) tile_ptrs();
      }
    }
    cp_commit();
  };

  // ---- before the dependency wait: the norm gains (a weight) by bulk copy and the
  // ring's first kStages - 1 stages; neither depends on the previous kernel
  const uint32_t row_bytes = (uint32_t)units * 128u;
  if (threadIdx.x == 0) {
    tc::mbar_arrive_expect_tx(bar, row_bytes * (uint32_t)(p.batch + (norm ? 1 : 0)));
    if (norm) tc::bulk_copy_g2s(tc::smem_u32(smem + L.gs), p.norm_g + uoff * 32, row_bytes, bar);
  }
  for (int s = 0; s < kStages - 1; ++s) issue(s);

  pdl_wait();  // x (and y, for accumulation) belong to the previous kernel
  if (threadIdx.x == 0) {
    for (int b = 0; b < p.batch; ++b)
      tc::bulk_copy_g2s(tc::smem_u32(xs + b * L.x_row), p.x + b * p.x_stride + uoff * 32, row_bytes, bar);
  }
  for (int i = threadIdx.x; i < nxg * kMaxCols; i += W * 32) {
    if ((i % kMaxCols) >= p.batch) sxs[i] = ssq[i] = 0.f;  // columns without a batch row
  }
  if (!__syncthreads_and(tc::mbar_wait_sleep(bar, 0))) {
    // the copies did not land in time: report it, give them one more bounded wait (they
    // target this CTA's shared memory), drain the ring and leave
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, kErrTimeout);
    tc::mbar_wait_sleep(bar, 0);
    cp_wait_n<0>();
    if constexpr (SPLIT) {  // the cluster barrier's phases as the other CTAs go through them
      cluster_wait();
      cluster_arrive();
      cluster_wait();
    }
    return;
  }

  // x in place, 8 batch rows a pass (rows 8-15 with their scale and norm columns offset)
  if (p.batch <= 4) convert_x<4, W>(xs, L.x_row, gs, sxs, ssq, units, nxg, p.batch, norm, warp, lane);
  else convert_x<8, W>(xs, L.x_row, gs, sxs, ssq, units, nxg, min(p.batch, 8), norm, warp, lane);
  if constexpr (NC > 1) {
    if (p.batch > 8)
      convert_x<8, W>(xs + 8 * L.x_row, L.x_row, gs, sxs + 8, ssq + 8, units, nxg, p.batch - 8, norm, warp, lane);
  }
  __syncthreads();
  // RMSNorm factors of this lane's columns 8c + 2t, 8c + 2t + 1 (group sums in group order:
  // every CTA forms the same value)
  float inv[NC][2];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      inv[c][j] = 1.f;
      if (norm) {
        float tt = 0.f;
        for (int s = 0; s < nxg; ++s) tt += ssq[s * kMaxCols + 8 * c + 2 * t + j];
        inv[c][j] = 1.0f / sqrtf(tt / (float)(units * 32) + p.eps);
      }
    }
  pdl_trigger();

  // this lane's B column of block c: batch row 8c + g, or (no such row) the last staged
  // one, whose sums land in a column the epilogue never stores
  const uint8_t* xrow[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) xrow[c] = xs + min(8 * c + g, p.batch - 1) * L.x_row;
  unsigned long long best[NC][2];  // argmax keys of columns 8c + 2t, 8c + 2t + 1
#pragma unroll
  for (int c = 0; c < NC; ++c) best[c][0] = best[c][1] = 0ull;
  float acc[NC][4];
  int cs = 0, it = 0;
  // ---- end of a tile (first warp of the group): rows tile + g, + 8; columns 8c + 2t,
  // 8c + 2t + 1
  auto finish = [&](int64_t tl) {
    const int64_t rbase = tl * kTileRows;
    float rsc[2] = {1.f, 1.f};  // INT8 row scales of rows g, g + 8
    if constexpr (FMT == QD_I8_ROW) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
        rsc[h] = __ldg(reinterpret_cast<const float*>(Wm.scales + min(rbase + g + 8 * h, Wm.rows - 1) * Wm.row_scale_bytes));
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = acc[c][i] * inv[c][i & 1] * rsc[i >> 1];
      // the next row's values (row g + 1 is lane + 4) for the pair epilogues
      float nx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) nx[i] = __shfl_down_sync(0xffffffffu, v[i], 4);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t r = rbase + g + (i >= 2 ? 8 : 0);
        const int b = 8 * c + 2 * t + (i & 1);
        if (b >= p.batch || r >= Wm.rows) continue;
        if (p.mode == kGemvSwiGLU) {
          if ((g & 1) == 0 && r + 1 < Wm.rows)
            p.y[(int64_t)b * (Wm.rows / 2) + r / 2] = v[i] / (1.0f + expf(-v[i])) * nx[i];
        } else if (p.mode == kGemvQKV) {
          if ((g & 1) == 0 && r + 1 < Wm.rows) qkv_pair(p, r, b, v[i], nx[i]);
        } else {
          float* dst = p.y + (int64_t)b * Wm.rows + r;
          if (p.mode == kGemvAccumulate || p.accumulate) *dst = __ldcg(dst) + v[i];
          else *dst = v[i];
          if (p.mode == kGemvArgmax) {
            const unsigned long long key = argmax_key(v[i], (uint32_t)r);
            best[c][i & 1] = key > best[c][i & 1] ? key : best[c][i & 1];
          }
        }
      }
    }
  };
  int64_t split_tile = -1;  // split launches: the group's tile, finished after the exchange
  for (int64_t tl = gslot; tl < tiles_end; tl += ngs, ++it) {  // uniform over the group
#pragma unroll
    for (int c = 0; c < NC; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
    for (int st = st0; st < st1; ++st) {
      __syncwarp();
      issue(cs == 0 ? kStages - 1 : cs - 1);
      cp_wait_dyn(kStages - 1);
      __syncwarp();
      const uint8_t* slot = ring + (size_t)cs * kSlot;
      const uint8_t* xst[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) xst[c] = xrow[c] + (size_t)st * SU * 128;
      const int nu = min(SU, units - st * SU);
      float as[NC][4];
#pragma unroll
      for (int c = 0; c < NC; ++c) as[c][0] = as[c][1] = as[c][2] = as[c][3] = 0.f;
      if (nu == SU) stage_mma<FMT, SU, SU, NC>(as, slot, xst, g, t, nu);
      else stage_mma<FMT, SU, 0, NC>(as, slot, xst, g, t, nu);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        // the x scales of columns 8c + 2t, 8c + 2t + 1 in the stage's scale group
        const float2 sx = *reinterpret_cast<const float2*>(sxs + (st / (kXUnits / SU)) * kMaxCols + 8 * c + 2 * t);
        acc[c][0] = fmaf(sx.x, as[c][0], acc[c][0]);
        acc[c][1] = fmaf(sx.y, as[c][1], acc[c][1]);
        acc[c][2] = fmaf(sx.x, as[c][2], acc[c][2]);
        acc[c][3] = fmaf(sx.y, as[c][3], acc[c][3]);
      }
      cs = (cs + 1 == kStages) ? 0 : cs + 1;
    }
    if (KS > 1) {
      // the group's column parts, summed in part order by its first warp
      float* pt = partial + (size_t)(p.pdepth == 2 ? (it & 1) : 0) * W * 32 * 4 * NC;
#pragma unroll
      for (int c = 0; c < NC; ++c)
        *reinterpret_cast<float4*>(pt + ((warp * 32 + lane) * NC + c) * 4) =
            make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
      asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(KS * 32) : "memory");
      if (ks != 0) continue;  // uniform per warp
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
        for (int k = 0; k < KS; ++k) {
          const float4 q = *reinterpret_cast<const float4*>(pt + (((grp * KS + k) * 32 + lane) * NC + c) * 4);
          acc[c][0] += q.x;
          acc[c][1] += q.y;
          acc[c][2] += q.z;
          acc[c][3] += q.w;
        }
      }
    }
    if constexpr (SPLIT) split_tile = tl;
    else finish(tl);
  }
  cp_wait_n<0>();  // no copy may still target this CTA's shared memory at exit
  if constexpr (SPLIT) {
    // the other CTAs' tile sums into the first CTA's slots, one cluster barrier, then the
    // first CTA adds them in CTA order and runs the epilogue
    const int groups = W / KS;
    const uint32_t spl = tc::smem_u32(smem + L.spl);
    cluster_wait();  // the first CTA has started: its slots exist
    if (rank != 0 && ks == 0 && split_tile >= 0) {
#pragma unroll
      for (int c = 0; c < NC; ++c)
        st_cluster4(spl + (uint32_t)(((((rank - 1) * groups + grp) * 32 + lane) * NC + c) * 16), 0, acc[c][0], acc[c][1],
                    acc[c][2], acc[c][3]);
    }
    cluster_arrive();
    cluster_wait();
    if (rank != 0) return;
    if (ks == 0 && split_tile >= 0) {
      const float* sp = reinterpret_cast<const float*>(smem + L.spl);
      for (int r = 1; r < C; ++r) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float4 q = *reinterpret_cast<const float4*>(sp + ((((r - 1) * groups + grp) * 32 + lane) * NC + c) * 4);
          acc[c][0] += q.x;
          acc[c][1] += q.y;
          acc[c][2] += q.z;
          acc[c][3] += q.w;
        }
      }
      finish(split_tile);
    }
  }
  if (p.mode == kGemvArgmax) {
    // per batch column: max over the lanes holding it (same t), one atomicMax per warp;
    // the last CTA to arrive finalises the tokens and re-arms keys and counter
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        unsigned long long kk = best[c][j];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, kk, off);
          kk = o > kk ? o : kk;
        }
        const int b = 8 * c + 2 * t + j;
        if (g == 0 && kk != 0 && b < p.batch) atomicMax(p.am.key + b, kk);
      }
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned int old;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.am.counter) : "memory");
      if (old == gridDim.x - 1) {
        for (int b = 0; b < p.batch; ++b) {
          const unsigned long long kk = atomicExch(p.am.key + b, 0ull);
          p.am.tok_out[b] = (int32_t)argmax_key_index(kk);
          p.am.pos[b] += 1;
        }
        *p.am.counter = 0u;
      }
    }
  }
}


constexpr size_t kSmemCap = 220 * 1024;

int sm_count() {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      v <= 0) {
    cudaGetLastError();
    return 152;
  }
  return v;
}

template <int FMT, int NC, int W, bool SPLIT = false>
bool smem_attr_set() {
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!done[dev]) {
    if (cudaFuncSetAttribute(k_gemv_mma<FMT, NC, W, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemCap) !=
        cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    done[dev] = true;
  }
  return true;
}

bool fmt_taken(int fmt) { return fmt == QD_Q4_0 || fmt == QD_Q8_0 || fmt == QD_I8_ROW; }

template <int W>
size_t smem_for_w(int fmt, int units, int batch, bool norm, int stages, int depth) {
  switch (fmt) {
    case QD_Q4_0: return layout<QD_Q4_0, W>(units, batch, norm, stages, 0, depth).total;
    case QD_Q8_0: return layout<QD_Q8_0, W>(units, batch, norm, stages, 0, depth).total;
    default: return layout<QD_I8_ROW, W>(units, batch, norm, stages, 0, depth).total;
  }
}
size_t smem_for(int fmt, int warps, int units, int batch, bool norm, int stages, int depth) {
  return warps == 16 ? smem_for_w<16>(fmt, units, batch, norm, stages, depth)
                     : smem_for_w<8>(fmt, units, batch, norm, stages, depth);
}

int ks_for(int64_t tiles, int nst, int sms, int warps);

// One launch over `units` columns with CTAs of `warps` warps: warps per tile, grid,
// partial-sum buffers and ring depth (the deepest, up to 8 slots a warp, that fits the
// shared memory; 0: none does).
struct RangePlan {
  int ks = 1;
  int64_t ctas = 0;
  int depth = 2;
  int stages = 0;
};
RangePlan range_plan(int fmt, int warps, int64_t rows, int units, int batch, bool norm) {
  RangePlan r;
  const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
  const int su = warps == 16 ? stage_units<16>() : stage_units<8>();
  const int sms = sm_count();
  r.ks = ks_for(tiles, (units + su - 1) / su, sms, warps);
  const int64_t groups_per_cta = warps / r.ks;
  r.ctas = (tiles + groups_per_cta - 1) / groups_per_cta;
  if (r.ctas > sms) r.ctas = sms;
  r.depth = r.ks == 1 ? 0 : tiles <= r.ctas * groups_per_cta ? 1 : 2;
  for (int s = 8; s >= 2 && !r.stages; --s)
    if (smem_for(fmt, warps, units, batch, norm, s, r.depth) <= kSmemCap) r.stages = s;
  return r;
}
int stages_for(int fmt, int warps, int64_t rows, int units, int batch, bool norm) {
  return range_plan(fmt, warps, rows, units, batch, norm).stages;
}

// Warps per CTA for a launch over `units` columns: 16 (4-unit stages) where their ring
// can be three stages deep, otherwise 8 (8-unit stages).
int warps_for(int fmt, int64_t rows, int units, int batch, bool norm) {
  return stages_for(fmt, 16, rows, units, batch, norm) >= 3 ? 16 : 8;
}

// Ring stages a column range is sized for: about 64 KB of weights in flight per SM (8 warps).
int ring_floor(int fmt) {
  const int slot = fmt == QD_Q4_0 ? slot_bytes<QD_Q4_0, 8>() : fmt == QD_Q8_0 ? slot_bytes<QD_Q8_0, 8>() : slot_bytes<QD_I8_ROW, 8>();
  return max(2, (65536 + 8 * slot - 1) / (8 * slot));
}

// Units per column range: all of them when x fits beside a ring of two stages or more;
// otherwise the widest multiple of an x scale group that leaves room for ring_floor stages
// of the 8-warp CTA.
int range_units(int fmt, int64_t rows, int units, int batch, bool norm) {
  if (stages_for(fmt, 8, rows, units, batch, norm) >= 2) return units;
  const int floor_st = ring_floor(fmt);
  int ru = (units / kXUnits) * kXUnits;
  while (ru > kXUnits && smem_for(fmt, 8, ru, batch, norm, floor_st, 2) > kSmemCap) ru -= kXUnits;
  return smem_for(fmt, 8, ru, batch, norm, floor_st, 2) <= kSmemCap ? ru : 0;
}

// Warps per tile (1, 2, 4, or 8 in a 16-warp CTA): the fewest rounds of stages on the
// busiest warp, counting the CTAs the grid can hold (a small extra cost per split for the
// partial sums).
int ks_for(int64_t tiles, int nst, int sms, int warps) {
  int best = 1;
  double best_cost = 1e30;
  for (int ks : {1, 2, 4, 8}) {
    if (ks == 8 && warps < 16) break;
    const int64_t groups_per_cta = warps / ks;
    int64_t ctas = (tiles + groups_per_cta - 1) / groups_per_cta;
    if (ctas > sms) ctas = sms;
    const int64_t rounds = (tiles + ctas * groups_per_cta - 1) / (ctas * groups_per_cta);
    const double cost = (double)rounds * ((nst + ks - 1) / ks) * (1.0 + 0.05 * (ks - 1));
    if (cost < best_cost) {
      best_cost = cost;
      best = ks;
    }
  }
  return best;
}

// One launch over the column range [p.u0, p.u0 + p.units) with CTAs of W warps.
template <int FMT, int W>
qd_status launch_range(Params p, bool pdl, cudaStream_t stream) {
  if (!(col_blocks(p.batch) == 2 ? smem_attr_set<FMT, 2, W>() : smem_attr_set<FMT, 1, W>())) return QD_ERR_CUDA;
  const bool norm = p.norm_g != nullptr;
  const RangePlan rp = range_plan(FMT, W, p.W.rows, p.units, p.batch, norm);
  if (rp.stages < 2) return QD_ERR_UNSUPPORTED;
  p.stages = rp.stages;
  p.ks = rp.ks;
  p.pdepth = rp.depth;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rp.ctas);
  cfg.blockDim = dim3(W * 32);
  cfg.dynamicSmemBytes = layout<FMT, W>(p.units, p.batch, norm, p.stages, 0, p.pdepth).total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (col_blocks(p.batch) == 2)
    return cudaLaunchKernelEx(&cfg, k_gemv_mma<FMT, 2, W, false>, p) == cudaSuccess ? QD_OK : QD_ERR_CUDA;
  return cudaLaunchKernelEx(&cfg, k_gemv_mma<FMT, 1, W, false>, p) == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

// ---- split launches (8-warp CTAs in clusters of 2 or 4 over the columns)
struct SplitPlan {
  int c = 0;       // CTAs per cluster; 0: no split fits
  int ks = 1;      // warps per tile
  int stages = 0;  // ring depth
  int64_t clusters = 0;
};

// Clusters of `c` CTAs with `smem` bytes each that the GPU holds at once (the grid must
// not run in waves: every CTA takes its tile up front); 0 on error.
template <int FMT, int NC>
int max_active_clusters(int c, size_t smem) {
  struct Entry {
    int dev, c;
    size_t smem;
    int n;
  };
  static Entry cache[32];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].c == c && cache[i].smem == smem) return cache[i].n;
  if (!smem_attr_set<FMT, NC, 8, true>()) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c);
  cfg.blockDim = dim3(8 * 32);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeClusterDimension;
  a[0].val.clusterDim.x = (unsigned)c;
  a[0].val.clusterDim.y = 1;
  a[0].val.clusterDim.z = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)k_gemv_mma<FMT, NC, 8, true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (used < 32) cache[used++] = Entry{dev, c, smem, n};
  return n;
}

// The split with the fewest ring stages on the busiest warp (a shallow ring costs a
// quarter more) among clusters of 2 or 4 whose CTAs each hold their share of x beside a
// ring of two stages or more and whose groups take one tile each.
template <int FMT>
SplitPlan split_plan(int64_t rows, int units, int batch) {
  SplitPlan best;
  double best_cost = 1e30;
  const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
  const int nxg = (units + kXUnits - 1) / kXUnits;
  const int nc = col_blocks(batch);
  for (int c : {2, 4}) {
    if (nxg < 2 * c) continue;
    const int cap = split_units_cap(units, c);
    const int nst = (cap + stage_units<8>() - 1) / stage_units<8>();
    for (int ks : {1, 2, 4}) {
      const size_t sb = split_slot_bytes(c, 8 / ks, nc);
      int st = 0;
      for (int s2 = 8; s2 >= 2 && !st; --s2)
        if (layout<FMT, 8>(cap, batch, false, s2, sb, 1).total <= kSmemCap) st = s2;
      if (st < 2) continue;
      const int64_t need = (tiles + 8 / ks - 1) / (8 / ks);  // clusters for one tile per group
      const size_t smem = layout<FMT, 8>(cap, batch, false, st, sb, 1).total;
      const int64_t fit = nc == 2 ? max_active_clusters<FMT, 2>(c, smem) : max_active_clusters<FMT, 1>(c, smem);
      if (need > fit) continue;
      const double cost = (double)((nst + ks - 1) / ks) * (1.0 + 0.05 * (ks - 1)) * (st >= 3 ? 1.0 : 1.25);
      if (cost < best_cost) {
        best_cost = cost;
        best.c = c;
        best.ks = ks;
        best.stages = st;
        best.clusters = need;
      }
    }
  }
  return best;
}

template <int FMT, int NC>
qd_status launch_split_nc(Params p, const SplitPlan& sp, bool pdl, cudaStream_t stream) {
  if (!smem_attr_set<FMT, NC, 8, true>()) return QD_ERR_CUDA;
  p.ks = sp.ks;
  p.stages = sp.stages;
  p.ksplit = sp.c;
  p.pdepth = 1;  // one tile per warp group
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(sp.clusters * sp.c));
  cfg.blockDim = dim3(8 * 32);
  cfg.dynamicSmemBytes =
      layout<FMT, 8>(split_units_cap(p.units, sp.c), p.batch, false, sp.stages, split_slot_bytes(sp.c, 8 / sp.ks, NC), 1)
          .total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sp.c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_mma<FMT, NC, 8, true>, p) == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

// One launch with 16-warp CTAs where their ring fits three stages deep; otherwise 8-warp
// CTAs over all column ranges in order: the first stores (or accumulates, in accumulate
// mode), the rest accumulate, each a programmatic dependent of the one before.
template <int FMT>
qd_status launch(Params p, bool pdl, cudaStream_t stream) {
  const int units = (int)(p.W.cols / 32);
  const bool norm = p.norm_g != nullptr;
  if (warps_for(FMT, p.W.rows, units, p.batch, norm) == 16) return launch_range<FMT, 16>(p, pdl, stream);
  const int ru = range_units(FMT, p.W.rows, units, p.batch, norm);
  if (ru < units && !norm && (p.mode == kGemvStore || p.mode == kGemvAccumulate)) {
    // x too wide for one CTA: split the columns over a cluster where that fits
    const SplitPlan sp = split_plan<FMT>(p.W.rows, units, p.batch);
    if (sp.c > 0)
      return col_blocks(p.batch) == 2 ? launch_split_nc<FMT, 2>(p, sp, pdl, stream)
                                      : launch_split_nc<FMT, 1>(p, sp, pdl, stream);
  }
  if (ru <= 0) return QD_ERR_UNSUPPORTED;
  for (int u0 = 0; u0 < units; u0 += ru) {
    p.u0 = u0;
    p.units = min(ru, units - u0);
    p.accumulate = u0 > 0;
    const qd_status st = launch_range<FMT, 8>(p, u0 > 0 || pdl, stream);
    if (st != QD_OK) return st;
  }
  return QD_OK;
}

}  // namespace mma_gemv

namespace mma_gemv {

// Whether x too wide for one CTA splits over a cluster (store and accumulate without the
// fused norm).
bool split_fits(const GemvArgs& a) {
  const int units = (int)(a.W.cols / 32);
  if (a.norm_g || (a.mode != kGemvStore && a.mode != kGemvAccumulate)) return false;
  if (stages_for(a.fmt, 8, a.W.rows, units, a.batch, false) >= 2) return false;
  switch (a.fmt) {
    case QD_Q4_0: return split_plan<QD_Q4_0>(a.W.rows, units, a.batch).c > 0;
    case QD_Q8_0: return split_plan<QD_Q8_0>(a.W.rows, units, a.batch).c > 0;
    default: return split_plan<QD_I8_ROW>(a.W.rows, units, a.batch).c > 0;
  }
}

// Whether one launch sequence (a single launch, a split launch or column ranges) takes
// these arguments: x of every batch row beside a ring of two stages, or (store and
// accumulate without the fused norm) a split over a cluster or column ranges that fit.
bool one_pass_fits(const GemvArgs& a) {
  const int units = (int)(a.W.cols / 32);
  if (stages_for(a.fmt, 8, a.W.rows, units, a.batch, a.norm_g != nullptr) >= 2) return true;
  const bool splits = (a.mode == kGemvStore || a.mode == kGemvAccumulate) && !a.norm_g;
  return splits && range_units(a.fmt, a.W.rows, units, a.batch, false) > 0;
}

// Batch rows [b0, b0 + nb) of `a` as arguments of their own: x, y and every epilogue
// pointer moved to row b0.
GemvArgs row_slice(const GemvArgs& a, int b0, int nb) {
  GemvArgs s = a;
  s.batch = nb;
  s.x = a.x + (int64_t)b0 * a.W.cols;
  const int64_t ycols = a.mode == kGemvSwiGLU ? a.W.rows / 2 : a.W.rows;
  if (a.y) s.y = a.y + (int64_t)b0 * ycols;
  if (a.mode == kGemvQKV) {
    QkvEpilogue& e = s.qkv;
    e.pos = a.qkv.pos + b0;
    e.q_out = a.qkv.q_out + (int64_t)b0 * a.qkv.q_stride;
    const int64_t esz = a.qkv.kv_f16 ? 2 : 4;
    e.kc = static_cast<uint8_t*>(a.qkv.kc) + (int64_t)b0 * a.qkv.cache_batch_stride * esz;
    e.vc = static_cast<uint8_t*>(a.qkv.vc) + (int64_t)b0 * a.qkv.cache_batch_stride * esz;
  }
  if (a.mode == kGemvArgmax) {
    s.am.key = a.am.key + b0;
    s.am.tok_out = a.am.tok_out + b0;
    s.am.pos = a.am.pos + b0;
  }
  return s;
}

qd_status launch_args(const GemvArgs& a, cudaStream_t stream) {
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
  p.x_stride = a.W.cols;
  p.u0 = 0;
  p.units = (int)(a.W.cols / 32);
  p.stages = 0;
  p.ks = 1;
  p.ksplit = 1;
  p.pdepth = 2;
  p.accumulate = false;
  switch (a.fmt) {
    case QD_Q4_0: return launch<QD_Q4_0>(p, a.pdl, stream);
    case QD_Q8_0: return launch<QD_Q8_0>(p, a.pdl, stream);
    default: return launch<QD_I8_ROW>(p, a.pdl, stream);
  }
}

}  // namespace mma_gemv

// Batch 3-16, Q4_0 / Q8_0 / INT8 rows, even unit counts for the block formats (4-byte scale
// copies), x and norm_g on 16-byte boundaries (bulk copies).  One pass over the weights when
// x of every batch row fits beside a ring of two stages (or, store and accumulate without
// RMSNorm, split over a cluster's CTAs or in column ranges that fit).  At batch 9-16
// otherwise a split launch, or two passes of up to 8 rows for Q4_0 and Q8_0 (measured
// faster than column ranges: the second pass finds much of the weights in L2); INT8 rows
// then go to the batch-16 tcgen05 kernel, which measured faster there.
bool gemv_mma_supported(const GemvArgs& a) {
  using namespace mma_gemv;
  if (!fmt_taken(a.fmt) || a.batch < 3 || a.batch > kMaxCols || a.W.cols % 32 || a.W.cols > (1 << 22)) return false;
  if (reinterpret_cast<uintptr_t>(a.x) & 15) return false;
  if (a.norm_g && (reinterpret_cast<uintptr_t>(a.norm_g) & 15)) return false;
  const int units = (int)(a.W.cols / 32);
  if ((a.fmt == QD_Q4_0 || a.fmt == QD_Q8_0) && (units & 1)) return false;
  if (a.mode == kGemvSwiGLU || a.mode == kGemvQKV) {
    if (a.W.rows & 1) return false;
  }
  if (a.batch <= 8) return one_pass_fits(a);
  const int units_ok = stages_for(a.fmt, 8, a.W.rows, units, a.batch, a.norm_g != nullptr) >= 2;
  if (units_ok || split_fits(a)) return true;
  if (a.fmt == QD_I8_ROW) return false;
  return one_pass_fits(row_slice(a, 0, 8)) && one_pass_fits(row_slice(a, 8, a.batch - 8));
}

qd_status launch_q_gemv_mma(const GemvArgs& a, cudaStream_t stream) {
  using namespace mma_gemv;
  if (!gemv_mma_supported(a)) return QD_ERR_UNSUPPORTED;
  const int units = (int)(a.W.cols / 32);
  if (a.batch <= 8 || stages_for(a.fmt, 8, a.W.rows, units, a.batch, a.norm_g != nullptr) >= 2 || split_fits(a))
    return launch_args(a, stream);
  // two passes of up to 8 batch rows, the second a programmatic dependent of the first
  const qd_status st = launch_args(row_slice(a, 0, 8), stream);
  if (st != QD_OK) return st;
  GemvArgs hi = row_slice(a, 8, a.batch - 8);
  hi.pdl = true;
  return launch_args(hi, stream);
}

}  // namespace qd
