// Decode-attention building blocks shared by the split-KV kernels and the fused
// attention block: the tiled online-softmax walk over cached positions (llmoxide blog s5,
// dasLLAMA 8.7.1.6.2 attention) and the q load.
#pragma once
#include "qd_internal.cuh"

namespace qd {
namespace attn {

constexpr int kAttnWarps = 4;
constexpr int kHeadDim = 64;
constexpr int kMaxGroup = 8;

constexpr int kMaxCluster = 8;

// Walk of positions [p_begin, p_end) by the CTA's W warps in tiles: warp w takes
// positions tile + w * P + i (i < P) of each tile of W * P positions.
//  * scores: L lanes share one position, lane j holding dims [j * 64/L, (j+1) * 64/L)
//    of its key row and of every q head; the dot is finished with log2(L) shuffles.
//    Scores are in log2 units (q was pre-scaled by log2(e) / sqrt(head_dim)).
//  * softmax: one running max / sum update per tile and head (online softmax over
//    tiles), weights 2^(s - m).
//  * values: lane j holds dims 2j, 2j+1 of the P value rows; each position's weight
//    is broadcast from its lane group.
// The next tile's rows are loaded before the current tile is used.
template <int G>
struct AttnLayout {
  static constexpr int L = G <= 4 ? 4 : 8;  // lanes per key row
  static constexpr int P = 32 / L;          // positions per warp per tile
  static constexpr int D = kHeadDim / L;    // key dims per lane
};

template <int G, int DEP, int W = kAttnWarps>
__device__ __forceinline__ void attn_tiles(const float* kb, const float* vb, int p_begin, int p_end, int warp,
                                           int lane, const float (&qs)[G][AttnLayout<G>::D], float (&m)[G],
                                           float (&l)[G], float2 (&o)[G]) {
  using A = AttnLayout<G>;
  constexpr int L = A::L, P = A::P, D = A::D;
  constexpr int kTile = W * P;
  // DEP tiles in flight per warp: the rows of DEP tiles load while one is used (a
  // register ring with static slots)
  const int j = lane % L, pi = lane / L;  // this lane's dim slice and position in the warp tile
  float4 kr[DEP][D / 4];
  float2 vr[DEP][P];
  auto load = [&](int tile, float4 (&kd)[D / 4], float2 (&vd)[P]) {
    const int p = min(tile + warp * P + pi, p_end - 1);
    const float4* krow = reinterpret_cast<const float4*>(kb + (int64_t)p * kHeadDim + j * D);
#pragma unroll
    for (int t = 0; t < D / 4; ++t) kd[t] = __ldcg(krow + t);
#pragma unroll
    for (int i = 0; i < P; ++i) {
      const int pv = min(tile + warp * P + i, p_end - 1);
      vd[i] = __ldcg(reinterpret_cast<const float2*>(vb + (int64_t)pv * kHeadDim) + lane);
    }
  };
  // one tile: scores, online-softmax update, weighted values
  auto use = [&](int tile, const float4 (&kd)[D / 4], const float2 (&vd)[P]) {
    const bool live = tile + warp * P + pi < p_end;  // this lane's position exists
    const int nvalid = min(P, max(0, p_end - tile - warp * P));  // positions of this warp's tile
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float sc = 0.f;
#pragma unroll
      for (int t = 0; t < D / 4; ++t) {
        sc = fmaf(qs[g][4 * t], kd[t].x, sc);
        sc = fmaf(qs[g][4 * t + 1], kd[t].y, sc);
        sc = fmaf(qs[g][4 * t + 2], kd[t].z, sc);
        sc = fmaf(qs[g][4 * t + 3], kd[t].w, sc);
      }
#pragma unroll
      for (int off = 1; off < L; off <<= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
      sc = live ? sc : -INFINITY;
      float tm = sc;
#pragma unroll
      for (int off = L; off < 32; off <<= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, off));
      const float mn = fmaxf(m[g], tm);
      const float corr = m[g] == mn ? 1.f : exp2f(m[g] - mn);
      const float w = sc == -INFINITY ? 0.f : exp2f(sc - mn);
      float ws = w;
#pragma unroll
      for (int off = L; off < 32; off <<= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
      l[g] = fmaf(l[g], corr, ws);  // offsets >= L: one lane per position took part
      float2 acc = make_float2(o[g].x * corr, o[g].y * corr);
#pragma unroll
      for (int i = 0; i < P; ++i) {
        const float wi = __shfl_sync(0xffffffffu, w, i * L);
        if (i < nvalid) {
          acc.x = fmaf(wi, vd[i].x, acc.x);
          acc.y = fmaf(wi, vd[i].y, acc.y);
        }
      }
      o[g] = acc;
      m[g] = mn;
    }
  };
  if (p_begin >= p_end) return;
#pragma unroll
  for (int d = 0; d < DEP; ++d)
    if (p_begin + d * kTile < p_end) load(p_begin + d * kTile, kr[d], vr[d]);
  for (int base = p_begin; base < p_end; base += DEP * kTile) {
#pragma unroll
    for (int d = 0; d < DEP; ++d) {
      const int tile = base + d * kTile;
      if (tile >= p_end) break;
      use(tile, kr[d], vr[d]);
      if (tile + DEP * kTile < p_end) load(tile + DEP * kTile, kr[d], vr[d]);  // refill this slot
    }
  }
}

// q head g of kv head kvh, pre-scaled, as this lane's key-dim slice.
template <int G>
__device__ __forceinline__ void attn_load_q(const float* qb, int kvh, int lane, float scale,
                                            float (&qs)[G][AttnLayout<G>::D]) {
  using A = AttnLayout<G>;
  const int j = lane % A::L;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float4* src = reinterpret_cast<const float4*>(qb + (int64_t)(kvh * G + g) * kHeadDim + j * A::D);
#pragma unroll
    for (int t = 0; t < A::D / 4; ++t) {
      const float4 v = __ldcg(src + t);
      qs[g][4 * t] = v.x * scale;
      qs[g][4 * t + 1] = v.y * scale;
      qs[g][4 * t + 2] = v.z * scale;
      qs[g][4 * t + 3] = v.w * scale;
    }
  }
}

}  // namespace attn
}  // namespace qd
