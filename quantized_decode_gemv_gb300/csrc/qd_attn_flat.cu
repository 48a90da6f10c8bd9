// Split-KV decode attention with a flat, even split, for long walks over the cache
// (llmoxide blog s5 and dasLLAMA 8.7.1.6.2 attention: scores q.k / sqrt(head_dim),
// softmax over positions 0..pos, weighted sum of the value rows).
//
// The cluster kernel gives each (sequence, kv head) pair S <= 8 CTAs.  When the pairs are
// few and the walks long (32 kv heads at batch 1 and context 4096: 32 pairs of 4096
// positions, 67 MB of f32 cache per layer) that grid cannot cover 152 SMs evenly, and the
// walk must keep enough bytes in flight per SM to run at HBM speed.  Here:
//  * every pair's positions 0..pos are cut into tiles of 64 positions; the tiles of all
//    pairs are laid end to end (sequence-major, then kv head) and CTA i of a grid of C
//    CTAs (one per SM) takes tiles [floor(i T / C), floor((i+1) T / C)), so every SM
//    streams the same number of bytes whatever the pair count;
//  * a tile's key rows and value rows are each one contiguous run of the cache (64 rows
//    of 256 bytes).  One thread of a producer warp copies them into a ring of NS stages
//    in shared memory with two bulk copies (cp.async.bulk, completion counted in bytes on
//    the stage's "full" mbarrier), up to NS tiles ahead; eight consumer warps take 8
//    positions each of every tile and release the stage on its "empty" mbarrier;
//  * scores: 8 lanes per key row (8 dims each, three shuffles), 4 rows per step; one
//    online-softmax update per tile and q head (log2 units: q is pre-scaled by
//    log2(e) / sqrt(head_dim)); values: lane j holds dims 2j, 2j+1 of the output;
//  * where its run leaves a pair, each warp parks its online-softmax state (m, l, o) in a
//    shared-memory slot area and walks on, with no barrier.  At the end of the run the CTA
//    merges its warps per pair, stores one partial per (CTA, pair) in a global workspace
//    and counts itself in on the arrival counter of every pair the run covered.  The CTA
//    that completes a pair's count merges that pair's CTA partials in CTA order (the same
//    log-sum-exp merge, so the result does not depend on arrival order), writes the output
//    and sets the counter back to zero for the next launch.  No CTA waits for another.
// Every mbarrier wait is bounded: on a timeout the kernel sets kErrTimeout, stops
// waiting and computing (its output is then undefined) and still reaches every barrier.
#include <cmath>
#include <type_traits>

#include "qd_attn.cuh"
#include "qd_tc.cuh"

namespace qd {
namespace {

using namespace attn;

constexpr int kFlatRows = 8;  // positions per consumer warp per tile
// The shape of a launch: W consumer warps take a tile of W x 8 positions, whose key rows
// and value rows (each one contiguous run of the cache) fill one stage of an NS-stage
// ring.  Eight warps (64 positions, f32 4 x 32 KB, binary16 6 x 16 KB) except for a
// binary16 cache with one query head per kv head: there the consumer's dependent chain,
// not the bytes, sets the pace, so sixteen warps (128 positions, 4 x 32 KB) run two tiles'
// chains each (120 registers: 17 warps fill the register file).
template <int G, typename T>
struct FlatShape {
  static constexpr int W = (G == 1 && sizeof(T) == 2) ? 16 : 8;
  static constexpr int kTile = W * kFlatRows;       // positions per tile
  static constexpr int kHalf = kTile * kHeadDim;    // elements of one tile's key (or value) rows
  static constexpr int kStageBytes = 2 * kHalf * (int)sizeof(T);  // key rows, then value rows
  static constexpr int NS = kStageBytes >= 32768 ? 4 : 6;
  static constexpr int kThreads = (W + 1) * 32;     // + the producer warp
};
constexpr int kPartFloats = 2 + kHeadDim;            // one head's partial: m, l, o[64]
constexpr int kFlatSlotHeads = 8;  // parked (pair, head) warp states a CTA holds before settling them
using tc::mbar_arrive;  // mbarrier helpers: every wait is a bounded poll (tc::kSpinLimit)
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
// `bytes` (a multiple of 16) from global `src` to shared `dst`, counted on `mbar`
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  tc::bulk_copy_g2s(dst, src, bytes, mbar);
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
template <int W>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(W * 32) : "memory");
}

struct Cursor {
  int b, kvh, tt;  // sequence, kv head, tile of that pair
};

// K, V rows of the cache's element type (f32, or binary16 read back exactly), widened to
// f32 in the consumers.
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __half* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float2 load2(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load2(const __half* p) { return __half22float2(*reinterpret_cast<const __half2*>(p)); }

// Packed pair arithmetic: fma.rn.f32x2 rounds each half as fmaf does.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<const float2*>(&r);
}

template <int G, typename CT>
__global__ void __launch_bounds__(FlatShape<G, CT>::kThreads, 1)
    k_attn_flat(const float* __restrict__ q, int64_t q_stride, const CT* __restrict__ kc,
                const CT* __restrict__ vc, int64_t cache_batch_stride, int n_heads, int n_kv,
                const int32_t* __restrict__ pos, int max_ctx, int batch, float scale, float* __restrict__ out,
                float* __restrict__ ws, unsigned int* __restrict__ cnt, uint32_t* err) {
  using Shape = FlatShape<G, CT>;
  constexpr int W = Shape::W, NS = Shape::NS, kStageBytes = Shape::kStageBytes;
  constexpr int kFlatTile = Shape::kTile, kFlatHalf = Shape::kHalf;
  extern __shared__ __align__(128) float ring[];  // [NS][key rows | value rows] of CT, then the slots
  __shared__ __align__(8) uint64_t full_bar[NS], empty_bar[NS];
  __shared__ int s_n[QD_MAX_BATCH], s_tiles[QD_MAX_BATCH];
  __shared__ int64_t s_off[QD_MAX_BATCH + 1];  // tiles before sequence b (all its kv heads)
  __shared__ int s_pairs[kFlatSlotHeads], s_last[kFlatSlotHeads];  // pairs of this run not yet settled
  constexpr int kFuse = G == 1 ? 2 : 1;  // tiles a consumer step may take (see use_tiles)
  __shared__ __align__(16) float2 s_w[W][G][kFuse * kFlatRows];  // a warp's weights of a step, each twice
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring_s = (uint32_t)__cvta_generic_to_shared(ring);
  const uint32_t full0 = (uint32_t)__cvta_generic_to_shared(full_bar);
  const uint32_t empty0 = (uint32_t)__cvta_generic_to_shared(empty_bar);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, W);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // Before the dependency wait: the positions (advanced by the previous step) and every
  // cache row before them (written by earlier steps) are final once this kernel runs,
  // because each kernel of the step lets its successor launch only after its own wait, so
  // the kernel two launches back has completed.  q and the row at each position come
  // from the QKV projection that precedes this kernel.
  if (threadIdx.x < batch) {
    const int p = pos[threadIdx.x];
    const bool ok = p >= 0 && p < max_ctx;
    s_n[threadIdx.x] = ok ? p + 1 : 0;
    s_tiles[threadIdx.x] = ok ? p / kFlatTile + 1 : 0;
    if (!ok && err && blockIdx.x == 0) atomicOr(err, kErrPosition);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t a = 0;
    for (int b = 0; b < batch; ++b) {
      s_off[b] = a;
      a += (int64_t)s_tiles[b] * n_kv;
    }
    s_off[batch] = a;
  }
  __syncthreads();
  const int64_t T = s_off[batch];
  const int64_t C = min((int64_t)gridDim.x, T);  // CTAs with work: each gets >= 1 tile
  if ((int64_t)blockIdx.x >= C || warp < W) {
    pdl_wait();     // q and the rows at the current positions come from the QKV projection
    pdl_trigger();  // let the next kernel start its weight prefetch
    // a sequence whose position is out of range has no tiles: its rows are zeros
    for (int b = 0; b < batch; ++b)
      if (s_n[b] == 0 && b % (int)gridDim.x == (int)blockIdx.x && warp < W)
        for (int t = threadIdx.x; t < n_heads * kHeadDim; t += W * 32)
          out[(int64_t)b * n_heads * kHeadDim + t] = 0.f;
  }
  if ((int64_t)blockIdx.x >= C) return;
  const int64_t t_begin = (int64_t)blockIdx.x * T / C, t_end = ((int64_t)blockIdx.x + 1) * T / C;
  const int nst = (int)(t_end - t_begin);
  auto advance = [&](Cursor& c) {
    if (++c.tt == s_tiles[c.b]) {
      c.tt = 0;
      if (++c.kvh == n_kv) {
        c.kvh = 0;
        do {
          ++c.b;
        } while (c.b < batch && s_tiles[c.b] == 0);
      }
    }
  };
  Cursor start;
  {
    int b = 0;
    while (b + 1 < batch && s_off[b + 1] <= t_begin) ++b;
    const int64_t rem = t_begin - s_off[b];
    start = Cursor{b, (int)(rem / s_tiles[b]), (int)(rem % s_tiles[b])};
  }

  if (warp == W) {
    // ---- producer: one thread copies tile after tile into the ring, starting before the
    // dependency wait; it waits only before a pair's last tile (the row the QKV
    // projection appends)
    if (lane == 0) {
      Cursor c = start;
      int slot = 0, issued = 0;
      uint32_t use = 0;  // completed uses of this slot before this one
      bool waited = false;
      for (int s = 0; s < nst; ++s) {
        if (use > 0 && !mbar_wait(empty0 + 8 * slot, (use - 1) & 1u)) {
          if (err) atomicOr(err, kErrTimeout);
          break;  // the consumers then time out on this stage's full barrier
        }
        if (!waited && c.tt == s_tiles[c.b] - 1) {
          pdl_wait();
          waited = true;
        }
        const int p0 = c.tt * kFlatTile;
        const int rows = min(kFlatTile, s_n[c.b] - p0);
        const int64_t off =
            (int64_t)c.b * cache_batch_stride + ((int64_t)c.kvh * max_ctx + p0) * kHeadDim;  // row p0 of the pair
        const uint32_t bytes = (uint32_t)rows * kHeadDim * (uint32_t)sizeof(CT);
        const uint32_t dst = ring_s + (uint32_t)slot * kStageBytes;
        mbar_arrive_expect_tx(full0 + 8 * slot, 2 * bytes);
        bulk_copy(dst, kc + off, bytes, full0 + 8 * slot);
        bulk_copy(dst + kFlatHalf * (uint32_t)sizeof(CT), vc + off, bytes, full0 + 8 * slot);
        ++issued;
        advance(c);
        if (++slot == NS) {
          slot = 0;
          ++use;
        }
      }
      // stay until the last copy into each slot has landed: no copy may target the
      // CTA's shared memory after it exits
      for (int k = max(0, issued - NS); k < issued; ++k)
        if (!mbar_wait(full0 + 8 * (k % NS), (uint32_t)(k / NS) & 1u) && err) atomicOr(err, kErrTimeout);
    }
    return;
  }

  // ---- consumers
  auto cta_of = [&](int64_t x) { return (int)(((x + 1) * C + T - 1) / T - 1); };  // CTA holding tile x
  const int j = lane & 7, pi = lane >> 3;  // dim slice (dims 4j.., 32+4j..) and row of a step
  float2 qs[G][4];  // (scaled) q dims 4j..4j+3, 32+4j..32+4j+3 as pairs
  float m[G], l[G];  // l: the weight sum of the rows this lane owned (see use_tiles)
  float2 o[G];
  auto start_pair = [&](const Cursor& c) {
    const float* qb = q + (int64_t)c.b * q_stride + (int64_t)c.kvh * G * kHeadDim;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(qb + g * kHeadDim + 4 * j));
      const float4 bq = __ldcg(reinterpret_cast<const float4*>(qb + g * kHeadDim + 32 + 4 * j));
      qs[g][0] = make_float2(a.x * scale, a.y * scale);
      qs[g][1] = make_float2(a.z * scale, a.w * scale);
      qs[g][2] = make_float2(bq.x * scale, bq.y * scale);
      qs[g][3] = make_float2(bq.z * scale, bq.w * scale);
      m[g] = -INFINITY;
      l[g] = 0.f;
      o[g] = make_float2(0.f, 0.f);
    }
  };
  // This warp's 8 positions of NT consecutive tiles of one pair (stages s, s + 1, ...).
  // Lane (pi, j) forms the partial dot products of rows pi and 4 + pi of each tile over its
  // dims; exchanges with lanes j ^ 1 (and j ^ 2 for two tiles) leave each lane one row to
  // finish (row pi or 4 + pi by bit 0 of j, the tile by bit 1), so the max, the weight
  // and the weight sum take one value per lane, and lanes j < 2 NT own distinct rows.
  // The weights reach every lane through shared memory as (w, w) pairs and meet the value
  // rows in packed FMAs.  Rows past the pair's last position hold stale ring data: their
  // scores are -inf and their values zero.  Two tiles at a time give a warp two
  // independent chains of shared loads, shuffles and FMAs where one head per kv head
  // would leave it one.
  auto use_tiles = [&](auto ntc, int s, const Cursor& c) {
    constexpr int NT = decltype(ntc)::value;
    const CT* kt[NT];
    int live_rows[NT];  // may be <= 0 or > 8
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      kt[t] = reinterpret_cast<const CT*>(reinterpret_cast<const uint8_t*>(ring) + ((s + t) % NS) * kStageBytes) +
              warp * kFlatRows * kHeadDim;
      live_rows[t] = s_n[c.b] - (c.tt + t) * kFlatTile - warp * kFlatRows;
    }
    const bool odd = j & 1, hi = NT == 2 && (j & 2);
    const int r = odd ? 4 + pi : pi;  // the row this lane finishes, of tile `hi`
    const bool owner = j < 2 * NT;
    const bool live = r < (hi ? live_rows[NT - 1] : live_rows[0]);
    float4 ka[NT][2], kb[NT][2];  // rows pi and 4 + pi: dims 4j.., 32 + 4j..
    float2 v[NT][kFlatRows];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ka[t][h] = load4(kt[t] + (4 * h + pi) * kHeadDim + 4 * j);
        kb[t][h] = load4(kt[t] + (4 * h + pi) * kHeadDim + 32 + 4 * j);
      }
#pragma unroll
      for (int i = 0; i < kFlatRows; ++i) v[t][i] = load2(kt[t] + kFlatHalf + i * kHeadDim + 2 * lane);
      if (live_rows[t] < kFlatRows) {  // the pair's last tile (warp-uniform)
#pragma unroll
        for (int i = 0; i < kFlatRows; ++i)
          if (i >= live_rows[t]) v[t][i] = make_float2(0.f, 0.f);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float x[NT];  // after the first exchange: row r of tile t, summed over j and j ^ 1
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float sp[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float2 p = make_float2(qs[g][0].x * ka[t][h].x, qs[g][0].y * ka[t][h].y);
          p = ffma2(qs[g][1], make_float2(ka[t][h].z, ka[t][h].w), p);
          p = ffma2(qs[g][2], make_float2(kb[t][h].x, kb[t][h].y), p);
          p = ffma2(qs[g][3], make_float2(kb[t][h].z, kb[t][h].w), p);
          sp[h] = p.x + p.y;
        }
        x[t] = (odd ? sp[1] : sp[0]) + __shfl_xor_sync(0xffffffffu, odd ? sp[0] : sp[1], 1);
      }
      float sc;
      if constexpr (NT == 2)
        sc = (hi ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, hi ? x[0] : x[1], 2);
      else
        sc = x[0] + __shfl_xor_sync(0xffffffffu, x[0], 2);
      sc += __shfl_xor_sync(0xffffffffu, sc, 4);
      sc = live ? sc : -INFINITY;
      float tm = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 1));
      if constexpr (NT == 2) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
      const float mn = fmaxf(m[g], tm);
      const float corr = m[g] == mn ? 1.f : exp2f(m[g] - mn);
      const float w = live ? exp2f(sc - mn) : 0.f;
      l[g] = fmaf(l[g], corr, owner ? w : 0.f);
      if (owner) s_w[warp][g][(hi ? kFlatRows : 0) + r] = make_float2(w, w);
      __syncwarp();
      const float4* wq = reinterpret_cast<const float4*>(s_w[warp][g]);
      float2 acc[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        acc[t] = t == 0 ? ffma2(o[g], make_float2(corr, corr), make_float2(0.f, 0.f)) : make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kFlatRows / 2; ++i) {
          const float4 w2 = wq[t * kFlatRows / 2 + i];
          acc[t] = ffma2(make_float2(w2.x, w2.y), v[t][2 * i], acc[t]);
          acc[t] = ffma2(make_float2(w2.z, w2.w), v[t][2 * i + 1], acc[t]);
        }
      }
      if constexpr (NT == 2) acc[0] = make_float2(acc[0].x + acc[1].x, acc[0].y + acc[1].y);
      o[g] = acc[0];
      m[g] = mn;
    }
  };
  // Pairs this run has left and not yet settled: each warp parks its state for pair slot t
  // in shared memory (slots after the ring: m[W][G], l[W][G], o[W][G][64] per slot).
  constexpr int kSlots = kFlatSlotHeads / G > 0 ? kFlatSlotHeads / G : 1;
  constexpr int kSlotFloats = W * G * kPartFloats;
  float* slots = ring + NS * (kStageBytes / 4);
  int npairs = 0;  // the same in every consumer thread: all walk the same tiles
  auto end_pair = [&](const Cursor& c) {
    float* sl = slots + npairs * kSlotFloats;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      // the weight sum over the warp's rows: each row's weights were taken by one lane
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], off);
      if (lane == 0) {
        sl[warp * G + g] = m[g];
        sl[W * G + warp * G + g] = l[g];
      }
      reinterpret_cast<float2*>(sl + 2 * W * G + (warp * G + g) * kHeadDim)[lane] = o[g];
    }
    if (warp == 0 && lane == 0) s_pairs[npairs] = c.b * n_kv + c.kvh;
    ++npairs;
  };
  auto pair_ctas = [&](int pair, int& i0, int& i1) {
    const int b = pair / n_kv, kvh = pair % n_kv;
    const int64_t first = s_off[b] + (int64_t)kvh * s_tiles[b];
    i0 = cta_of(first);
    i1 = cta_of(first + s_tiles[b] - 1);
  };
  // Settle the parked pairs: merge each pair's W warp states into this CTA's partial (m, l,
  // o) in the global workspace (slot i + pair), count in on the pair's arrival counter,
  // and, for each pair this CTA completes, merge the pair's CTA partials i0..i1 and write
  // the output.  That merge is spread over the warps: warp w takes head w % G and the CTAs
  // i0 + w / G, i0 + w / G + S, ... (S = W / G subsets), eight partials' loads at a time;
  // the subsets are then combined in subset order.
  auto settle = [&]() {
    consumers_sync<W>();  // every warp's parked states are in shared memory
    const int np = npairs;
    for (int it = warp; it < np * G; it += W) {
      const int t = it / G, g = it % G;
      const float* sl = slots + t * kSlotFloats;
      float mx = -INFINITY;
#pragma unroll
      for (int w2 = 0; w2 < W; ++w2) mx = fmaxf(mx, sl[w2 * G + g]);
      float lt = 0.f;
      float2 ot = make_float2(0.f, 0.f);
#pragma unroll
      for (int w2 = 0; w2 < W; ++w2) {
        const float mw = sl[w2 * G + g];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - mx);  // a warp may have seen no position
        lt = fmaf(sl[W * G + w2 * G + g], f, lt);
        const float2 ow = reinterpret_cast<const float2*>(sl + 2 * W * G + (w2 * G + g) * kHeadDim)[lane];
        ot.x = fmaf(ow.x, f, ot.x);
        ot.y = fmaf(ow.y, f, ot.y);
      }
      float* part = ws + (((int64_t)blockIdx.x + s_pairs[t]) * G + g) * kPartFloats;
      if (lane == 0) {
        part[0] = mx;
        part[1] = lt;
      }
      reinterpret_cast<float2*>(part + 2)[lane] = ot;
    }
    consumers_sync<W>();  // the CTA's partial stores are ordered before the counting threads' fences
    if (threadIdx.x < np) {
      int i0, i1;
      pair_ctas(s_pairs[threadIdx.x], i0, i1);
      fence_acq_rel_gpu();  // release: this CTA's partials before its count
      s_last[threadIdx.x] = atomicAdd(cnt + s_pairs[threadIdx.x], 1u) == (unsigned)(i1 - i0);
      fence_acq_rel_gpu();  // acquire: the partials of the CTAs counted before this one
    }
    consumers_sync<W>();
    constexpr int S = W / G;  // CTA subsets per head in the final merge
    for (int t = 0; t < np; ++t) {
      if (!s_last[t]) continue;
      const int pair = s_pairs[t];
      int i0, i1;
      pair_ctas(pair, i0, i1);
      float* scratch = slots;  // [W][kPartFloats]: the parked states are no longer needed
      if (warp < G * S) {
        const int g = warp % G, sub = warp / G;
        float mx = -INFINITY, lt = 0.f;
        float2 acc = make_float2(0.f, 0.f);
        for (int i = i0 + sub; i <= i1; i += 8 * S) {
          float mk[8], lk[8];
          float2 ok[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {  // the loads of eight partials, then their use
            const int ii = i + u * S;
            const float* part = ws + (((int64_t)(ii <= i1 ? ii : i) + pair) * G + g) * kPartFloats;
            mk[u] = ii <= i1 ? __ldcg(part) : -INFINITY;
            lk[u] = __ldcg(part + 1);
            ok[u] = __ldcg(reinterpret_cast<const float2*>(part + 2) + lane);
          }
          float mb = mx;
#pragma unroll
          for (int u = 0; u < 8; ++u) mb = fmaxf(mb, mk[u]);
          const float corr = mx == mb ? 1.f : exp2f(mx - mb);
          lt *= corr;
          acc.x *= corr;
          acc.y *= corr;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float f = mk[u] == -INFINITY ? 0.f : exp2f(mk[u] - mb);
            lt = fmaf(lk[u], f, lt);
            acc.x = fmaf(ok[u].x, f, acc.x);
            acc.y = fmaf(ok[u].y, f, acc.y);
          }
          mx = mb;
        }
        if (lane == 0) {
          scratch[warp * kPartFloats] = mx;
          scratch[warp * kPartFloats + 1] = lt;
        }
        reinterpret_cast<float2*>(scratch + warp * kPartFloats + 2)[lane] = acc;
      }
      consumers_sync<W>();
      if (warp < G) {
        const int g = warp;
        float mx = -INFINITY;
#pragma unroll
        for (int sub = 0; sub < S; ++sub) mx = fmaxf(mx, scratch[(sub * G + g) * kPartFloats]);
        float lt = 0.f;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int sub = 0; sub < S; ++sub) {
          const float* sp = scratch + (sub * G + g) * kPartFloats;
          const float f = sp[0] == -INFINITY ? 0.f : exp2f(sp[0] - mx);  // a subset may be empty
          lt = fmaf(sp[1], f, lt);
          const float2 so2 = reinterpret_cast<const float2*>(sp + 2)[lane];
          acc.x = fmaf(so2.x, f, acc.x);
          acc.y = fmaf(so2.y, f, acc.y);
        }
        const int b = pair / n_kv, kvh = pair % n_kv;
        float2* dst = reinterpret_cast<float2*>(out + ((int64_t)b * n_heads + kvh * G + g) * kHeadDim);
        dst[lane] = make_float2(acc.x / lt, acc.y / lt);
      }
      if (threadIdx.x == 0) cnt[pair] = 0u;
      consumers_sync<W>();  // the scratch is reused by the next pair
    }
    npairs = 0;
  };

  Cursor cc = start, cur{-1, -1, 0};
  bool bad = false;
  for (int s = 0; s < nst;) {
    if (!bad && !mbar_wait(full0 + 8 * (s % NS), (uint32_t)(s / NS) & 1u)) {
      bad = true;
      if (err && lane == 0) atomicOr(err, kErrTimeout);
    }
    if (cc.b != cur.b || cc.kvh != cur.kvh) {
      if (cur.b >= 0) {
        end_pair(cur);
        if (npairs == kSlots) settle();  // (short pairs: more in one run than the slots hold)
      }
      cur = cc;
      start_pair(cc);
    }
    // take the next tile too when it is this run's and the same pair's (the same in every
    // consumer thread)
    const bool two = kFuse == 2 && s + 1 < nst && cc.tt + 1 < s_tiles[cc.b];
    if (two && !bad && !mbar_wait(full0 + 8 * ((s + 1) % NS), (uint32_t)((s + 1) / NS) & 1u)) {
      bad = true;
      if (err && lane == 0) atomicOr(err, kErrTimeout);
    }
    if (!bad) {
      if (two)
        use_tiles(std::integral_constant<int, kFuse>{}, s, cc);
      else
        use_tiles(std::integral_constant<int, 1>{}, s, cc);
    }
    __syncwarp();
    if (lane == 0) {  // this warp is done with the slots
      mbar_arrive(empty0 + 8 * (s % NS));
      if (two) mbar_arrive(empty0 + 8 * ((s + 1) % NS));
    }
    advance(cc);
    if (two) advance(cc);
    s += two ? 2 : 1;
  }
  if (cur.b >= 0) {
    end_pair(cur);
    settle();
  }
}

// ring stages, then the parked warp states (at least one pair's worth)
template <int G, typename T>
constexpr int flat_smem_bytes() {
  using Shape = FlatShape<G, T>;
  return Shape::NS * Shape::kStageBytes +
         (kFlatSlotHeads / G > 0 ? kFlatSlotHeads / G : 1) * Shape::W * G * kPartFloats * 4;
}

template <int G, typename T>
cudaError_t launch_flat_gt(cudaLaunchConfig_t& cfg, const float* q, int64_t q_stride, const void* kc,
                           const void* vc, int64_t cache_batch_stride, int n_heads, int n_kv, const int32_t* pos,
                           int max_ctx, int batch, float scale, float* out, float* ws, unsigned int* cnt,
                           uint32_t* err) {
  auto kern = k_attn_flat<G, T>;
  constexpr int smem = flat_smem_bytes<G, T>();
  static_assert(smem <= 220 * 1024, "ring and parked states exceed the shared memory of a CTA");
  static bool done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!done[dev]) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    done[dev] = true;
  }
  cfg.blockDim = dim3(FlatShape<G, T>::kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  return cudaLaunchKernelEx(&cfg, kern, q, q_stride, static_cast<const T*>(kc), static_cast<const T*>(vc),
                            cache_batch_stride, n_heads, n_kv, pos, max_ctx, batch, scale, out, ws, cnt, err);
}

template <int G>
cudaError_t launch_flat_g(cudaLaunchConfig_t& cfg, bool kv_f16, const float* q, int64_t q_stride, const void* kc,
                          const void* vc, int64_t cache_batch_stride, int n_heads, int n_kv, const int32_t* pos,
                          int max_ctx, int batch, float scale, float* out, float* ws, unsigned int* cnt,
                          uint32_t* err) {
  return kv_f16 ? launch_flat_gt<G, __half>(cfg, q, q_stride, kc, vc, cache_batch_stride, n_heads, n_kv, pos, max_ctx,
                                            batch, scale, out, ws, cnt, err)
                : launch_flat_gt<G, float>(cfg, q, q_stride, kc, vc, cache_batch_stride, n_heads, n_kv, pos, max_ctx,
                                           batch, scale, out, ws, cnt, err);
}

}  // namespace

int attn_flat_ctas() { return attn_sm_count(); }

size_t attn_flat_ws_floats(int n_heads, int n_kv, int batch, int ctas) {
  const int G = n_heads / n_kv;
  return (size_t)(ctas + n_kv * batch) * G * kPartFloats;
}

bool attn_use_flat(int n_kv, int batch, int max_ctx) {
  // f32 key and value rows of every pair at full context: 512 bytes per position
  return (int64_t)n_kv * batch * max_ctx * 2 * kHeadDim * 4 >= kAttnFlatMinBytes;
}

qd_status launch_attention_flat(const float* q, int64_t q_stride, const void* kc, const void* vc, bool kv_f16,
                                int64_t cache_batch_stride, float* out, int n_heads, int n_kv, int head_dim,
                                const int32_t* pos, int max_ctx, int batch, int ctas, float* ws, unsigned int* cnt,
                                uint32_t* err, cudaStream_t stream, bool pdl) {
  if (head_dim != kHeadDim || n_kv < 1 || n_heads % n_kv || batch < 1 || batch > QD_MAX_BATCH || ctas < 1)
    return QD_ERR_SHAPE;
  const int G = n_heads / n_kv;
  const float scale = 1.4426950408889634f / sqrtf((float)head_dim);  // scores in log2 units
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t rc = cudaErrorInvalidValue;
#define QD_FLAT_G(GG)                                                                                            \
  case GG:                                                                                                       \
    rc = launch_flat_g<GG>(cfg, kv_f16, q, q_stride, kc, vc, cache_batch_stride, n_heads, n_kv, pos, max_ctx, batch, \
                           scale, out, ws, cnt, err);                                                            \
    break;
  switch (G) {
    QD_FLAT_G(1)
    QD_FLAT_G(2)
    QD_FLAT_G(3)
    QD_FLAT_G(4)
    QD_FLAT_G(5)
    QD_FLAT_G(6)
    QD_FLAT_G(7)
    QD_FLAT_G(8)
    default: return QD_ERR_UNSUPPORTED;
  }
#undef QD_FLAT_G
  return rc == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

}  // namespace qd
