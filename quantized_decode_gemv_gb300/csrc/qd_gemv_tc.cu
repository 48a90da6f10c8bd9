// Batched q_gemv on the 5th-generation tensor cores: per-row INT8 weights, 9-16 batch
// rows (independent sequences).
//
// y[b][r] = s_r * sum_c q[r][c] x[b][c]  (minillm-cpp README "Quantization": symmetric
// per-row INT8, one f32 scale per output row; the row dot of llmoxide blog s1).  With
// 16 sequences the product is a small dense contraction (M = rows, N = 16, K = cols), so
// it runs as tcgen05.mma kind::f16 with an f32 accumulator in tensor memory.
//
//  * B (N = 32 x K) is x: each sequence's K-slice is scaled by a power of two (its largest
//    |x| lands in [2^13, 2^14), exact) and split into an f16 high part and the f16 rounding
//    of the remainder, columns 0-15 high, 16-31 low.  hi + lo holds x to about 2^-22
//    relative; the tensor core's products of f16 values are exact and sum in f32.  B is
//    staged once per CTA in shared memory (K-major, no-swizzle canonical layout).
//  * A (M = 128 rows x 16 K per instruction) is the weight tile, held in tensor memory
//    (row r in lane r, two f16 per 32-bit column).  Warp-specialised pipeline over stages
//    of 128 columns: eight converter warps stream the int8 codes through a per-thread
//    cp.async ring; thread (w, l) owns row 32 (w % 4) + l of the tile (a warp reaches only
//    its quarter of the tensor-memory lanes) and half of each stage: it copies its 64
//    codes, converts them exactly to f16 (q ^ 0x80 placed in the mantissa of 1024, then
//    1152 subtracted) and writes them with one tcgen05.st into one of five A stages in
//    tensor memory; each warp then arrives once on the stage's "full" mbarrier.  Two MMA
//    lanes (lane 0 of warps 8 and 9) take a tile's even and odd stages: each waits for
//    "full", issues the stage's eight MMAs (A from tensor memory, B from shared memory)
//    into its half of the tile's accumulator and commits them to the stage's "empty"
//    mbarrier, which the converters wait for before refilling it.  (Per stage, the MMA
//    issue and the converters each pay a fixed hand-off cost; 128-column stages halve it
//    per byte, and a second issuing thread keeps about 1.7 times the MMAs in flight.)
//    Tiles alternate between two accumulators in tensor memory; after its last stage of a
//    tile each MMA lane commits to the accumulator's "done" barrier, and converter warps
//    0-3 read both halves out (tcgen05.ld, one row per thread) a few stages into the next
//    tile, then arrive on its "drained" barrier.
//  * Many row tiles: one cluster-free CTA per SM walks tiles cta, cta + CTAs, ... with the
//    weight ring running on across tiles.  Few row tiles: the columns split over up to 8
//    CTAs of a thread-block cluster (one tile each); the partials are summed through
//    distributed shared memory in rank order (deterministic) at the end.
//  * Epilogue: s_r, then store, accumulate into y, or SwiGLU of interleaved gate/up rows.
//
// Every mbarrier wait is bounded; on a timeout the kernel sets kErrTimeout, stops issuing
// MMAs, finishes its loops without waiting, frees its tensor memory and returns.
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "qd_internal.cuh"
#include "qd_tc.cuh"

namespace qd {
namespace tc_gemv {

using namespace tc;

constexpr int kM = 128;       // weight rows per tile (the MMA's M)
constexpr int kN = 32;        // B columns: 16 sequences x (high, low)
constexpr int kNB = 16;       // sequences
constexpr int kKT = 128;      // K elements per pipeline stage
#ifndef QD_TC_CONV_WARPS
#define QD_TC_CONV_WARPS 8
#endif
constexpr int kConvWarps = QD_TC_CONV_WARPS;  // converter warps; warps 0-3 also read the accumulators
constexpr int kConv = 32 * kConvWarps;        // converter threads
constexpr int kEpi = 128;                     // accumulator readout threads (TMEM lanes 0-127)
constexpr int kMmaWarp = kConvWarps;          // the two warps after the converters issue the MMAs
constexpr int kThreads = kConv + 64;
static_assert(kConvWarps == 4 || kConvWarps == 8, "converter warps");
constexpr int kMaxKc = 2048;  // K elements per CTA at most (shared memory for B)
constexpr int kRing = 5;      // int8 weight stages in the cp.async ring
constexpr int kEpiDelay = 2;  // stages into the next tile before the previous one is read out
constexpr int kMaxCluster = 8;
// Tensor memory: two tiles' accumulators, each two 32-column f32 halves (one per MMA lane:
// lane 0 takes a tile's even stages, lane 1 its odd ones; the epilogue adds the halves),
// then kNA f16 A stages of kKT / 2 columns (row r of the tile in lane r, two K elements per
// 32-bit column).
constexpr int kNA = 5;
constexpr uint32_t kAccCols = 128;
constexpr uint32_t kACols = kKT / 2;
constexpr uint32_t kTmemCols = 512;
static_assert(kAccCols + kNA * kACols <= kTmemCols, "tensor memory columns");

constexpr uint32_t kI8Bytes = kM * kKT;             // one int8 weight stage
constexpr uint32_t kPartBytes = kNB * kM * 4;       // the CTA's f32 partial tile (split-K)
constexpr int kChunks = kM * kKT / 16 / kConv;      // 16-byte chunks per converter thread and stage
// Converter thread (warp w, lane l) owns row 32 (w % 4) + l of the tile (a warp reaches only
// its quarter of the tensor-memory lanes) and K elements [kPartK (w / 4), + kPartK) of
// each stage: it copies, converts and stores exactly those.
constexpr int kPartK = kKT / (kConvWarps / 4);
static_assert(kConvWarps == 8 && kPartK == 64 && kChunks == 4, "converter layout");

struct Params {
  const int8_t* codes;
  const float* row_scale;
  int64_t rows, cols;
  const float* x;
  float* y;
  int batch;
  int kc;  // columns per CTA
  int mode;
  uint32_t* err;
};

__host__ __device__ constexpr uint32_t b_bytes(int kc) { return (uint32_t)kN * (uint32_t)kc * 2u; }
// dynamic shared memory, from its first 128-byte boundary: B | int8 ring | partial tile
__host__ __device__ constexpr uint32_t smem_bytes(int kc) { return 128 + b_bytes(kc) + kRing * kI8Bytes + kPartBytes; }

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B, both K-major, N, M.
constexpr uint32_t kIdesc = idesc_f16(kM, kN);

// D (tensor memory) += A (tensor memory, K-major: row i in lane i) x B (shared memory).
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t accumulate) {
  mma_f16_ts(tmem_d, tmem_a, bdesc, kIdesc, accumulate);
}

__device__ __forceinline__ void conv_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kConv) : "memory"); }

__global__ void __launch_bounds__(kThreads, 1) k_gemv_tc_i8(const Params p) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bar_full[kNA], bar_empty[kNA], bar_done[2], bar_drained[2];
  __shared__ uint32_t tmem_base;
  __shared__ float unscale[kNB];
  __shared__ float wmax[kNB];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t tiles = (p.rows + kM - 1) / kM;
  // S == 1: CTA blockIdx.y walks tiles blockIdx.y, + gridDim.y, ...; S > 1: one tile each
  const int64_t first = blockIdx.y, stride = gridDim.y;
  const int64_t my_tiles = first < tiles ? (tiles - first + stride - 1) / stride : 0;
  const int kc = p.kc;
  const int64_t k0 = (int64_t)rank * kc;
  const int nst = kc / kKT;  // stages per tile
  const int64_t total = my_tiles * nst;
  uint8_t* Bs = smem + ((128u - (smem_u32(smem) & 127u)) & 127u);
  uint8_t* ring = Bs + b_bytes(kc);
  float* part = reinterpret_cast<float*>(ring + kRing * kI8Bytes);  // [kNB][kM]
  const uint32_t bsbo = (uint32_t)(kc / 8) * kCoreBytes;
  const uint32_t full0 = smem_u32(&bar_full[0]), empty0 = smem_u32(&bar_empty[0]);
  const uint32_t done0 = smem_u32(&bar_done[0]), drained0 = smem_u32(&bar_drained[0]);

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < kNA; ++i) {
      mbar_init(full0 + 8 * i, kConvWarps);  // one arrival per converter warp
      mbar_init(empty0 + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(done0 + 8 * i, nst >= 2 ? 2 : 1);  // one commit per MMA lane with a stage in the tile
      mbar_init(drained0 + 8 * i, kEpi);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t taddr = tmem_base;

  if (warp < kConvWarps) {
    // ======================= converter / epilogue warps =======================
    bool bad = false;
    const uint32_t ring_s = smem_u32(ring);
    // weight ring: global stage g = tile index t * nst + s.  This thread's row of the
    // tile and K offset within a stage; chunk j of its kChunks 16-byte chunks sits at
    // 16 (kConv j + tid) of a ring slot (the thread reads back only what it copied, and a
    // warp's lanes touch consecutive 16-byte words: no bank conflicts).
    const int r = 32 * (warp & 3) + lane, kb = (warp >> 2) * kPartK;
    // copy cursor: the next stage to copy (tile it, stage is, ring slot islot); 32-bit
    // counters updated by one step (no division in the loop)
    int ig = 0, is = 0, islot = 0;
    int64_t irow0 = first * kM;
    auto issue = [&]() {
      if (ig < total) {
        const int64_t row = min(irow0 + r, p.rows - 1);  // rows past the end: any valid row
        const int8_t* src = p.codes + row * p.cols + k0 + (int64_t)is * kKT + kb;
        const uint32_t slot = ring_s + (uint32_t)islot * kI8Bytes + 16u * (uint32_t)tid;
#pragma unroll
        for (int j = 0; j < kChunks; ++j)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(slot + 16u * kConv * j), "l"(src + 16 * j)
                       : "memory");
        ++ig;
        if (++is == nst) {
          is = 0;
          irow0 += stride * kM;
        }
        if (++islot == kRing) islot = 0;
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // The epilogue of local tile t: wait for its accumulator, read it out (row 32 warp +
    // lane), release the accumulator, then finish the row (S == 1) or park the partial.
    auto epilogue = [&](int64_t t) {
      if (warp >= 4) return;  // warps 0-3 map onto the accumulator's 128 lanes
      const int acc = (int)(t & 1);
      const int64_t row0 = (first + t * stride) * kM;
      const bool ok = mbar_wait(done0 + 8 * acc, (uint32_t)(t >> 1) & 1u);
      if (!ok) bad = true;
      fence_after_sync();
      float v[32];
      tmem_ld32(taddr + (uint32_t)(64 * acc) + ((uint32_t)(32 * warp) << 16), v);
      if (nst >= 2) {  // the odd stages' half
        float w[32];
        tmem_ld32(taddr + (uint32_t)(64 * acc + 32) + ((uint32_t)(32 * warp) << 16), w);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += w[i];
      }
      fence_before_sync();
      mbar_arrive(drained0 + 8 * acc);
      const int r = 32 * warp + lane;
      const int64_t row = row0 + r;
      if (S > 1) {
#pragma unroll
        for (int b = 0; b < kNB; ++b) part[b * kM + r] = bad ? 0.f : (v[b] + v[kNB + b]) * unscale[b];
        return;
      }
      const float rs = row < p.rows ? __ldg(p.row_scale + row) : 0.f;
#pragma unroll
      for (int b = 0; b < kNB; ++b) {
        const float val = bad ? 0.f : (v[b] + v[kNB + b]) * unscale[b] * rs;
        const bool in = b < p.batch && row < p.rows;
        if (p.mode == kGemvSwiGLU) {
          const float up = __shfl_down_sync(0xffffffffu, val, 1);  // row + 1 sits in the next lane
          if (in && (r & 1) == 0 && row + 1 < p.rows)
            p.y[(int64_t)b * (p.rows / 2) + row / 2] = val / (1.0f + expf(-val)) * up;
        } else if (in) {
          float* dst = p.y + (int64_t)b * p.rows + row;
          if (p.mode == kGemvAccumulate)
            *dst += val;
          else
            *dst = val;
        }
      }
    };

#pragma unroll
    for (int g = 0; g < kRing - 1; ++g) issue();

    pdl_wait();  // x comes from the previous kernel

    // ---- B: per sequence, the largest |x| of this CTA's columns, then the scaled high and
    // low f16 parts in the canonical layout (row n = sequence n high, 16 + n low)
    for (int b = warp; b < kNB; b += kConvWarps) {
      float m = 0.f;
      if (b < p.batch) {
        const float4* xr = reinterpret_cast<const float4*>(p.x + (int64_t)b * p.cols + k0);
        for (int i = lane; i < kc / 4; i += 32) {
          const float4 v = __ldcg(xr + i);
          m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
          if (isnan(v.x) || isnan(v.y) || isnan(v.z) || isnan(v.w)) m = INFINITY;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) wmax[b] = m;
    }
    conv_bar();
    float sc_b[kNB];  // multiplier into f16 range per sequence
#pragma unroll
    for (int b = 0; b < kNB; ++b) {
      const float m = wmax[b];
      const int F = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
      // m in [2^F, 2^(F+1)) -> scale 2^(13 - F); zero / tiny rows keep scale 1; a
      // non-finite row gets a NaN unscale so its outputs become NaN
      const bool live = m > 0.f && F > -100 && F < 128;
      sc_b[b] = live ? __uint_as_float((uint32_t)(127 + 13 - F) << 23) : 1.f;
      if (tid == 0)
        unscale[b] =
            F == 128 ? __uint_as_float(0x7FC00000u) : (live ? __uint_as_float((uint32_t)(127 - 13 + F) << 23) : 1.f);
    }
    // 8 chunks (of 8 columns) per pass: all loads first, then the conversions and stores
    const int nchunk = kNB * (kc / 8);
    for (int c0 = tid; c0 < nchunk; c0 += 8 * kConv) {
      float4 v[8][2];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * kConv, b = c / (kc / 8), k8 = c % (kc / 8);
        v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < nchunk && b < p.batch) {
          const float4* src = reinterpret_cast<const float4*>(p.x + (int64_t)b * p.cols + k0 + 8 * k8);
          v[u][0] = __ldcg(src);
          v[u][1] = __ldcg(src + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * kConv, b = c / (kc / 8), k8 = c % (kc / 8);
        if (c >= nchunk) break;
        float sc = 1.f;
#pragma unroll
        for (int bb = 0; bb < kNB; ++bb) sc = bb == b ? sc_b[bb] : sc;
        const float f[8] = {v[u][0].x * sc, v[u][0].y * sc, v[u][0].z * sc, v[u][0].w * sc,
                            v[u][1].x * sc, v[u][1].y * sc, v[u][1].z * sc, v[u][1].w * sc};
        uint32_t h[4], l[4];
#pragma unroll
        for (int t2 = 0; t2 < 4; ++t2) {
          const __half a = __float2half_rn(f[2 * t2]), bq = __float2half_rn(f[2 * t2 + 1]);
          const __half la = __float2half_rn(f[2 * t2] - __half2float(a));
          const __half lb = __float2half_rn(f[2 * t2 + 1] - __half2float(bq));
          __half2 hh = __halves2half2(a, bq), ll = __halves2half2(la, lb);
          h[t2] = *reinterpret_cast<uint32_t*>(&hh);
          l[t2] = *reinterpret_cast<uint32_t*>(&ll);
        }
        const int nh = b, nl = kNB + b;
        *reinterpret_cast<uint4*>(Bs + (nh >> 3) * bsbo + k8 * kCoreBytes + (nh & 7) * 16) =
            make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(Bs + (nl >> 3) * bsbo + k8 * kCoreBytes + (nl & 7) * 16) =
            make_uint4(l[0], l[1], l[2], l[3]);
      }
    }
    conv_bar();     // unscale is written; B is complete (made visible to the MMAs below)
    pdl_trigger();  // the next kernel may launch (it waits for this one before reading y)

    // ---- stage loop: convert this thread's kPartK codes of stage g into A stage `ab` of
    // tensor memory (its row's lane, columns kb / 2 .. kb / 2 + kPartK / 2 - 1 of the stage)
    const int epi_at = nst - 1 < kEpiDelay ? nst - 1 : kEpiDelay;
    int t = 0, s = 0, slot_i = 0;  // tile, stage and ring slot of stage g
    int ab = 0;                    // A stage in tensor memory
    uint32_t afills = 0;           // earlier fills of A stage ab
    int64_t row0 = first * kM;
    const uint32_t ta_row = taddr + ((uint32_t)(32 * (warp & 3)) << 16) + kAccCols + (uint32_t)(kb / 2);
    for (int g = 0; g < (int)total; ++g) {
      issue();  // stage g + kRing - 1
      asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");  // stage g landed
      if (afills > 0 && !bad && !mbar_wait(empty0 + 8 * ab, (afills - 1) & 1u)) bad = true;  // A stage free
      fence_after_sync();
      const uint8_t* slot = ring + slot_i * kI8Bytes + 16 * tid;
      uint4 q[kChunks];
#pragma unroll
      for (int j = 0; j < kChunks; ++j) q[j] = *reinterpret_cast<const uint4*>(slot + 16 * kConv * j);
      uint32_t h[kPartK / 2] = {};
      if (row0 + r < p.rows) {
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          i8x4_to_h2x2(q[j].x, h[8 * j + 0], h[8 * j + 1]);
          i8x4_to_h2x2(q[j].y, h[8 * j + 2], h[8 * j + 3]);
          i8x4_to_h2x2(q[j].z, h[8 * j + 4], h[8 * j + 5]);
          i8x4_to_h2x2(q[j].w, h[8 * j + 6], h[8 * j + 7]);
        }
      }
      tmem_st32(ta_row + (uint32_t)ab * kACols, h);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(full0 + 8 * ab);
      if (s == epi_at && t >= 1) epilogue(t - 1);
      if (++slot_i == kRing) slot_i = 0;
      if (++ab == kNA) {
        ab = 0;
        ++afills;
      }
      if (++s == nst) {
        s = 0;
        ++t;
        row0 += stride * kM;
      }
    }
    if (my_tiles >= 1) epilogue(my_tiles - 1);
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy in flight at exit
    if (bad && p.err) atomicOr(p.err, kErrTimeout);
  } else if (lane == 0 && (warp == kMmaWarp || nst >= 2)) {
    // ======================= MMA lanes =======================
    // Lane L (warp kMmaWarp + L) issues the MMAs of the stages s of every tile with
    // s % 2 == L into half L of the tile's accumulator: two issuing threads keep about
    // 1.7 times the MMAs in flight of one.
    const int L = warp - kMmaWarp;
    const int s_last = nst - 1 - ((nst - 1 - L) & 1);  // this lane's last stage of a tile
    bool bad = false;
    int t = 0, s = 0;     // tile and stage of stage g
    int ab = 0;           // A stage in tensor memory
    uint32_t afills = 0;  // earlier fills of A stage ab
    for (int g = 0; g < (int)total && !bad; ++g) {
      const int acc = t & 1;
      if ((s & 1) == L) {
        if (s == L && t >= 2 && !mbar_wait(drained0 + 8 * acc, (uint32_t)((t - 2) >> 1) & 1u)) bad = true;
        if (!bad && !mbar_wait(full0 + 8 * ab, afills & 1u)) bad = true;
        if (bad) break;
        fence_after_sync();
        const uint32_t a0 = taddr + kAccCols + (uint32_t)ab * kACols;
        const uint32_t b0 = smem_u32(Bs) + (uint32_t)(s * kKT / 8) * kCoreBytes;
        const uint32_t d = taddr + (uint32_t)(64 * acc + 32 * L);
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk)  // 16 K elements = 8 columns of A per instruction
          mma_f16_ta(d, a0 + 8u * kk, smem_desc(b0 + kk * 2 * kCoreBytes, kCoreBytes, bsbo), (s > L || kk > 0) ? 1u : 0u);
        mma_commit(empty0 + 8 * ab);
        if (s == s_last) mma_commit(done0 + 8 * acc);
      }
      if (++ab == kNA) {
        ab = 0;
        ++afills;
      }
      if (++s == nst) {
        s = 0;
        ++t;
      }
    }
    if (bad && p.err) atomicOr(p.err, kErrTimeout);
  }

  // ---- split-K: rank-order sum of the cluster's partials; CTA `rank` finishes rows
  // [rank * R, (rank+1) * R) of its (single) tile
  if (S > 1) {
    cluster.sync();  // every CTA's partial is in place
    if (warp < kConvWarps && my_tiles == 1) {
      const int R = kM / S;
      const int64_t row0 = first * kM;
      for (int i = tid; i < kNB * R; i += kConv) {
        const int b = i / R, rr = rank * R + i % R;
        float acc = 0.f;
        for (int q = 0; q < S; ++q) acc += *cluster.map_shared_rank(part + b * kM + rr, q);
        const int64_t row = row0 + rr;
        const bool in = b < p.batch && row < p.rows;
        const float val = in ? acc * __ldg(p.row_scale + row) : 0.f;
        if (p.mode == kGemvSwiGLU) {
          const float up = __shfl_down_sync(0xffffffffu, val, 1);  // row + 1 sits in the next lane
          if (in && (rr & 1) == 0 && row + 1 < p.rows)
            p.y[(int64_t)b * (p.rows / 2) + row / 2] = val / (1.0f + expf(-val)) * up;
        } else if (in) {
          float* dst = p.y + (int64_t)b * p.rows + row;
          if (p.mode == kGemvAccumulate)
            *dst += val;
          else
            *dst = val;
        }
      }
    }
    cluster.sync();  // keep this CTA's partial alive until every reader is done
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols)
                              : "memory");
}

int sm_count_tc() {
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

// Cluster size S (columns per CTA = cols / S).  With at least half as many row tiles as
// SMs: the smallest legal S (S == 1 runs persistent CTAs over the tiles).  Otherwise the
// largest power of two up to 8 with tiles x S within the SMs.  Legal: cols divisible by
// S * kKT and at most kMaxKc columns per CTA.
int choose_split(int64_t rows, int64_t cols) {
  const int64_t tiles = (rows + kM - 1) / kM;
  const int64_t nsm = sm_count_tc();
  int best = 0;
  for (int s = 1; s <= kMaxCluster; s *= 2) {
    if (cols % ((int64_t)s * kKT) || cols / s > kMaxKc) continue;
    if (best == 0) {
      best = s;  // smallest legal split
      if (2 * tiles >= nsm) break;
    } else if (tiles * s <= nsm) {
      best = s;
    }
  }
  return best;
}

}  // namespace tc_gemv

bool gemv_tc_supported(const GemvArgs& a) {
  using namespace tc_gemv;
  if (a.fmt != QD_I8_ROW || a.batch <= 8 || a.batch > kNB || a.norm_g) return false;
  if (a.mode != kGemvStore && a.mode != kGemvAccumulate && a.mode != kGemvSwiGLU) return false;
  if (a.mode == kGemvSwiGLU && (a.W.rows & 1)) return false;
  return choose_split(a.W.rows, a.W.cols) > 0;
}

qd_status launch_q_gemv_tc(const GemvArgs& a, cudaStream_t stream) {
  using namespace tc_gemv;
  if (!gemv_tc_supported(a)) return QD_ERR_UNSUPPORTED;
  const int S = choose_split(a.W.rows, a.W.cols);
  Params p;
  p.codes = reinterpret_cast<const int8_t*>(a.W.codes);
  p.row_scale = reinterpret_cast<const float*>(a.W.scales);
  p.rows = a.W.rows;
  p.cols = a.W.cols;
  p.x = a.x;
  p.y = a.y;
  p.batch = a.batch;
  p.kc = (int)(a.W.cols / S);
  p.mode = a.mode;
  p.err = a.err;
  const uint32_t smem = smem_bytes(p.kc);
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_done[dev]) {
    if (cudaFuncSetAttribute(k_gemv_tc_i8, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes(kMaxKc)) !=
        cudaSuccess)
      return QD_ERR_CUDA;
    attr_done[dev] = true;
  }
  // S == 1: persistent CTAs, one per SM at most; S > 1: one cluster per row tile
  const int64_t tiles = (a.W.rows + kM - 1) / kM;
  int64_t ny = S == 1 ? (tiles < sm_count_tc() ? tiles : sm_count_tc()) : tiles;
  if (ny < 1) ny = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S, (unsigned)ny);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_gemv_tc_i8, p) == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

}  // namespace qd
