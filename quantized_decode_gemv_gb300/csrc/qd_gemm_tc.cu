// Batched prefill product on the 5th-generation tensor cores: y[n][r] = sum_c deq(W)[r][c]
// x[n][c] for t tokens n (llmoxide blog s11: prefill is the decode product with t rows of x
// through one read of the weights, and becomes compute-bound; its Metal GEMM dequantises a
// tile of weights once into on-chip memory and runs it on the matrix units).
//
//  * A (the weights): a CTA tile is 256 rows (two MMA tiles of M = 128) by 64 tokens.  Eight
//    converter warps, one thread per row, stream the packed codes of each 64-column stage
//    through a per-thread cp.async ring (six stages deep), dequantise them to f16 and write
//    them with one tcgen05.st into one of four A stages in tensor memory (row r of an MMA
//    tile in lane r, two f16 per 32-bit column).  Q4_0 and Q8_0: the code is widened
//    exactly (magic-number f16) and multiplied by the block's f16 scale in f16: the weight
//    enters as the binary16 rounding of d * q.  INT8 rows: the code enters exactly, the row
//    scale is applied in f32 at the end.
//  * B (x): a prologue kernel scales each token's x by a power of two (its largest |x| in
//    [2^13, 2^14), exact) and splits it into an f16 high part and the f16 rounding of the
//    remainder (about 2^-22 relative together), laid out in a workspace as the exact
//    shared-memory image of each (64-token tile, stage): 64 high rows, then 64 low rows
//    (K-major, no-swizzle canonical layout).  One thread streams the images into a
//    six-stage ring with bulk copies.
//  * MMAs: one thread issues, per stage, 2 x 4 tcgen05.mma kind::f16 (M = 128, N = 128,
//    K = 16; A from tensor memory, B from shared memory) into the tile's two 128-column
//    accumulators.  The A stages take the rest of tensor memory, so there is one
//    accumulator set: the converter warps read a tile out (tcgen05.ld) right after the
//    next tile's first stage, y = (high + low) * 2^-e (* row scale), and the MMAs of the
//    next tile start once the read-out has released the accumulators.
//  * Tiles (row tile, token tile), token tile fastest, are dealt to persistent CTAs (one
//    per SM): CTAs running at the same time share row tiles, so the weights come from
//    HBM about once and from L2 for the other token tiles.
//
// Every mbarrier wait is bounded; on a timeout the kernel sets kErrTimeout (when given an
// error word), stops issuing, finishes its loops without waiting, frees its tensor memory
// and returns.
#include <cuda_fp16.h>

#include "qd_internal.cuh"
#include "qd_tc.cuh"

namespace qd {
namespace tc_gemm {

using namespace tc;

constexpr int kMT = 256;          // weight rows per CTA tile
constexpr int kTN = 64;           // tokens per CTA tile
constexpr int kN = 2 * kTN;       // MMA N: the tokens' high parts, then their low parts
constexpr int kKS = 64;           // K elements per stage
constexpr int kAStages = 4;       // A stages in tensor memory
constexpr int kBStages = 6;       // B stages in shared memory
constexpr int kCodeRing = 6;      // code stages in flight per converter thread
constexpr int kConvWarps = 8;     // converter thread = weight row of the tile
constexpr int kConv = 32 * kConvWarps;
constexpr int kMmaWarp = kConvWarps, kBWarp = kConvWarps + 1;
constexpr int kThreads = kConv + 64;
constexpr uint32_t kBBytes = kN * kKS * 2;            // one B image (16 KB)
constexpr uint32_t kCodeSlot = kConv * 64;            // up to 64 code bytes per row and stage
constexpr uint32_t kScaleSlot = kConv * 4;            // two f16 block scales per row and stage
constexpr uint32_t kSbo = (kKS / 8) * kCoreBytes;     // core-matrix step along M/N (1 KB)
// Tensor memory: the two 128-row accumulators (kN columns each), then kAStages A stages,
// each the two 128-row halves of the tile (row r in lane r, two f16 per 32-bit column).
constexpr uint32_t kAccCols = kN;
constexpr uint32_t kACols = kKS / 2;                  // one 128-row half of an A stage
constexpr uint32_t kAStageCols = 2 * kACols;
constexpr uint32_t kTmemCols = 512;
static_assert(2 * kAccCols + kAStages * kAStageCols <= kTmemCols, "tensor memory columns");
constexpr uint32_t kIdesc = idesc_f16(128, kN);
constexpr uint32_t kSmemBytes = 1024 + kBStages * kBBytes + kCodeRing * (kCodeSlot + kScaleSlot);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// code bytes of one row and stage, in 16-byte chunks
template <int FMT>
constexpr int code_chunks() {
  return FMT == QD_Q4_0 ? 2 : 4;
}

struct Params {
  const uint8_t* codes;
  const uint8_t* scales;
  int64_t row_code_bytes, row_scale_bytes;
  int64_t rows;
  int cols, t, nks, tt_tiles;
  int64_t tiles;
  const uint8_t* bimg;    // [token tile][stage] B images
  const float* unscale;   // [token tiles * 64]
  float* y;               // [t][rows] ([t][rows / 2] for SwiGLU)
  uint32_t* err;
  int mode;               // kGemmStore, kGemmAccumulate (y += product), kGemmSwiGLU
};

// ---- the prologue: x -> scaled f16 high / low parts in B-image layout
__global__ void __launch_bounds__(256) k_gemm_split_x(const float* __restrict__ x, int t, int cols, int nks,
                                                      uint8_t* __restrict__ bimg, float* __restrict__ unscale) {
  __shared__ float red[8];
  const int n = blockIdx.x, tt = n / kTN, nn = n % kTN;
  const bool live = n < t;
  const float4* xr = reinterpret_cast<const float4*>(x + (int64_t)(live ? n : 0) * cols);
  float m = 0.f;
  if (live)
    for (int i = threadIdx.x; i < cols / 4; i += blockDim.x) {
      const float4 v = __ldg(xr + i);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      if (isnan(v.x) || isnan(v.y) || isnan(v.z) || isnan(v.w)) m = INFINITY;
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  // m in [2^F, 2^(F+1)) -> multiplier 2^(13 - F); zero / tiny rows keep 1; a non-finite
  // row gets a NaN unscale (its outputs become NaN)
  const int F = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  const bool scaled = m > 0.f && F > -100 && F < 128;
  const float sc = scaled ? __uint_as_float((uint32_t)(127 + 13 - F) << 23) : 1.f;
  if (threadIdx.x == 0)
    unscale[n] = !live ? 0.f
                       : (F == 128 ? __uint_as_float(0x7FC00000u)
                                   : (scaled ? __uint_as_float((uint32_t)(127 - 13 + F) << 23) : 1.f));
  const uint32_t hi_off = (uint32_t)(nn >> 3) * kSbo + (uint32_t)(nn & 7) * 16;
  const uint32_t lo_off = (uint32_t)((kTN + nn) >> 3) * kSbo + (uint32_t)((kTN + nn) & 7) * 16;
  for (int c = threadIdx.x; c < cols / 8; c += blockDim.x) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (live) {
      a = __ldg(xr + 2 * c);
      b = __ldg(xr + 2 * c + 1);
    }
    const float f[8] = {a.x * sc, a.y * sc, a.z * sc, a.w * sc, b.x * sc, b.y * sc, b.z * sc, b.w * sc};
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half h0 = __float2half_rn(f[2 * i]), h1 = __float2half_rn(f[2 * i + 1]);
      const __half l0 = __float2half_rn(f[2 * i] - __half2float(h0));
      const __half l1 = __float2half_rn(f[2 * i + 1] - __half2float(h1));
      __half2 hh = __halves2half2(h0, h1), ll = __halves2half2(l0, l1);
      h[i] = *reinterpret_cast<uint32_t*>(&hh);
      l[i] = *reinterpret_cast<uint32_t*>(&ll);
    }
    const int ks = c / (kKS / 8), k8 = c % (kKS / 8);
    uint8_t* img = bimg + ((int64_t)tt * nks + ks) * kBBytes + (uint32_t)k8 * kCoreBytes;
    *reinterpret_cast<uint4*>(img + hi_off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(img + lo_off) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// The dequantised f16 values of one row and stage: 8 chunks of 8 consecutive columns.
// Q4_0: two 18-byte blocks (element j of a block: low nibble of byte j, element j + 16: high
// nibble of byte j); Q8_0: two blocks of 32 int8 codes; INT8 rows: 64 codes.
template <int FMT>
__device__ __forceinline__ void dequant_stage(const uint4 (&q)[4], uint32_t dd, uint4 (&out)[8]) {
  if constexpr (FMT == QD_I8_ROW) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = q[c >> 1];
      const uint32_t w0 = (c & 1) ? v.z : v.x, w1 = (c & 1) ? v.w : v.y;
      i8x4_to_h2x2(w0, out[c].x, out[c].y);
      i8x4_to_h2x2(w1, out[c].z, out[c].w);
    }
  } else {
#pragma unroll
    for (int bi = 0; bi < 2; ++bi) {
      const uint32_t dbits = bi ? (dd >> 16) : (dd & 0xFFFFu);
      const __half2 d2 = __halves2half2(__ushort_as_half((unsigned short)dbits), __ushort_as_half((unsigned short)dbits));
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w0, w1;
        uint32_t h[4];
        if constexpr (FMT == QD_Q4_0) {
          const uint4 v = q[bi];
          const uint32_t a0 = (c & 1) ? v.z : v.x, a1 = (c & 1) ? v.w : v.y;
          const int sh = (c >> 1) * 4;  // chunks 0, 1: low nibbles; 2, 3: high nibbles
          w0 = (a0 >> sh) & 0x0F0F0F0Fu;
          w1 = (a1 >> sh) & 0x0F0F0F0Fu;
          u4x4_to_h2x2(w0, h[0], h[1]);
          u4x4_to_h2x2(w1, h[2], h[3]);
        } else {  // Q8_0
          const uint4 v = q[2 * bi + (c >> 1)];
          w0 = (c & 1) ? v.z : v.x;
          w1 = (c & 1) ? v.w : v.y;
          i8x4_to_h2x2(w0, h[0], h[1]);
          i8x4_to_h2x2(w1, h[2], h[3]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __half2 p = __hmul2(*reinterpret_cast<__half2*>(&h[i]), d2);  // binary16 rounding of d * q
          h[i] = *reinterpret_cast<uint32_t*>(&p);
        }
        out[4 * bi + c] = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) k_gemm_tc(const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_fa[kAStages], bar_ea[kAStages], bar_fb[kBStages], bar_eb[kBStages];
  __shared__ __align__(8) uint64_t bar_done, bar_drained;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* Bs = smem;                              // [kBStages][B image]
  uint8_t* codes = Bs + kBStages * kBBytes;        // [kCodeRing][chunk][thread] 16 B
  uint8_t* dsc = codes + kCodeRing * kCodeSlot;    // [kCodeRing][thread] 4 B
  const uint32_t fa0 = smem_u32(&bar_fa[0]), ea0 = smem_u32(&bar_ea[0]);
  const uint32_t fb0 = smem_u32(&bar_fb[0]), eb0 = smem_u32(&bar_eb[0]);
  const uint32_t done = smem_u32(&bar_done), drained = smem_u32(&bar_drained);
  const int64_t G = gridDim.x, first = blockIdx.x;
  const int64_t my_tiles = first < p.tiles ? (p.tiles - first + G - 1) / G : 0;
  const int nks = p.nks;
  const int64_t total = my_tiles * nks;

  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(fa0 + 8 * i, kConvWarps);  // one arrival per converter warp
      mbar_init(ea0 + 8 * i, 1);           // the MMA commit
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(fb0 + 8 * i, 1);  // the B copy (bytes)
      mbar_init(eb0 + 8 * i, 1);  // the MMA commit
    }
    mbar_init(done, 1);
    mbar_init(drained, kConvWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t taddr = tmem_base;

  if (warp < kConvWarps) {
    // ======================= converters (and the accumulator read-out) =======================
    bool bad = false;
    constexpr int CH = code_chunks<FMT>();
    const uint32_t codes_s = smem_u32(codes), dsc_s = smem_u32(dsc);
    // copy cursor: the next stage to copy (stage is of tile itile, ring slot islot); the
    // row moves once per tile
    int64_t ig = 0;
    int64_t itile = first;
    int is = 0, islot = 0;
    // this thread's row of tile `tile` (rows past the end: any valid row)
    auto row_of = [&](int64_t tile) { return min((tile / p.tt_tiles) * kMT + tid, p.rows - 1); };
    int64_t irow = row_of(itile);
    auto issue = [&]() {
      if (ig < total) {
        const uint8_t* src = p.codes + irow * p.row_code_bytes + (int64_t)is * (CH * 16);
        const uint32_t slot = codes_s + (uint32_t)islot * kCodeSlot + 16u * (uint32_t)tid;
#pragma unroll
        for (int j = 0; j < CH; ++j)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(slot + 16u * kConv * j), "l"(src + 16 * j)
                       : "memory");
        if constexpr (FMT != QD_I8_ROW) {
          const uint8_t* ssrc = p.scales + irow * p.row_scale_bytes + (int64_t)is * 4;
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dsc_s + (uint32_t)islot * kScaleSlot +
                                                                          4u * (uint32_t)tid),
                       "l"(ssrc)
                       : "memory");
        }
        ++ig;
        if (++is == nks) {
          is = 0;
          itile += G;
          irow = row_of(itile);
        }
        if (++islot == kCodeRing) islot = 0;
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    // Read out local tile i: wait for its accumulators, load this thread's row (high and
    // low columns), release them, then scale and store.
    const int sub = warp >> 2, quarter = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
    auto epilogue = [&](int64_t i) {
      const int64_t tile = first + i * G;
      const int64_t row = (tile / p.tt_tiles) * kMT + tid;
      const int n0 = (int)(tile % p.tt_tiles) * kTN;
      if (!bad && !mbar_wait_sleep(done, (uint32_t)i & 1u)) bad = true;
      fence_after_sync();
      const uint32_t acc = taddr + lane_base + (uint32_t)(kAccCols * sub);
      const float rs = (FMT == QD_I8_ROW && row < p.rows)
                           ? __ldg(reinterpret_cast<const float*>(p.scales + row * p.row_scale_bytes))
                           : 1.f;
      float v[kTN];
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // tokens 32 h .. 32 h + 31: high part + low part
        float hi[32], lo[32];
        tmem_ld32(acc + (uint32_t)(32 * h), hi);
        tmem_ld32(acc + (uint32_t)(kTN + 32 * h), lo);
#pragma unroll
        for (int k = 0; k < 32; ++k) v[32 * h + k] = hi[k] + lo[k];
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(drained);  // the accumulators may be overwritten
      if (p.mode == kGemmSwiGLU) {
        // rows (2i, 2i + 1) = (gate_i, up_i) sit in lanes (2j, 2j + 1): y[n][i] = silu(gate) * up
#pragma unroll
        for (int k = 0; k < kTN; ++k) {
          const int n = n0 + k;
          const float val = (row < p.rows && n < p.t && !bad) ? v[k] * __ldg(p.unscale + n) * rs : 0.f;
          const float up = __shfl_down_sync(0xffffffffu, val, 1);
          if ((tid & 1) == 0 && row + 1 < p.rows && n < p.t)
            p.y[(int64_t)n * (p.rows / 2) + row / 2] = val / (1.0f + expf(-val)) * up;
        }
      } else if (row < p.rows) {
#pragma unroll
        for (int k = 0; k < kTN; ++k) {
          const int n = n0 + k;
          if (n < p.t) {
            const float val = bad ? 0.f : v[k] * __ldg(p.unscale + n) * rs;
            float* dst = p.y + (int64_t)n * p.rows + row;
            *dst = p.mode == kGemmAccumulate ? *dst + val : val;
          }
        }
      }
    };

#pragma unroll
    for (int g = 0; g < kCodeRing - 1; ++g) issue();
    int64_t t = 0;
    int s = 0, cslot = 0, aslot = 0;
    uint32_t afills = 0;  // earlier fills of A stage aslot
    const uint32_t a_row = taddr + lane_base + kAccCols * 2 + (uint32_t)(kACols * sub);
    for (int64_t g = 0; g < total; ++g) {
      issue();  // stage g + kCodeRing - 1
      asm volatile("cp.async.wait_group %0;" ::"n"(kCodeRing - 1) : "memory");  // stage g landed
      uint4 q[4];
      const uint8_t* cs = codes + cslot * kCodeSlot + 16 * tid;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        q[j] = j < CH ? *reinterpret_cast<const uint4*>(cs + 16 * kConv * j) : make_uint4(0, 0, 0, 0);
      const uint32_t dd =
          FMT != QD_I8_ROW ? *reinterpret_cast<const uint32_t*>(dsc + cslot * kScaleSlot + 4 * tid) : 0u;
      uint4 out[8];
      dequant_stage<FMT>(q, dd, out);
      uint32_t h[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        h[4 * c + 0] = out[c].x;
        h[4 * c + 1] = out[c].y;
        h[4 * c + 2] = out[c].z;
        h[4 * c + 3] = out[c].w;
      }
      if (afills > 0 && !bad && !mbar_wait_sleep(ea0 + 8 * aslot, (afills - 1) & 1u)) bad = true;  // A stage free
      fence_after_sync();
      tmem_st32(a_row + (uint32_t)aslot * kAStageCols, h);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(fa0 + 8 * aslot);
      // the previous tile's read-out, once this tile's first stage is on its way
      if (s == 0 && t >= 1) epilogue(t - 1);
      if (++cslot == kCodeRing) cslot = 0;
      if (++aslot == kAStages) {
        aslot = 0;
        ++afills;
      }
      if (++s == nks) {
        s = 0;
        ++t;
      }
    }
    if (my_tiles >= 1) epilogue(my_tiles - 1);
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy in flight at exit
    if (bad && p.err) atomicOr(p.err, kErrTimeout);
  } else if (warp == kMmaWarp && lane == 0) {
    // ======================= MMA issue =======================
    bool bad = false;
    int64_t g = 0;
    const uint32_t b_s = smem_u32(Bs);
    for (int64_t i = 0; i < my_tiles && !bad; ++i) {
      if (i >= 1 && !mbar_wait(drained, (uint32_t)(i - 1) & 1u)) bad = true;  // the last tile is read out
      fence_after_sync();
      for (int ks = 0; ks < nks && !bad; ++ks, ++g) {
        const int as = (int)(g % kAStages), bs = (int)(g % kBStages);
        if (!mbar_wait(fa0 + 8 * as, (uint32_t)(g / kAStages) & 1u) ||
            !mbar_wait(fb0 + 8 * bs, (uint32_t)(g / kBStages) & 1u)) {
          bad = true;
          break;
        }
        fence_after_sync();
        const uint32_t b0 = b_s + (uint32_t)bs * kBBytes;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          const uint32_t d = taddr + (uint32_t)(kAccCols * m);
          const uint32_t a0 = taddr + kAccCols * 2 + (uint32_t)as * kAStageCols + (uint32_t)(kACols * m);
#pragma unroll
          for (int kk = 0; kk < kKS / 16; ++kk)  // 16 K elements: 8 columns of A, two core matrices of B
            mma_f16_ts(d, a0 + 8u * kk, smem_desc(b0 + kk * 2 * kCoreBytes, kCoreBytes, kSbo), kIdesc,
                       (ks > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(ea0 + 8 * as);
        mma_commit(eb0 + 8 * bs);
        if (ks == nks - 1) mma_commit(done);
      }
    }
    if (bad && p.err) atomicOr(p.err, kErrTimeout);
  } else if (warp == kBWarp && lane == 0) {
    // ======================= B images =======================
    bool bad = false;
    int slot = 0;
    uint32_t fills = 0;
    int64_t issued = 0;
    const uint32_t b_s = smem_u32(Bs);
    for (int64_t i = 0; i < my_tiles && !bad; ++i) {
      const int64_t tt = (first + i * G) % p.tt_tiles;
      for (int ks = 0; ks < nks; ++ks) {
        if (fills > 0 && !mbar_wait(eb0 + 8 * slot, (fills - 1) & 1u)) {
          bad = true;
          break;
        }
        mbar_arrive_expect_tx(fb0 + 8 * slot, kBBytes);
        bulk_copy_g2s(b_s + (uint32_t)slot * kBBytes, p.bimg + (tt * nks + ks) * (int64_t)kBBytes, kBBytes,
                      fb0 + 8 * slot);
        ++issued;
        if (++slot == kBStages) {
          slot = 0;
          ++fills;
        }
      }
    }
    // stay until the last copy into each stage has landed: no copy may target the CTA's
    // shared memory after it exits
    for (int64_t k = issued > kBStages ? issued - kBStages : 0; k < issued; ++k)
      if (!mbar_wait(fb0 + 8 * (int)(k % kBStages), (uint32_t)(k / kBStages) & 1u)) bad = true;
    if (bad && p.err) atomicOr(p.err, kErrTimeout);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
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

template <int FMT>
qd_status launch_fmt(const Params& p, int grid, cudaStream_t stream) {
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return QD_ERR_CUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(k_gemm_tc<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
      return QD_ERR_CUDA;
    attr_done[dev] = true;
  }
  k_gemm_tc<FMT><<<grid, kThreads, kSmemBytes, stream>>>(p);
  return launch_status();
}

}  // namespace tc_gemm

size_t gemm_workspace_bytes(int64_t cols, int t) {
  using namespace tc_gemm;
  const int64_t tt = (t + kTN - 1) / kTN, nks = cols / kKS;
  return align_up((size_t)(tt * nks) * kBBytes, 16) + align_up((size_t)(tt * kTN) * 4, 16);
}

qd_status launch_q_gemm(int fmt, const PackedView& W, const float* x, float* y, int t, void* ws, uint32_t* err,
                        cudaStream_t stream, int mode) {
  using namespace tc_gemm;
  if (mode != kGemmStore && mode != kGemmAccumulate && mode != kGemmSwiGLU) return QD_ERR_INVALID_ARG;
  if (mode == kGemmSwiGLU && (W.rows & 1)) return QD_ERR_SHAPE;
  Params p;
  p.mode = mode;
  p.codes = W.codes;
  p.scales = W.scales;
  p.row_code_bytes = W.row_code_bytes;
  p.row_scale_bytes = W.row_scale_bytes;
  p.rows = W.rows;
  p.cols = (int)W.cols;
  p.t = t;
  p.nks = (int)(W.cols / kKS);
  p.tt_tiles = (t + kTN - 1) / kTN;
  p.tiles = ((W.rows + kMT - 1) / kMT) * p.tt_tiles;
  uint8_t* base = static_cast<uint8_t*>(ws);
  p.bimg = base;
  p.unscale = reinterpret_cast<const float*>(base + align_up((size_t)p.tt_tiles * p.nks * kBBytes, 16));
  p.y = y;
  p.err = err;
  k_gemm_split_x<<<p.tt_tiles * kTN, 256, 0, stream>>>(x, t, p.cols, p.nks, base, const_cast<float*>(p.unscale));
  qd_status st = launch_status();
  if (st != QD_OK) return st;
  const int grid = (int)(p.tiles < sm_count() ? p.tiles : sm_count());
  switch (fmt) {
    case QD_Q4_0: return launch_fmt<QD_Q4_0>(p, grid, stream);
    case QD_Q8_0: return launch_fmt<QD_Q8_0>(p, grid, stream);
    case QD_I8_ROW: return launch_fmt<QD_I8_ROW>(p, grid, stream);
    default: return QD_ERR_UNSUPPORTED;
  }
}

}  // namespace qd
