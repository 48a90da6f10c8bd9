// The decode step's operations other than the GEMV: RMSNorm, RoPE, KV-cache
// append, split-KV grouped-query decode attention, SwiGLU, argmax, embedding.
#include <cooperative_groups.h>

#include <cmath>
#include <mutex>

#include "qd_attn.cuh"

namespace qd {
namespace {

using namespace attn;

inline int grid1d(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  return (int)(g < 1 ? 1 : (g > 1048576 ? 1048576 : g));
}

// ------------------------------------------------------------------ RMSNorm
// out = x * g / sqrt(mean(x^2) + eps)  (llmoxide s4 rms_norm_mul; dasLLAMA
// 8.7.1.6.2 rmsnorm).  One CTA per batch row.
__global__ void __launch_bounds__(512) k_rmsnorm(const float* __restrict__ x, const float* __restrict__ g,
                                                 float* __restrict__ out, int n, float eps) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const float* xr = x + (int64_t)blockIdx.x * n;
  float* orow = out + (int64_t)blockIdx.x * n;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = 1.0f / sqrtf(v / (float)n + eps);
  }
  __syncthreads();
  const float scale = red[0];
  for (int i = threadIdx.x; i < n; i += blockDim.x) orow[i] = xr[i] * scale * g[i];
}

// ------------------------------------------------------------------ RoPE
// Pair i of each head turns by the angle of (pos, i) from the host-built table
// (llmoxide s6 rope: pairs (2i,2i+1) "adjacent" or (i, i+hd/2) "half").
__global__ void k_rope(float* __restrict__ v, int n_heads, int head_dim, int64_t batch_stride,
                       const int32_t* __restrict__ pos, int pairing, const float* __restrict__ cs, int max_ctx,
                       uint32_t* err) {
  const int b = blockIdx.y;
  const int p = pos[b];
  if (p < 0 || p >= max_ctx) {
    if (err && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(err, kErrPosition);
    return;
  }
  const int half = head_dim / 2;
  const int total = n_heads * half;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
    const int h = t / half, i = t % half;
    float* hv = v + (int64_t)b * batch_stride + (int64_t)h * head_dim;
    const int ia = pairing == QD_ROPE_ADJACENT ? 2 * i : i;
    const int ib = pairing == QD_ROPE_ADJACENT ? 2 * i + 1 : i + half;
    const float c = cs[((int64_t)p * half + i) * 2], s = cs[((int64_t)p * half + i) * 2 + 1];
    const float x0 = hv[ia], x1 = hv[ib];
    hv[ia] = x0 * c - x1 * s;
    hv[ib] = x0 * s + x1 * c;
  }
}

// ------------------------------------------------------------------ KV append
__global__ void k_kv_append(const float* __restrict__ k, const float* __restrict__ v, int64_t src_stride,
                            float* __restrict__ kc, float* __restrict__ vc, int n_kv, int head_dim,
                            const int32_t* __restrict__ pos, int max_ctx, int64_t cache_batch_stride,
                            uint32_t* err) {
  const int b = blockIdx.y;
  const int p = pos[b];
  if (p < 0 || p >= max_ctx) {
    if (err && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(err, kErrPosition);
    return;
  }
  const int total = n_kv * head_dim;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total; t += gridDim.x * blockDim.x) {
    const int h = t / head_dim, i = t % head_dim;
    const int64_t dst = (int64_t)b * cache_batch_stride + ((int64_t)h * max_ctx + p) * head_dim + i;
    kc[dst] = k[(int64_t)b * src_stride + t];
    vc[dst] = v[(int64_t)b * src_stride + t];
  }
}

// ------------------------------------------------------------------ attention
// Split-KV decode attention (llmoxide s5; dasLLAMA 8.7.1.6.2).  The positions
// 0..pos of one (sequence, kv head) are cut into chunks of kChunk; one CTA of 4
// warps takes one chunk for all the q heads of the group that share the kv head.
// Each warp walks its positions with an online softmax (running max m, running
// sum l, running weighted value o); lanes hold 2 of the 64 dimensions.  The CTA
// merges its warps and writes (m, l, o) to the workspace; a second kernel merges
// the chunks with the weights exp(m_s - max_s m_s).
__host__ __device__ inline int attn_chunk(int max_ctx) { return max_ctx <= 1024 ? 32 : 128; }
__host__ __device__ inline int attn_splits(int max_ctx) {
  const int c = attn_chunk(max_ctx);
  return (max_ctx + c - 1) / c;
}

template <int G>
__global__ void __launch_bounds__(kAttnWarps * 32) k_attn_partial(
    const float* __restrict__ q, int64_t q_stride, const float* __restrict__ kc, const float* __restrict__ vc,
    int64_t cache_batch_stride, int n_heads, int n_kv, const int32_t* __restrict__ pos, int max_ctx,
    float scale, float* __restrict__ ws_ml, float* __restrict__ ws_o, uint32_t* err) {
  const int kvh = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int splits = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p_cur = pos[b];
  const bool valid = p_cur >= 0 && p_cur < max_ctx;
  if (!valid && err && threadIdx.x == 0 && split == 0 && kvh == 0) atomicOr(err, kErrPosition);
  const int chunk = attn_chunk(max_ctx);
  const int p_begin = split * chunk;
  const int p_end = valid ? min(p_begin + chunk, p_cur + 1) : p_begin;  // exclusive

  float qs[G][AttnLayout<G>::D];
  attn_load_q<G>(q + (int64_t)b * q_stride, kvh, lane, scale, qs);
  float m[G], l[G];
  float2 o[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
    o[g] = make_float2(0.f, 0.f);
  }
  const float* kb = kc + (int64_t)b * cache_batch_stride + (int64_t)kvh * max_ctx * kHeadDim;
  const float* vb = vc + (int64_t)b * cache_batch_stride + (int64_t)kvh * max_ctx * kHeadDim;
  attn_tiles<G, 2>(kb, vb, p_begin, p_end, warp, lane, qs, m, l, o);
  // merge the warps of this CTA
  __shared__ float sm[kAttnWarps][kMaxGroup], sl[kAttnWarps][kMaxGroup];
  __shared__ float2 so[kAttnWarps][kMaxGroup][32];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      sm[warp][g] = m[g];
      sl[warp][g] = l[g];
    }
    so[warp][g][lane] = o[g];
  }
  __syncthreads();
  for (int g = warp; g < G; g += kAttnWarps) {
    float mx = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < kAttnWarps; ++w2) mx = fmaxf(mx, sm[w2][g]);
    float lt = 0.f;
    float2 ot = make_float2(0.f, 0.f);
#pragma unroll
    for (int w2 = 0; w2 < kAttnWarps; ++w2) {
      const float f = (sm[w2][g] == -INFINITY) ? 0.f : exp2f(sm[w2][g] - mx);
      lt = fmaf(sl[w2][g], f, lt);
      ot.x = fmaf(so[w2][g][lane].x, f, ot.x);
      ot.y = fmaf(so[w2][g][lane].y, f, ot.y);
    }
    const int h = kvh * G + g;
    const int64_t slot = ((int64_t)b * n_heads + h) * splits + split;
    if (lane == 0) {
      ws_ml[slot * 2] = mx;
      ws_ml[slot * 2 + 1] = lt;
    }
    reinterpret_cast<float2*>(ws_o + slot * kHeadDim)[lane] = ot;
  }
}

__global__ void k_attn_merge(const float* __restrict__ ws_ml, const float* __restrict__ ws_o, int n_heads,
                             int splits, const int32_t* __restrict__ pos, int max_ctx, float* __restrict__ out) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;  // 64 threads
  float* dst = out + ((int64_t)b * n_heads + h) * kHeadDim;
  const int p = pos[b];
  if (p < 0 || p >= max_ctx) {
    dst[d] = 0.f;
    return;
  }
  const int used = p / attn_chunk(max_ctx) + 1;  // splits holding positions 0..p
  const int64_t base = ((int64_t)b * n_heads + h) * splits;
  float mx = -INFINITY;
  for (int s = 0; s < used; ++s) mx = fmaxf(mx, ws_ml[(base + s) * 2]);
  float lt = 0.f, acc = 0.f;
  for (int s = 0; s < used; ++s) {
    const float f = exp2f(ws_ml[(base + s) * 2] - mx);
    lt = fmaf(ws_ml[(base + s) * 2 + 1], f, lt);
    acc = fmaf(ws_o[(base + s) * kHeadDim + d], f, acc);
  }
  dst[d] = acc / lt;
}

// Single-kernel form for the decode step: one thread-block cluster of S CTAs per
// (sequence, kv head).  The positions 0..pos are cut into S equal chunks at run time
// (pos is read on the device), each CTA walks its chunk as in k_attn_partial, merges
// its warps, and stores its partial (m, l, o) per q head into the shared memory of the
// cluster's first CTA (distributed shared memory, no global workspace, atomics or
// fences).  After one cluster barrier that CTA merges the S partials (the same
// log-sum-exp merge, in chunk order) and writes the output.
template <int G, int DEP, int W>
__global__ void __launch_bounds__(W * 32) k_attn_cluster(
    const float* __restrict__ q, int64_t q_stride, const float* __restrict__ kc, const float* __restrict__ vc,
    int64_t cache_batch_stride, int n_heads, const int32_t* __restrict__ pos, int max_ctx, float scale,
    float* __restrict__ out, uint32_t* err) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float sm[W][kMaxGroup], sl[W][kMaxGroup];
  __shared__ float2 so[W][kMaxGroup][32];
  // filled in the first CTA of the cluster by every CTA: partial of CTA r for head g
  __shared__ float pm[kMaxCluster][kMaxGroup], pl[kMaxCluster][kMaxGroup];
  __shared__ float2 po[kMaxCluster][kMaxGroup][32];
  pdl_wait();     // q and the cache rows come from the QKV projection
  pdl_trigger();  // let the next kernel start its weight prefetch
  const int p_cur = pos[b];
  const bool valid = p_cur >= 0 && p_cur < max_ctx;
  if (!valid && err && threadIdx.x == 0 && rank == 0 && kvh == 0) atomicOr(err, kErrPosition);
  const int n = valid ? p_cur + 1 : 0;
  const int chunk = (n + S - 1) / S;
  const int p_begin = min(rank * chunk, n), p_end = min(p_begin + chunk, n);

  float qs[G][AttnLayout<G>::D];
  attn_load_q<G>(q + (int64_t)b * q_stride, kvh, lane, scale, qs);
  float m[G], l[G];
  float2 o[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
    o[g] = make_float2(0.f, 0.f);
  }
  const float* kb = kc + (int64_t)b * cache_batch_stride + (int64_t)kvh * max_ctx * kHeadDim;
  const float* vb = vc + (int64_t)b * cache_batch_stride + (int64_t)kvh * max_ctx * kHeadDim;
  attn_tiles<G, DEP, W>(kb, vb, p_begin, p_end, warp, lane, qs, m, l, o);

#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (lane == 0) {
      sm[warp][g] = m[g];
      sl[warp][g] = l[g];
    }
    so[warp][g][lane] = o[g];
  }
  __syncthreads();
  float* rpm = cluster.map_shared_rank(&pm[0][0], 0);
  float* rpl = cluster.map_shared_rank(&pl[0][0], 0);
  float2* rpo = cluster.map_shared_rank(&po[0][0][0], 0);
  for (int g = warp; g < G; g += W) {
    float mx = -INFINITY;
#pragma unroll
    for (int w2 = 0; w2 < W; ++w2) mx = fmaxf(mx, sm[w2][g]);
    float lt = 0.f;
    float2 ot = make_float2(0.f, 0.f);
#pragma unroll
    for (int w2 = 0; w2 < W; ++w2) {
      const float f = (sm[w2][g] == -INFINITY) ? 0.f : exp2f(sm[w2][g] - mx);
      lt = fmaf(sl[w2][g], f, lt);
      ot.x = fmaf(so[w2][g][lane].x, f, ot.x);
      ot.y = fmaf(so[w2][g][lane].y, f, ot.y);
    }
    if (lane == 0) {
      rpm[rank * kMaxGroup + g] = mx;
      rpl[rank * kMaxGroup + g] = lt;
    }
    rpo[(rank * kMaxGroup + g) * 32 + lane] = ot;
  }
  cluster.sync();  // the partials have landed in the first CTA
  if (rank != 0) return;
  for (int g = warp; g < G; g += W) {
    const int h = kvh * G + g;
    float2* dst = reinterpret_cast<float2*>(out + ((int64_t)b * n_heads + h) * kHeadDim);
    float mr[kMaxCluster];
    float mx = -INFINITY;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      mr[r] = r < S ? pm[r][g] : -INFINITY;
      mx = fmaxf(mx, mr[r]);
    }
    float lt = 0.f;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      if (r < S) {
        const float f = mr[r] == -INFINITY ? 0.f : exp2f(mr[r] - mx);
        lt = fmaf(pl[r][g], f, lt);
        acc.x = fmaf(po[r][g][lane].x, f, acc.x);
        acc.y = fmaf(po[r][g][lane].y, f, acc.y);
      }
    }
    dst[lane] = lt > 0.f ? make_float2(acc.x / lt, acc.y / lt) : make_float2(0.f, 0.f);
  }
}

// ------------------------------------------------------------------ QKV post-processing
// The kGemvQKV epilogue as a kernel, for projections computed by the register-path
// GEMV: qkv[b] holds the packed-order rows (RoPE pairs adjacent in q and k).
__global__ void k_qkv_post(const float* __restrict__ qkv, int64_t qkv_stride, QkvEpilogue e, int v_rows,
                           uint32_t* err) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y;
  const int pos = e.pos[b];
  if (pos < 0 || pos >= e.max_ctx) {
    if (err && threadIdx.x == 0 && blockIdx.x == 0) atomicOr(err, kErrPosition);
    return;
  }
  const int hd = e.head_dim, half = hd / 2;
  const int pairs = (e.q_rows + e.k_rows + v_rows) / 2;
  const float* src = qkv + (int64_t)b * qkv_stride;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < pairs; t += gridDim.x * blockDim.x) {
    const int r = 2 * t;
    const float a = src[r], bb = src[r + 1];
    if (r < e.q_rows + e.k_rows) {
      const bool isq = r < e.q_rows;
      const int local = isq ? r : r - e.q_rows;
      const int h = local / hd, pi = (local % hd) / 2;
      const int d0 = e.pairing == QD_ROPE_HALF ? pi : 2 * pi;
      const int d1 = e.pairing == QD_ROPE_HALF ? pi + half : 2 * pi + 1;
      const float c = e.rope[((int64_t)pos * half + pi) * 2], s = e.rope[((int64_t)pos * half + pi) * 2 + 1];
      if (isq) {
        float* dst = e.q_out + (int64_t)b * e.q_stride + (int64_t)h * hd;
        dst[d0] = a * c - bb * s;
        dst[d1] = a * s + bb * c;
      } else {
        const int64_t row = (int64_t)b * e.cache_batch_stride + ((int64_t)h * e.max_ctx + pos) * hd;
        cache_store(e.kc, e.kv_f16, row + d0, a * c - bb * s);
        cache_store(e.kc, e.kv_f16, row + d1, a * s + bb * c);
      }
    } else {
      const int local = r - e.q_rows - e.k_rows;
      const int h = local / hd, d = local % hd;
      const int64_t row = (int64_t)b * e.cache_batch_stride + ((int64_t)h * e.max_ctx + pos) * hd;
      cache_store(e.vc, e.kv_f16, row + d, a);
      cache_store(e.vc, e.kv_f16, row + d + 1, bb);
    }
  }
}

// ------------------------------------------------------------------ SwiGLU
__global__ void k_swiglu(const float* __restrict__ g, const float* __restrict__ u, float* __restrict__ out,
                         int64_t n) {
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n; t += (int64_t)gridDim.x * blockDim.x) {
    const float z = g[t];
    out[t] = z / (1.0f + expf(-z)) * u[t];
  }
}

// ------------------------------------------------------------------ argmax
// Largest value, first index on ties (Go "llm" index: Argmax; dasLLAMA
// 8.7.1.6.4 most_likely).  One CTA per batch row.
__device__ __forceinline__ void better(float& bv, int& bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__global__ void __launch_bounds__(1024) k_argmax(const float* __restrict__ logits, int64_t n,
                                                 int32_t* __restrict__ out, int32_t* __restrict__ pos_adv) {
  __shared__ float sv[32];
  __shared__ int si[32];
  pdl_wait();
  pdl_trigger();
  const float* row = logits + (int64_t)blockIdx.x * n;
  float bv = -INFINITY;
  int bi = (int)n;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) better(bv, bi, row[i], (int)i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    better(bv, bi, ov, oi);
  }
  if ((threadIdx.x & 31) == 0) {
    sv[threadIdx.x >> 5] = bv;
    si[threadIdx.x >> 5] = bi;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = blockDim.x >> 5;
    bv = threadIdx.x < nw ? sv[threadIdx.x] : -INFINITY;
    bi = threadIdx.x < nw ? si[threadIdx.x] : (int)n;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      better(bv, bi, ov, oi);
    }
    if (threadIdx.x == 0) {
      out[blockIdx.x] = bi >= (int)n ? 0 : bi;
      if (pos_adv) pos_adv[blockIdx.x] += 1;
    }
  }
}

// ------------------------------------------------------------------ embedding
__global__ void k_embed(int fmt, PackedView E, const int32_t* __restrict__ tokens, float* __restrict__ x,
                        uint32_t* err) {
  const int b = blockIdx.x;
  const int t = tokens[b];
  float* xr = x + (int64_t)b * E.cols;
  if (t < 0 || t >= E.rows) {
    if (err && threadIdx.x == 0) atomicOr(err, kErrToken);
    for (int64_t c = threadIdx.x; c < E.cols; c += blockDim.x) xr[c] = 0.f;
    return;
  }
  for (int64_t c = threadIdx.x; c < E.cols; c += blockDim.x) xr[c] = dequant_elem(fmt, E, t, c);
}

}  // namespace

qd_status launch_rmsnorm(const float* x, const float* g, float* out, int n, int batch, float eps,
                         cudaStream_t stream) {
  const int threads = n >= 2048 ? 512 : 256;
  k_rmsnorm<<<batch, threads, 0, stream>>>(x, g, out, n, eps);
  return launch_status();
}

qd_status launch_rope(float* v, int n_heads, int head_dim, int64_t batch_stride, const int32_t* pos, int pairing,
                      const float* cos_sin, int max_ctx, int batch, uint32_t* err, cudaStream_t stream) {
  const int total = n_heads * head_dim / 2;
  dim3 grid((unsigned)grid1d(total, 256), (unsigned)batch);
  k_rope<<<grid, 256, 0, stream>>>(v, n_heads, head_dim, batch_stride, pos, pairing, cos_sin, max_ctx, err);
  return launch_status();
}

qd_status launch_kv_append(const float* k, const float* v, int64_t src_stride, float* kc, float* vc, int n_kv,
                           int head_dim, const int32_t* pos, int max_ctx, int batch, int64_t cache_batch_stride,
                           uint32_t* err, cudaStream_t stream) {
  dim3 grid((unsigned)grid1d((int64_t)n_kv * head_dim, 256), (unsigned)batch);
  k_kv_append<<<grid, 256, 0, stream>>>(k, v, src_stride, kc, vc, n_kv, head_dim, pos, max_ctx, cache_batch_stride,
                                        err);
  return launch_status();
}

size_t attn_workspace_bytes(int n_heads, int head_dim, int max_ctx, int batch) {
  const size_t slots = (size_t)batch * n_heads * attn_splits(max_ctx);
  return align_up(slots * 2 * sizeof(float), 256) + slots * (size_t)head_dim * sizeof(float);
}

qd_status launch_attention(const float* q, int64_t q_stride, const float* kc, const float* vc,
                           int64_t cache_batch_stride, float* out, int n_heads, int n_kv, int head_dim,
                           const int32_t* pos, int max_ctx, int batch, void* ws, uint32_t* err,
                           cudaStream_t stream) {
  const int splits = attn_splits(max_ctx);
  const int G = n_heads / n_kv;
  const size_t slots = (size_t)batch * n_heads * splits;
  float* ws_ml = static_cast<float*>(ws);
  float* ws_o = reinterpret_cast<float*>(static_cast<char*>(ws) + align_up(slots * 2 * sizeof(float), 256));
  const float scale = 1.4426950408889634f / sqrtf((float)head_dim);  // scores in log2 units
  dim3 grid((unsigned)n_kv, (unsigned)splits, (unsigned)batch);
  const int threads = kAttnWarps * 32;
#define QD_ATTN_CASE(GG)                                                                                      \
  case GG:                                                                                                    \
    k_attn_partial<GG><<<grid, threads, 0, stream>>>(q, q_stride, kc, vc, cache_batch_stride, n_heads, n_kv, \
                                                     pos, max_ctx, scale, ws_ml, ws_o, err);                  \
    break;
  switch (G) {
    QD_ATTN_CASE(1)
    QD_ATTN_CASE(2)
    QD_ATTN_CASE(3)
    QD_ATTN_CASE(4)
    QD_ATTN_CASE(5)
    QD_ATTN_CASE(6)
    QD_ATTN_CASE(7)
    QD_ATTN_CASE(8)
    default: return QD_ERR_UNSUPPORTED;
  }
#undef QD_ATTN_CASE
  qd_status st = launch_status();
  if (st != QD_OK) return st;
  k_attn_merge<<<dim3((unsigned)n_heads, (unsigned)batch), kHeadDim, 0, stream>>>(ws_ml, ws_o, n_heads, splits, pos,
                                                                                  max_ctx, out);
  return launch_status();
}

// CTAs per cluster for the decode-step attention: enough clusters x CTAs to cover the
// SMs a few times over, at most 8 (the portable cluster size) and at most one CTA per
// 32 positions of the cache.
int attn_sm_count() {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 152;
  if (!sms[dev] && (cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                    sms[dev] <= 0))
    sms[dev] = 152;
  return sms[dev];
}

int attn_cluster_size(int n_kv, int batch, int max_ctx) {
  const int nsm = attn_sm_count();
  const int pairs = n_kv * batch;
  const int target = 4 * nsm;
  int s = 1;
  while (s < kMaxCluster && s * pairs < target && s * 32 < max_ctx) s *= 2;
  return s;
}

// Warps per CTA and tiles in flight per warp for the cluster attention.  Four tiles in
// flight when a tile is small (one or two q heads per kv head) and the CTAs still fit in
// one wave at two per SM; two otherwise.
struct AttnPlan {
  int warps, dep;
};

AttnPlan attn_plan(int G, int S, int n_kv, int batch) {
  const bool deep = G <= 2 && (int64_t)S * n_kv * batch <= 2 * attn_sm_count();
  return AttnPlan{kAttnWarps, deep ? 4 : 2};
}

template <int G>
cudaError_t launch_attn_cluster_g(cudaLaunchConfig_t& cfg, const AttnPlan& plan, const float* q, int64_t q_stride,
                                  const float* kc, const float* vc, int64_t cache_batch_stride, int n_heads,
                                  const int32_t* pos, int max_ctx, float scale, float* out, uint32_t* err) {
  if constexpr (G <= 2) {
    if (plan.warps == 8)
      return cudaLaunchKernelEx(&cfg, plan.dep == 4 ? k_attn_cluster<G, 4, 8> : k_attn_cluster<G, 2, 8>, q, q_stride,
                                kc, vc, cache_batch_stride, n_heads, pos, max_ctx, scale, out, err);
    return cudaLaunchKernelEx(&cfg, plan.dep == 4 ? k_attn_cluster<G, 4, 4> : k_attn_cluster<G, 2, 4>, q, q_stride,
                              kc, vc, cache_batch_stride, n_heads, pos, max_ctx, scale, out, err);
  } else {
    return cudaLaunchKernelEx(&cfg, k_attn_cluster<G, 2, 4>, q, q_stride, kc, vc, cache_batch_stride, n_heads, pos,
                              max_ctx, scale, out, err);
  }
}

qd_status launch_attention_cluster(const float* q, int64_t q_stride, const float* kc, const float* vc,
                                   int64_t cache_batch_stride, float* out, int n_heads, int n_kv, int head_dim,
                                   const int32_t* pos, int max_ctx, int batch, uint32_t* err, cudaStream_t stream,
                                   bool pdl) {
  const int G = n_heads / n_kv;
  const int S = attn_cluster_size(n_kv, batch, max_ctx);
  const float scale = 1.4426950408889634f / sqrtf((float)head_dim);  // scores in log2 units
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)S, (unsigned)n_kv, (unsigned)batch);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const AttnPlan plan = attn_plan(G, S, n_kv, batch);
  cfg.blockDim = dim3((unsigned)plan.warps * 32);
  cudaError_t rc = cudaErrorInvalidValue;
#define QD_ATTN_G(GG)                                                                                         \
  case GG:                                                                                                    \
    rc = launch_attn_cluster_g<GG>(cfg, plan, q, q_stride, kc, vc, cache_batch_stride, n_heads, pos, max_ctx, scale, \
                                   out, err);                                                                 \
    break;
  switch (G) {
    QD_ATTN_G(1)
    QD_ATTN_G(2)
    QD_ATTN_G(3)
    QD_ATTN_G(4)
    QD_ATTN_G(5)
    QD_ATTN_G(6)
    QD_ATTN_G(7)
    QD_ATTN_G(8)
    default: return QD_ERR_UNSUPPORTED;
  }
#undef QD_ATTN_G
  return rc == cudaSuccess ? QD_OK : QD_ERR_CUDA;
}

qd_status launch_qkv_post(const float* qkv, int64_t qkv_stride, int batch, const QkvEpilogue& e, uint32_t* err,
                          cudaStream_t stream, bool pdl) {
  const int v_rows = e.k_rows;  // as many value rows as key rows
  const int pairs = (e.q_rows + e.k_rows + v_rows) / 2;
  const dim3 grid((unsigned)grid1d(pairs, 256), (unsigned)batch);
  return launch_k(k_qkv_post, grid, dim3(256), 0, stream, pdl, qkv, qkv_stride, e, v_rows, err);
}

qd_status launch_swiglu(const float* g, const float* u, float* out, int64_t n, int batch, cudaStream_t stream) {
  const int64_t total = n * batch;
  k_swiglu<<<grid1d(total, 256), 256, 0, stream>>>(g, u, out, total);
  return launch_status();
}

qd_status launch_argmax(const float* logits, int64_t n, int batch, int32_t* out, int32_t* pos_to_advance,
                        cudaStream_t stream) {
  k_argmax<<<batch, 1024, 0, stream>>>(logits, n, out, pos_to_advance);
  return launch_status();
}

qd_status launch_embed(int fmt, const PackedView& E, const int32_t* tokens, int batch, float* x, uint32_t* err,
                       cudaStream_t stream) {
  k_embed<<<batch, 256, 0, stream>>>(fmt, E, tokens, x, err);
  return launch_status();
}

// ------------------------------------------------------------------ fixed scratch
// Scratch for qd_gqa_decode_attn_noalloc: a file-scope device array that the driver
// reserves when the library's module is loaded on a device and keeps until the process
// exits.  Host code must not use its name as an address; the device address comes from
// cudaGetSymbolAddress, looked up once per device.
constexpr size_t kAttnScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_attn_scratch[kAttnScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up on first use).
qd_status attn_scratch_ptr(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return QD_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QD_OK;
}
}  // namespace

}  // namespace qd

using namespace qd;

extern "C" {

qd_status qd_rmsnorm(const float* x, const float* g, float* out, int n, int batch, float eps, qd_stream_t stream) {
  if (!x || !g || !out) return QD_ERR_INVALID_ARG;
  if (n < 1 || n > 65536 || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  if (!(eps >= 0.f)) return QD_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(g) || !aligned16(out)) return QD_ERR_ALIGN;
  return launch_rmsnorm(x, g, out, n, batch, eps, (cudaStream_t)stream);
}

// Angles p * theta^(-2i/hd) in double, (cos, sin) rounded to f32 (Go "llm"
// "Design points": RoPE angles are computed on the CPU in double precision).
qd_status qd_rope_table(float theta, int head_dim, int ctx, float* dst_host) {
  if (!dst_host) return QD_ERR_INVALID_ARG;
  if (head_dim < 2 || (head_dim & 1) || ctx < 1) return QD_ERR_SHAPE;
  if (!(theta > 0.f)) return QD_ERR_INVALID_ARG;
  const int half = head_dim / 2;
  for (int p = 0; p < ctx; ++p)
    for (int i = 0; i < half; ++i) {
      const double a = (double)p * std::pow((double)theta, -2.0 * (double)i / (double)head_dim);
      dst_host[((int64_t)p * half + i) * 2] = (float)std::cos(a);
      dst_host[((int64_t)p * half + i) * 2 + 1] = (float)std::sin(a);
    }
  return QD_OK;
}

qd_status qd_rope(float* v, int n_heads, int head_dim, int64_t batch_stride, const int32_t* pos,
                  qd_rope_pairing pairing, const float* cos_sin, int max_ctx, int batch, qd_stream_t stream) {
  if (!v || !pos || !cos_sin) return QD_ERR_INVALID_ARG;
  if (pairing != QD_ROPE_ADJACENT && pairing != QD_ROPE_HALF) return QD_ERR_UNSUPPORTED;
  if (n_heads < 1 || head_dim < 2 || (head_dim & 1) || max_ctx < 1 || batch < 1 || batch > QD_MAX_BATCH)
    return QD_ERR_SHAPE;
  if (batch_stride < (int64_t)n_heads * head_dim && batch > 1) return QD_ERR_SHAPE;
  if (!aligned16(v) || !aligned16(cos_sin)) return QD_ERR_ALIGN;
  return launch_rope(v, n_heads, head_dim, batch_stride, pos, pairing, cos_sin, max_ctx, batch, nullptr,
                     (cudaStream_t)stream);
}

qd_status qd_kv_append(const float* k, const float* v, int64_t src_batch_stride, float* k_cache, float* v_cache,
                       int n_kv_heads, int head_dim, const int32_t* pos, int max_ctx, int batch,
                       qd_stream_t stream) {
  if (!k || !v || !k_cache || !v_cache || !pos) return QD_ERR_INVALID_ARG;
  if (n_kv_heads < 1 || head_dim < 1 || max_ctx < 1 || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return QD_ERR_ALIGN;
  const int64_t cbs = (int64_t)n_kv_heads * max_ctx * head_dim;
  return launch_kv_append(k, v, src_batch_stride, k_cache, v_cache, n_kv_heads, head_dim, pos, max_ctx, batch, cbs,
                          nullptr, (cudaStream_t)stream);
}

size_t qd_gqa_decode_attn_workspace(int n_heads, int head_dim, int max_ctx, int batch) {
  if (n_heads < 1 || head_dim != 64 || max_ctx < 1 || batch < 1 || batch > QD_MAX_BATCH) return 0;
  return attn_workspace_bytes(n_heads, head_dim, max_ctx, batch);
}

qd_status qd_gqa_decode_attn(const float* q, int64_t q_batch_stride, const float* k_cache, const float* v_cache,
                             float* out, int n_heads, int n_kv_heads, int head_dim, const int32_t* pos, int max_ctx,
                             int batch, void* workspace, size_t workspace_bytes, qd_stream_t stream) {
  if (!q || !k_cache || !v_cache || !out || !pos || !workspace) return QD_ERR_INVALID_ARG;
  if (head_dim != 64) return QD_ERR_UNSUPPORTED;
  if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || n_heads / n_kv_heads > 8) return QD_ERR_SHAPE;
  if (max_ctx < 1 || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  if (batch > 1 && q_batch_stride < (int64_t)n_heads * head_dim) return QD_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(workspace))
    return QD_ERR_ALIGN;
  if ((q_batch_stride & 1) != 0) return QD_ERR_ALIGN;
  if (workspace_bytes < attn_workspace_bytes(n_heads, head_dim, max_ctx, batch)) return QD_ERR_NOMEM;
  const int64_t cbs = (int64_t)n_kv_heads * max_ctx * head_dim;
  return launch_attention(q, q_batch_stride, k_cache, v_cache, cbs, out, n_heads, n_kv_heads, head_dim, pos, max_ctx,
                          batch, workspace, nullptr, (cudaStream_t)stream);
}

// The same attention as qd_gqa_decode_attn, with its partial results kept in the
// library's fixed device scratch instead of a caller-provided workspace, so the call
// allocates nothing.  Every call shares that one scratch array; each call writes every
// partial it later reads, so nothing needs clearing, but two calls that overlap on the GPU
// (on different streams) race on it.
qd_status qd_gqa_decode_attn_noalloc(const float* q, int64_t q_batch_stride, const float* k_cache,
                                     const float* v_cache, float* out, int n_heads, int n_kv_heads, int head_dim,
                                     const int32_t* pos, int max_ctx, int batch, qd_stream_t stream) {
  if (!q || !k_cache || !v_cache || !out || !pos) return QD_ERR_INVALID_ARG;
  if (head_dim != 64) return QD_ERR_UNSUPPORTED;
  if (n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || n_heads / n_kv_heads > 8) return QD_ERR_SHAPE;
  if (max_ctx < 1 || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  if (batch > 1 && q_batch_stride < (int64_t)n_heads * head_dim) return QD_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return QD_ERR_ALIGN;
  if ((q_batch_stride & 1) != 0) return QD_ERR_ALIGN;
  if (attn_workspace_bytes(n_heads, head_dim, max_ctx, batch) > kAttnScratchBytes) return QD_ERR_NOMEM;
  void* ws = nullptr;
  const qd_status st = attn_scratch_ptr(&ws);
  if (st != QD_OK) return st;
  const int64_t cbs = (int64_t)n_kv_heads * max_ctx * head_dim;
  return launch_attention(q, q_batch_stride, k_cache, v_cache, cbs, out, n_heads, n_kv_heads, head_dim, pos, max_ctx,
                          batch, ws, nullptr, (cudaStream_t)stream);
}

qd_status qd_swiglu(const float* gate, const float* up, float* out, int64_t n, int batch, qd_stream_t stream) {
  if (!gate || !up || !out) return QD_ERR_INVALID_ARG;
  if (n < 1 || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  return launch_swiglu(gate, up, out, n, batch, (cudaStream_t)stream);
}

qd_status qd_argmax(const float* logits, int64_t n, int batch, int32_t* out_idx, qd_stream_t stream) {
  if (!logits || !out_idx) return QD_ERR_INVALID_ARG;
  if (n < 1 || n > 0x7FFFFFFF || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  return launch_argmax(logits, n, batch, out_idx, nullptr, (cudaStream_t)stream);
}

qd_status qd_embed(qd_fmt fmt, const void* E, int64_t vocab, int64_t dim, const int32_t* tokens, int batch,
                   float* x, qd_stream_t stream) {
  if (!fmt_ok(fmt)) return QD_ERR_UNSUPPORTED;
  if (!E || !tokens || !x) return QD_ERR_INVALID_ARG;
  if (!shape_ok(fmt, vocab, dim) || batch < 1 || batch > QD_MAX_BATCH) return QD_ERR_SHAPE;
  if (!aligned16(E) || !aligned16(x)) return QD_ERR_ALIGN;
  return launch_embed(fmt, packed_view(fmt, E, vocab, dim), tokens, batch, x, nullptr, (cudaStream_t)stream);
}

}  // extern "C"
