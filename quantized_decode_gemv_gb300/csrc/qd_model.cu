// The decode-step driver: a llama-style model over caller-owned weight and state
// memory, one CUDA graph replay per token.
//
// Step order (llmoxide blog s7 "The block, and the residual stream"; dasLLAMA
// 8.7.1.6 forward):
//   x = embed(token)
//   per layer: xn = rmsnorm(x)*attn_norm; [q|k|v] = Wqkv xn; rope(q, k) at pos;
//              cache[pos] = k, v; o = attention(q, cache[0..pos]); x += Wo o;
//              xn = rmsnorm(x)*ffn_norm; a = silu(Wg xn) * (Wu xn); x += Wd a
//   logits = W_out (rmsnorm(x)*out_norm); token = argmax(logits); pos += 1
// As in the Go "llm" package ("Design points": one submit per token, only the
// 4-byte token read back), the whole step is recorded once and replayed: here as
// a CUDA graph per batch size whose kernels read each sequence's position from
// device memory, so the same graph serves every token.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "qd_internal.cuh"

using namespace qd;

namespace {

struct LayerOff {
  size_t attn_norm, ffn_norm, wqkv, wo, wgu, wd;
};

struct Layout {
  // weights
  size_t emb, head, out_norm;
  std::vector<LayerOff> layer;
  size_t weight_bytes;
  // state
  size_t kc, vc, x, xn, qkv, q, att, act, logits, am_key, am_cnt, tok_in, tok_out, pos, err,
      rope;
  size_t attn_ws, attn_cnt;  // flat-split attention: partials and per-pair counters
  size_t xq;                 // act_q8: the quantised input of each product, one slot each
  size_t xq_slot;            // bytes per slot
  bool attn_flat;
  int attn_ctas;  // its grid (one CTA per SM), fixed with the workspace size
  size_t state_bytes;
  int64_t qkv_rows, cache_batch_stride, cache_layer_stride;
};

// The format of each class of layer matrix (w_fmt for all of them unless mixed_fmt).
inline int fmt_qkv(const qd_config& c) { return c.mixed_fmt ? c.qkv_fmt : c.w_fmt; }
inline int fmt_wo(const qd_config& c) { return c.mixed_fmt ? c.wo_fmt : c.w_fmt; }
inline int fmt_gu(const qd_config& c) { return c.mixed_fmt ? c.gate_up_fmt : c.w_fmt; }
inline int fmt_down(const qd_config& c) { return c.mixed_fmt ? c.down_fmt : c.w_fmt; }
inline bool uniform_fmt(const qd_config& c) {
  return fmt_qkv(c) == fmt_wo(c) && fmt_wo(c) == fmt_gu(c) && fmt_gu(c) == fmt_down(c);
}
// Formats the decode step takes: every one but per-row INT4.  The streaming and tensor-
// core GEMVs fuse the norm and the epilogues for theirs; for the others the step runs the
// norm, the QKV epilogue and the argmax as separate kernels.
inline bool step_fmt_ok(int fmt) { return fmt_ok(fmt) && fmt != QD_I4_ROW; }
inline bool q8_fmt(int fmt) { return fmt == QD_Q4_0 || fmt == QD_Q8_0; }

bool config_ok(const qd_config* c) {
  if (!c) return false;
  if (c->layers < 1 || c->dim < 1 || c->ffn < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->vocab < 1) return false;
  if (c->head_dim != 64) return false;  // the decode-attention kernel's head width
  if (c->n_heads % c->n_kv_heads || c->n_heads / c->n_kv_heads > 8) return false;
  if (c->max_ctx < 1 || c->max_batch < 1 || c->max_batch > QD_MAX_BATCH) return false;
  if (c->pairing != QD_ROPE_ADJACENT && c->pairing != QD_ROPE_HALF) return false;
  if (c->kv_f16 != 0 && c->kv_f16 != 1) return false;
  if (c->act_q8 != 0 && c->act_q8 != 1) return false;
  if (c->mixed_fmt != 0 && c->mixed_fmt != 1) return false;
  const int fq = fmt_qkv(*c), fo = fmt_wo(*c), fg = fmt_gu(*c), fd = fmt_down(*c);
  if (!step_fmt_ok(fq) || !step_fmt_ok(fo) || !step_fmt_ok(fg) || !step_fmt_ok(fd) || !step_fmt_ok(c->emb_fmt))
    return false;
  // the integer products over Q8_0 activations take Q4_0 and Q8_0 weights
  if (c->act_q8 && !(q8_fmt(fq) && q8_fmt(fo) && q8_fmt(fg) && q8_fmt(fd) && q8_fmt(c->emb_fmt))) return false;
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.f)) return false;
  const int64_t QD = (int64_t)c->n_heads * c->head_dim, KD = (int64_t)c->n_kv_heads * c->head_dim;
  if (!shape_ok(fq, QD + 2 * KD, c->dim) || !shape_ok(fo, c->dim, QD) || !shape_ok(fg, 2 * (int64_t)c->ffn, c->dim) ||
      !shape_ok(fd, c->dim, c->ffn))
    return false;
  if (!shape_ok(c->emb_fmt, c->vocab, c->dim)) return false;
  return true;
}

Layout make_layout(const qd_config* c) {
  Layout L{};
  const int64_t D = c->dim, F = c->ffn, QD = (int64_t)c->n_heads * c->head_dim;
  const int64_t KD = (int64_t)c->n_kv_heads * c->head_dim, B = c->max_batch;
  L.qkv_rows = QD + 2 * KD;
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  L.emb = take(packed_bytes(c->emb_fmt, c->vocab, D));
  L.head = c->tied ? L.emb : take(packed_bytes(c->emb_fmt, c->vocab, D));
  L.out_norm = take(4 * D);
  L.layer.resize(c->layers);
  for (int l = 0; l < c->layers; ++l) {
    LayerOff& o = L.layer[l];
    o.attn_norm = take(4 * D);
    o.ffn_norm = take(4 * D);
    o.wqkv = take(packed_bytes(fmt_qkv(*c), L.qkv_rows, D));
    o.wo = take(packed_bytes(fmt_wo(*c), D, QD));
    o.wgu = take(packed_bytes(fmt_gu(*c), 2 * F, D));
    o.wd = take(packed_bytes(fmt_down(*c), D, F));
  }
  L.weight_bytes = off;

  off = 0;
  L.cache_batch_stride = KD * c->max_ctx;
  L.cache_layer_stride = L.cache_batch_stride * B;
  const size_t cache = (size_t)c->layers * L.cache_layer_stride * (c->kv_f16 ? 2 : 4);
  L.kc = take(cache);
  L.vc = take(cache);
  L.x = take(4 * B * D);
  L.xn = take(4 * B * D);
  L.qkv = take(4 * B * L.qkv_rows);
  L.q = take(4 * B * QD);
  L.att = take(4 * B * QD);
  L.act = take(4 * B * F);
  L.logits = take(4 * B * (size_t)c->vocab);
  L.am_key = take(8 * B);
  L.am_cnt = take(4);
  L.tok_in = take(4 * B);
  L.tok_out = take(4 * B);
  L.pos = take(4 * B);
  L.err = take(4);
  L.rope = take((size_t)c->max_ctx * c->head_dim * 4);
  L.attn_flat = c->kv_f16 || attn_use_flat(c->n_kv_heads, c->max_batch, c->max_ctx);
  L.attn_ctas = attn_flat_ctas();
  L.attn_ws = L.attn_flat ? take(4 * attn_flat_ws_floats(c->n_heads, c->n_kv_heads, c->max_batch, L.attn_ctas)) : 0;
  L.attn_cnt = L.attn_flat ? take(4 * (size_t)c->n_kv_heads * c->max_batch) : 0;
  // one slot per quantised input (4 per layer, then the head's), so after a step every
  // product's codes can still be read
  L.xq_slot = c->act_q8 ? align_up(q8_buffer_bytes((int)B, std::max(std::max(D, F), QD), false), 256) : 0;
  L.xq = c->act_q8 ? take(L.xq_slot * (4 * (size_t)c->layers + 1)) : 0;
  L.state_bytes = off;
  return L;
}

__global__ void k_fill_zero(uint4* __restrict__ p, int64_t n16) {
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < n16; t += (int64_t)gridDim.x * blockDim.x)
    p[t] = make_uint4(0, 0, 0, 0);
}

qd_status zero_region(void* p, size_t bytes, cudaStream_t s) {
  const int64_t n16 = (int64_t)(bytes / 16);
  if (n16 == 0) return QD_OK;
  int64_t g = (n16 + 255) / 256;
  if (g > 152 * 64) g = 152 * 64;
  k_fill_zero<<<(unsigned)g, 256, 0, s>>>(static_cast<uint4*>(p), n16);
  return launch_status();
}

}  // namespace

struct qd_model {
  qd_config cfg;
  Layout L;
  uint8_t* w;  // weight memory (caller-owned)
  uint8_t* s;  // state memory (caller-owned)
  // the layers as one thread-block cluster per sequence, when the model fits it
  StepClusterModel scm{};
  StepClusterPlan plan{};
  bool cluster_ok = false;
  int step_path = QD_STEP_AUTO;
  cudaStream_t capture_stream = nullptr;
  cudaGraphExec_t graph[QD_MAX_BATCH + 1] = {};
  int launches = 0;

  float* f(size_t off) { return reinterpret_cast<float*>(s + off); }
  int32_t* i(size_t off) { return reinterpret_cast<int32_t*>(s + off); }
  PackedView W(int fmt, size_t off, int64_t rows, int64_t cols) const { return packed_view(fmt, w + off, rows, cols); }
};

namespace {

#define QD_TRY(expr)                   \
  do {                                 \
    const qd_status st_ = (expr);      \
    if (st_ != QD_OK) return st_;      \
  } while (0)

// Enqueue one decode step for `batch` sequences; counts the kernels it launches.
// Every kernel after the first is launched as a programmatic dependent of its
// predecessor (it starts prefetching weights while the predecessor finishes).
qd_status enqueue_step(qd_model* m, int batch, cudaStream_t st) {
  const qd_config& c = m->cfg;
  const Layout& L = m->L;
  const int64_t D = c.dim, F = c.ffn, QD = (int64_t)c.n_heads * c.head_dim, KD = (int64_t)c.n_kv_heads * c.head_dim;
  uint32_t* err = reinterpret_cast<uint32_t*>(m->s + L.err);
  int32_t* pos = m->i(L.pos);
  float *x = m->f(L.x), *xn = m->f(L.xn), *qkv = m->f(L.qkv), *q = m->f(L.q), *att = m->f(L.att),
        *act = m->f(L.act);
  int n = 0;
  const bool cluster = m->cluster_ok && m->step_path == QD_STEP_CLUSTER;
  if (cluster) {
    // embedding and every layer in one cluster kernel per sequence; x is the head's input
    QD_TRY(launch_step_cluster(m->scm, m->plan, m->i(L.tok_in), pos, x, err, batch, st));
    ++n;
  } else {
    QD_TRY(launch_embed(c.emb_fmt, m->W(c.emb_fmt, L.emb, c.vocab, D), m->i(L.tok_in), batch, x, err, st));
    ++n;
  }
  auto args = [&](int fmt, PackedView W, const float* in, float* y, GemvMode mode) {
    GemvArgs a;
    a.fmt = fmt;
    a.W = W;
    a.x = in;
    a.y = y;
    a.batch = batch;
    a.mode = mode;
    a.err = err;
    a.pdl = true;
    return a;
  };
  // ggml-exact products (act_q8): the Q8_0 quantisation of the product's input (fused with
  // the RMSNorm when it has one), then the integer product; launched without programmatic
  // dependence (they run once their predecessor has completed and never let their
  // successor start early).
  auto q8prod = [&](int slot, int fmt, PackedView W, const float* in, const float* gains, float* y,
                    GemvMode mode) -> qd_status {
    void* xq = m->s + L.xq + (size_t)slot * L.xq_slot;
    if (gains)  // the norm quantised as it is formed (the same f32 values as the norm kernel)
      QD_TRY(launch_rmsnorm_q8(in, gains, (int)W.cols, c.eps, batch, xq, st));
    else
      QD_TRY(launch_quantize_q8(in, batch, W.cols, false, xq, st));
    QD_TRY(launch_q_gemv_q8(fmt, W, xq, batch, y, mode, st));
    n += 2;
    return QD_OK;
  };
  // GEMV with RMSNorm fused into its prologue when the streaming kernel runs; a
  // separate norm kernel (into xn) otherwise.
  auto normed = [&](GemvArgs a, const float* gains) -> qd_status {
    if (gemv_fuses_norm(a, gains)) {
      a.norm_g = gains;
      a.eps = c.eps;
      ++n;
      return launch_q_gemv(a, st);
    }
    QD_TRY(launch_rmsnorm(a.x, gains, xn, (int)D, batch, c.eps, st));
    a.x = xn;
    n += 2;
    return launch_q_gemv(a, st);
  };
  for (int l = 0; l < (cluster ? 0 : c.layers); ++l) {
    const LayerOff& o = L.layer[l];
    const int64_t esz = c.kv_f16 ? 2 : 4;  // bytes per cache element
    void* kc = m->s + L.kc + (int64_t)l * L.cache_layer_stride * esz;
    void* vc = m->s + L.vc + (int64_t)l * L.cache_layer_stride * esz;
    // QKV projection with RoPE and the cache append fused into its epilogue
    const int fq = fmt_qkv(c), fo = fmt_wo(c), fg = fmt_gu(c), fd = fmt_down(c);
    GemvArgs qa = args(fq, m->W(fq, o.wqkv, L.qkv_rows, D), x, qkv, kGemvQKV);
    QkvEpilogue& e = qa.qkv;
    e.q_rows = (int)QD;
    e.k_rows = (int)KD;
    e.head_dim = c.head_dim;
    e.pairing = c.pairing;
    e.pos = pos;
    e.rope = m->f(L.rope);
    e.q_out = q;
    e.q_stride = QD;
    e.kc = kc;
    e.vc = vc;
    e.kv_f16 = c.kv_f16 != 0;
    e.cache_batch_stride = L.cache_batch_stride;
    e.max_ctx = c.max_ctx;
    const float* attn_norm = reinterpret_cast<const float*>(m->w + o.attn_norm);
    if (c.act_q8) {
      QD_TRY(q8prod(4 * l, fq, qa.W, x, attn_norm, qkv, kGemvStore));
      QD_TRY(launch_qkv_post(qkv, L.qkv_rows, batch, e, err, st, true));
      ++n;
    } else if (gemv_fuses_norm(qa, attn_norm)) {
      QD_TRY(normed(qa, attn_norm));
    } else {
      GemvArgs raw = qa;
      raw.mode = kGemvStore;
      QD_TRY(normed(raw, attn_norm));
      QD_TRY(launch_qkv_post(qkv, L.qkv_rows, batch, e, err, st, true));
      ++n;
    }
    if (L.attn_flat)
      QD_TRY(launch_attention_flat(q, QD, kc, vc, c.kv_f16 != 0, L.cache_batch_stride, att, c.n_heads, c.n_kv_heads,
                                   c.head_dim, pos, c.max_ctx, batch, L.attn_ctas, m->f(L.attn_ws),
                                   reinterpret_cast<unsigned int*>(m->s + L.attn_cnt), err, st, true));
    else
      QD_TRY(launch_attention_cluster(q, QD, static_cast<const float*>(kc), static_cast<const float*>(vc),
                                      L.cache_batch_stride, att, c.n_heads, c.n_kv_heads,
                                      c.head_dim, pos, c.max_ctx, batch, err, st, true));
    ++n;
    if (c.act_q8) {
      QD_TRY(q8prod(4 * l + 1, fo, m->W(fo, o.wo, D, QD), att, nullptr, x, kGemvAccumulate));
      QD_TRY(q8prod(4 * l + 2, fg, m->W(fg, o.wgu, 2 * F, D), x, reinterpret_cast<const float*>(m->w + o.ffn_norm),
                    act, kGemvSwiGLU));
      QD_TRY(q8prod(4 * l + 3, fd, m->W(fd, o.wd, D, F), act, nullptr, x, kGemvAccumulate));
      continue;
    }
    QD_TRY(launch_q_gemv(args(fo, m->W(fo, o.wo, D, QD), att, x, kGemvAccumulate), st));
    ++n;
    QD_TRY(normed(args(fg, m->W(fg, o.wgu, 2 * F, D), x, act, kGemvSwiGLU),
                  reinterpret_cast<const float*>(m->w + o.ffn_norm)));
    QD_TRY(launch_q_gemv(args(fd, m->W(fd, o.wd, D, F), act, x, kGemvAccumulate), st));
    ++n;
  }
  // output head with the greedy argmax (and the position advance) fused in
  GemvArgs ha = args(c.emb_fmt, m->W(c.emb_fmt, L.head, c.vocab, D), x, m->f(L.logits), kGemvArgmax);
  ha.am.key = reinterpret_cast<unsigned long long*>(m->s + L.am_key);
  ha.am.counter = reinterpret_cast<unsigned int*>(m->s + L.am_cnt);
  ha.am.tok_out = m->i(L.tok_out);
  ha.am.pos = pos;
  const float* out_norm = reinterpret_cast<const float*>(m->w + L.out_norm);
  if (c.act_q8) {
    QD_TRY(q8prod(4 * c.layers, c.emb_fmt, ha.W, x, out_norm, m->f(L.logits), kGemvStore));
    QD_TRY(launch_argmax(m->f(L.logits), c.vocab, batch, m->i(L.tok_out), pos, st));
    ++n;
  } else if (gemv_fuses_norm(ha, out_norm)) {
    QD_TRY(normed(ha, out_norm));
  } else {
    ha.mode = kGemvStore;
    QD_TRY(normed(ha, out_norm));
    QD_TRY(launch_argmax(m->f(L.logits), c.vocab, batch, m->i(L.tok_out), pos, st));
    ++n;
  }
  m->launches = n;
  return QD_OK;
}

qd_status get_graph(qd_model* m, int batch, cudaGraphExec_t* out) {
  if (m->graph[batch]) {
    *out = m->graph[batch];
    return QD_OK;
  }
  cudaStream_t cs = m->capture_stream;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return QD_ERR_CUDA;
  const qd_status st = enqueue_step(m, batch, cs);
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(cs, &g);
  if (st != QD_OK || e != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return st != QD_OK ? st : QD_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&ex, g, 0);
  cudaGraphDestroy(g);
  if (ei != cudaSuccess) return QD_ERR_CUDA;
  m->graph[batch] = ex;
  *out = ex;
  return QD_OK;
}


// ---- batched prefill (llmoxide blog s11 "Prefill and decode": the prompt's t tokens go
// through every product as one t-row matrix, one read of each weight tile for all of them)

// ppos[i] = pos[seq] + i: each prompt token's position.
__global__ void k_prefill_pos(const int32_t* __restrict__ pos_seq, int32_t* __restrict__ ppos, int t) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < t; i += gridDim.x * blockDim.x) ppos[i] = *pos_seq + i;
}
// pos[seq] += n (the head's argmax adds the last one).
__global__ void k_pos_add(int32_t* pos_seq, int n) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *pos_seq += n;
}

struct PrefillLayout {
  size_t tok, ppos, x, xn, qkv, q, att, act, gemm_ws, attn_ws, attn_cnt, total;
};

constexpr int kPrefillChunk = 16;  // tokens per flat-attention launch (binary16 cache)
constexpr int kPrefillRows = 16;   // tokens per batched-GEMV launch (the tensor-core GEMV's widest)

PrefillLayout prefill_layout(const qd_config& c, int64_t qkv_rows, int t) {
  PrefillLayout P{};
  const int64_t D = c.dim, F = c.ffn, QD = (int64_t)c.n_heads * c.head_dim;
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  P.tok = take(4 * (size_t)t);
  P.ppos = take(4 * (size_t)t);
  P.x = take(4 * (size_t)t * D);
  P.xn = take(4 * (size_t)t * D);
  P.qkv = take(4 * (size_t)t * qkv_rows);
  P.q = take(4 * (size_t)t * QD);
  P.att = take(4 * (size_t)t * QD);
  P.act = take(4 * (size_t)t * F);
  P.gemm_ws = take(std::max(gemm_workspace_bytes(D, t), std::max(gemm_workspace_bytes(QD, t), gemm_workspace_bytes(F, t))));
  if (c.kv_f16) {
    P.attn_ws = take(4 * attn_flat_ws_floats(c.n_heads, c.n_kv_heads, kPrefillChunk, attn_flat_ctas()));
    P.attn_cnt = take(4 * (size_t)kPrefillChunk * c.n_kv_heads);
  } else {
    P.attn_ws = take(attn_workspace_bytes(c.n_heads, c.head_dim, c.max_ctx, t));
    P.attn_cnt = 0;
  }
  P.total = off;
  return P;
}

// Whether the prefill products may run on the tensor-core GEMM (binary16 weights) rather
// than the batched GEMVs (the decode step's arithmetic); each product also needs a format
// the GEMM takes (Q4_0, Q8_0, INT8 rows).
bool prefill_uses_gemm(const qd_config& c, int t, unsigned flags) {
  if (flags & QD_PREFILL_EXACT) return false;
  if (t <= kPrefillRows) return false;  // one GEMV launch per product is as fast
  const int64_t QD = (int64_t)c.n_heads * c.head_dim;
  return c.dim % 64 == 0 && QD % 64 == 0 && c.ffn % 64 == 0;
}
inline bool gemm_fmt(int fmt) { return fmt == QD_Q4_0 || fmt == QD_Q8_0 || fmt == QD_I8_ROW; }

qd_status enqueue_prefill(qd_model* m, int seq, int t, unsigned flags, uint8_t* ws, cudaStream_t st) {
  const qd_config& c = m->cfg;
  const Layout& L = m->L;
  const PrefillLayout P = prefill_layout(c, L.qkv_rows, t);
  const int64_t D = c.dim, F = c.ffn, QD = (int64_t)c.n_heads * c.head_dim, KD = (int64_t)c.n_kv_heads * c.head_dim;
  uint32_t* err = reinterpret_cast<uint32_t*>(m->s + L.err);
  int32_t* pos_seq = m->i(L.pos) + seq;
  int32_t* ppos = reinterpret_cast<int32_t*>(ws + P.ppos);
  float* x = reinterpret_cast<float*>(ws + P.x);
  float* xn = reinterpret_cast<float*>(ws + P.xn);
  float* qkv = reinterpret_cast<float*>(ws + P.qkv);
  float* q = reinterpret_cast<float*>(ws + P.q);
  float* att = reinterpret_cast<float*>(ws + P.att);
  float* act = reinterpret_cast<float*>(ws + P.act);
  const bool gemm = prefill_uses_gemm(c, t, flags);

  k_prefill_pos<<<(t + 255) / 256, 256, 0, st>>>(pos_seq, ppos, t);
  QD_TRY(launch_status());
  QD_TRY(launch_embed(c.emb_fmt, m->W(c.emb_fmt, L.emb, c.vocab, D), reinterpret_cast<int32_t*>(ws + P.tok), t, x,
                      err, st));
  if (c.kv_f16) QD_TRY(zero_region(ws + P.attn_cnt, align_up(4 * (size_t)kPrefillChunk * c.n_kv_heads, 16), st));

  // one product over the t rows of `in`: the GEMM, or batched GEMVs of up to 16 rows
  auto product = [&](int fmt, PackedView W, const float* in, float* y, GemvMode mode) -> qd_status {
    if (gemm && gemm_fmt(fmt)) {
      const int gm = mode == kGemvAccumulate ? kGemmAccumulate : mode == kGemvSwiGLU ? kGemmSwiGLU : kGemmStore;
      return launch_q_gemm(fmt, W, in, y, t, ws + P.gemm_ws, err, st, gm);
    }
    const int64_t ycols = mode == kGemvSwiGLU ? W.rows / 2 : W.rows;
    for (int c0 = 0; c0 < t; c0 += kPrefillRows) {
      GemvArgs a;
      a.fmt = fmt;
      a.W = W;
      a.x = in + (int64_t)c0 * W.cols;
      a.y = y + (int64_t)c0 * ycols;
      a.batch = std::min(kPrefillRows, t - c0);
      a.mode = mode;
      a.err = err;
      QD_TRY(launch_q_gemv(a, st));
    }
    return QD_OK;
  };

  for (int l = 0; l < c.layers; ++l) {
    const LayerOff& o = L.layer[l];
    const int64_t esz = c.kv_f16 ? 2 : 4;
    // this sequence's cache rows of layer l; every prompt token appends into the same one
    uint8_t* kc = m->s + L.kc + ((int64_t)l * L.cache_layer_stride + (int64_t)seq * L.cache_batch_stride) * esz;
    uint8_t* vc = m->s + L.vc + ((int64_t)l * L.cache_layer_stride + (int64_t)seq * L.cache_batch_stride) * esz;
    QD_TRY(launch_rmsnorm(x, reinterpret_cast<const float*>(m->w + o.attn_norm), xn, (int)D, t, c.eps, st));
    const int fq = fmt_qkv(c), fo = fmt_wo(c), fg = fmt_gu(c), fd = fmt_down(c);
    QD_TRY(product(fq, m->W(fq, o.wqkv, L.qkv_rows, D), xn, qkv, kGemvStore));
    QkvEpilogue e;
    e.q_rows = (int)QD;
    e.k_rows = (int)KD;
    e.head_dim = c.head_dim;
    e.pairing = c.pairing;
    e.pos = ppos;
    e.rope = m->f(L.rope);
    e.q_out = q;
    e.q_stride = QD;
    e.kc = kc;
    e.vc = vc;
    e.kv_f16 = c.kv_f16 != 0;
    e.cache_batch_stride = 0;
    e.max_ctx = c.max_ctx;
    QD_TRY(launch_qkv_post(qkv, L.qkv_rows, t, e, err, st, false));
    // causal attention: token i over positions 0 .. ppos[i] of the one cache
    if (c.kv_f16) {
      for (int c0 = 0; c0 < t; c0 += kPrefillChunk)
        QD_TRY(launch_attention_flat(q + (int64_t)c0 * QD, QD, kc, vc, true, 0, att + (int64_t)c0 * QD, c.n_heads,
                                     c.n_kv_heads, c.head_dim, ppos + c0, c.max_ctx, std::min(kPrefillChunk, t - c0),
                                     attn_flat_ctas(), reinterpret_cast<float*>(ws + P.attn_ws),
                                     reinterpret_cast<unsigned int*>(ws + P.attn_cnt), err, st, false));
    } else {
      QD_TRY(launch_attention(q, QD, reinterpret_cast<const float*>(kc), reinterpret_cast<const float*>(vc), 0, att,
                              c.n_heads, c.n_kv_heads, c.head_dim, ppos, c.max_ctx, t, ws + P.attn_ws, err, st));
    }
    QD_TRY(product(fo, m->W(fo, o.wo, D, QD), att, x, kGemvAccumulate));
    QD_TRY(launch_rmsnorm(x, reinterpret_cast<const float*>(m->w + o.ffn_norm), xn, (int)D, t, c.eps, st));
    QD_TRY(product(fg, m->W(fg, o.wgu, 2 * F, D), xn, act, kGemvSwiGLU));
    QD_TRY(product(fd, m->W(fd, o.wd, D, F), act, x, kGemvAccumulate));
  }

  // the last token's logits and greedy token, as the decode step's head; the position
  // ends at pos[seq] + t (the argmax adds the last one)
  k_pos_add<<<1, 32, 0, st>>>(pos_seq, t - 1);
  QD_TRY(launch_status());
  float* logits = m->f(L.logits) + (int64_t)seq * c.vocab;
  GemvArgs ha;
  ha.fmt = c.emb_fmt;
  ha.W = m->W(c.emb_fmt, L.head, c.vocab, D);
  ha.x = x + (int64_t)(t - 1) * D;
  ha.y = logits;
  ha.batch = 1;
  ha.mode = kGemvArgmax;
  ha.err = err;
  ha.am.key = reinterpret_cast<unsigned long long*>(m->s + L.am_key) + seq;
  ha.am.counter = reinterpret_cast<unsigned int*>(m->s + L.am_cnt);
  ha.am.tok_out = m->i(L.tok_out) + seq;
  ha.am.pos = pos_seq;
  const float* out_norm = reinterpret_cast<const float*>(m->w + L.out_norm);
  if (gemv_fuses_norm(ha, out_norm)) {
    ha.norm_g = out_norm;
    ha.eps = c.eps;
    return launch_q_gemv(ha, st);
  }
  QD_TRY(launch_rmsnorm(ha.x, out_norm, xn, (int)D, 1, c.eps, st));
  ha.x = xn;
  ha.mode = kGemvStore;
  QD_TRY(launch_q_gemv(ha, st));
  return launch_argmax(logits, c.vocab, 1, m->i(L.tok_out) + seq, pos_seq, st);
}

}  // namespace

extern "C" {

size_t qd_model_weight_bytes(const qd_config* cfg) { return config_ok(cfg) ? make_layout(cfg).weight_bytes : 0; }
size_t qd_model_state_bytes(const qd_config* cfg) { return config_ok(cfg) ? make_layout(cfg).state_bytes : 0; }

qd_status qd_model_create(const qd_config* cfg, const void* const* src, void* weight_mem, size_t weight_bytes,
                          void* state_mem, size_t state_bytes, qd_stream_t stream, qd_model** out) {
  if (!cfg || !src || !weight_mem || !state_mem || !out) return QD_ERR_INVALID_ARG;
  *out = nullptr;
  if (!config_ok(cfg)) return QD_ERR_UNSUPPORTED;
  const int nt = 3 + 9 * cfg->layers;
  for (int t = 0; t < nt; ++t)
    if (!src[t] && !(t == 2 && cfg->tied)) return QD_ERR_INVALID_ARG;
  if (!aligned16(weight_mem) || !aligned16(state_mem)) return QD_ERR_ALIGN;
  for (int l = 0; l < cfg->layers; ++l)
    if (!aligned16(src[3 + 9 * l]) || !aligned16(src[3 + 9 * l + 5])) return QD_ERR_ALIGN;
  if (!aligned16(src[1])) return QD_ERR_ALIGN;
  Layout L = make_layout(cfg);
  if (weight_bytes < L.weight_bytes || state_bytes < L.state_bytes) return QD_ERR_NOMEM;

  qd_model* m = new (std::nothrow) qd_model();
  if (!m) return QD_ERR_NOMEM;
  m->cfg = *cfg;
  m->L = L;
  m->w = static_cast<uint8_t*>(weight_mem);
  m->s = static_cast<uint8_t*>(state_mem);
  cudaStream_t st = (cudaStream_t)stream;
  const int64_t D = cfg->dim, F = cfg->ffn, QD = (int64_t)cfg->n_heads * cfg->head_dim;
  const int64_t KD = (int64_t)cfg->n_kv_heads * cfg->head_dim;
  auto fail = [m](qd_status s) {
    delete m;
    return s;
  };
  auto copy_f32 = [&](size_t off, const void* p, int64_t n) -> qd_status {
    return cudaMemcpyAsync(m->w + off, p, 4 * n, cudaMemcpyDeviceToDevice, st) == cudaSuccess ? QD_OK : QD_ERR_CUDA;
  };
  qd_status s;
  if ((s = launch_repack_rows(cfg->emb_fmt, src[0], cfg->vocab, D, m->w + L.emb, cfg->vocab, 0, 1, st))) return fail(s);
  if (!cfg->tied &&
      (s = launch_repack_rows(cfg->emb_fmt, src[2], cfg->vocab, D, m->w + L.head, cfg->vocab, 0, 1, st)))
    return fail(s);
  if ((s = copy_f32(L.out_norm, src[1], D))) return fail(s);
  const int fq = fmt_qkv(*cfg), fo = fmt_wo(*cfg), fg = fmt_gu(*cfg), fd = fmt_down(*cfg);
  for (int l = 0; l < cfg->layers; ++l) {
    const void* const* T = src + 3 + 9 * l;
    const LayerOff& o = L.layer[l];
    if ((s = copy_f32(o.attn_norm, T[0], D))) return fail(s);
    if ((s = copy_f32(o.ffn_norm, T[5], D))) return fail(s);
    // fused QKV: q rows, then k rows, then v rows; with half pairing the rows of each
    // RoPE pair (i, i + head_dim/2) are made adjacent for the projection's epilogue
    const int pair_hd = cfg->pairing == QD_ROPE_HALF ? cfg->head_dim : 0;
    if ((s = launch_repack_rows(fq, T[1], QD, D, m->w + o.wqkv, L.qkv_rows, 0, 1, st, pair_hd))) return fail(s);
    if ((s = launch_repack_rows(fq, T[2], KD, D, m->w + o.wqkv, L.qkv_rows, QD, 1, st, pair_hd))) return fail(s);
    if ((s = launch_repack_rows(fq, T[3], KD, D, m->w + o.wqkv, L.qkv_rows, QD + KD, 1, st))) return fail(s);
    if ((s = launch_repack_rows(fo, T[4], D, QD, m->w + o.wo, D, 0, 1, st))) return fail(s);
    // gate/up interleaved: row 2i = gate row i, row 2i+1 = up row i
    if ((s = launch_repack_rows(fg, T[6], F, D, m->w + o.wgu, 2 * F, 0, 2, st))) return fail(s);
    if ((s = launch_repack_rows(fg, T[7], F, D, m->w + o.wgu, 2 * F, 1, 2, st))) return fail(s);
    if ((s = launch_repack_rows(fd, T[8], D, F, m->w + o.wd, D, 0, 1, st))) return fail(s);
  }
  if ((s = zero_region(m->s, L.state_bytes, st))) return fail(s);
  std::vector<float> table((size_t)cfg->max_ctx * cfg->head_dim);
  if ((s = qd_rope_table(cfg->rope_theta, cfg->head_dim, cfg->max_ctx, table.data()))) return fail(s);
  if (cudaMemcpyAsync(m->s + L.rope, table.data(), table.size() * 4, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return fail(QD_ERR_CUDA);
  if (cudaStreamCreateWithFlags(&m->capture_stream, cudaStreamNonBlocking) != cudaSuccess) return fail(QD_ERR_CUDA);
  if (!cfg->act_q8 && !cfg->kv_f16 && uniform_fmt(*cfg)) {
    StepClusterModel& sc = m->scm;
    sc.fmt = fq;
    sc.emb_fmt = cfg->emb_fmt;
    sc.emb = m->W(cfg->emb_fmt, L.emb, cfg->vocab, D);
    sc.w = m->w;
    const LayerOff& l0 = L.layer[0];
    sc.layer0 = (int64_t)l0.attn_norm;
    sc.layer_stride = cfg->layers > 1 ? (int64_t)(L.layer[1].attn_norm - l0.attn_norm) : 0;
    bool uniform = true;
    for (int l = 1; l < cfg->layers; ++l) {
      const LayerOff& o = L.layer[l];
      const int64_t base = sc.layer0 + (int64_t)l * sc.layer_stride;
      uniform = uniform && (int64_t)o.attn_norm == base && o.ffn_norm - o.attn_norm == l0.ffn_norm - l0.attn_norm &&
                o.wqkv - o.attn_norm == l0.wqkv - l0.attn_norm && o.wo - o.attn_norm == l0.wo - l0.attn_norm &&
                o.wgu - o.attn_norm == l0.wgu - l0.attn_norm && o.wd - o.attn_norm == l0.wd - l0.attn_norm;
    }
    sc.off_attn_norm = 0;
    sc.off_ffn_norm = (int64_t)(l0.ffn_norm - l0.attn_norm);
    sc.off_qkv = (int64_t)(l0.wqkv - l0.attn_norm);
    sc.off_wo = (int64_t)(l0.wo - l0.attn_norm);
    sc.off_gu = (int64_t)(l0.wgu - l0.attn_norm);
    sc.off_wd = (int64_t)(l0.wd - l0.attn_norm);
    sc.layers = cfg->layers;
    sc.D = (int)D;
    sc.F = (int)F;
    sc.n_heads = cfg->n_heads;
    sc.n_kv = cfg->n_kv_heads;
    sc.max_ctx = cfg->max_ctx;
    sc.pairing = cfg->pairing;
    sc.vocab = cfg->vocab;
    sc.eps = cfg->eps;
    sc.kc = reinterpret_cast<float*>(m->s + L.kc);
    sc.vc = reinterpret_cast<float*>(m->s + L.vc);
    sc.cache_layer_stride = L.cache_layer_stride;
    sc.cache_batch_stride = L.cache_batch_stride;
    sc.rope = reinterpret_cast<const float*>(m->s + L.rope);
    m->cluster_ok = uniform && step_cluster_plan(sc, &m->plan);
  }
  *out = m;
  return QD_OK;
}

void qd_model_destroy(qd_model* m) {
  if (!m) return;
  for (auto& g : m->graph)
    if (g) cudaGraphExecDestroy(g);
  if (m->capture_stream) cudaStreamDestroy(m->capture_stream);
  delete m;
}

qd_status qd_decode_step(qd_model* m, const int32_t* tokens, int batch, int32_t* out_tokens, float* logits_out,
                         qd_stream_t stream) {
  if (!m || !tokens || !out_tokens) return QD_ERR_INVALID_ARG;
  if (batch < 1 || batch > m->cfg.max_batch) return QD_ERR_SHAPE;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGraphExec_t g;
  QD_TRY(get_graph(m, batch, &g));
  if (cudaMemcpyAsync(m->s + m->L.tok_in, tokens, 4 * (size_t)batch, cudaMemcpyDefault, st) != cudaSuccess)
    return QD_ERR_CUDA;
  if (cudaGraphLaunch(g, st) != cudaSuccess) return QD_ERR_CUDA;
  if (cudaMemcpyAsync(out_tokens, m->s + m->L.tok_out, 4 * (size_t)batch, cudaMemcpyDefault, st) != cudaSuccess)
    return QD_ERR_CUDA;
  if (logits_out &&
      cudaMemcpyAsync(logits_out, m->s + m->L.logits, 4 * (size_t)batch * m->cfg.vocab, cudaMemcpyDefault, st) !=
          cudaSuccess)
    return QD_ERR_CUDA;
  return QD_OK;
}

size_t qd_prefill_workspace(const qd_config* cfg, int t) {
  if (!config_ok(cfg) || cfg->act_q8 || t < 1 || t > QD_MAX_GEMM_TOKENS || t > cfg->max_ctx) return 0;
  const Layout L = make_layout(cfg);
  return prefill_layout(*cfg, L.qkv_rows, t).total;
}

qd_status qd_prefill(qd_model* m, int seq, const int32_t* tokens, int t, unsigned flags, void* workspace,
                     size_t workspace_bytes, int32_t* out_token, float* logits_out, qd_stream_t stream) {
  if (!m || !tokens || !out_token || !workspace) return QD_ERR_INVALID_ARG;
  if (flags & ~QD_PREFILL_EXACT) return QD_ERR_INVALID_ARG;
  if (m->cfg.act_q8) return QD_ERR_UNSUPPORTED;
  if (seq < 0 || seq >= m->cfg.max_batch || t < 1 || t > QD_MAX_GEMM_TOKENS || t > m->cfg.max_ctx)
    return QD_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return QD_ERR_INVALID_ARG;
  const size_t need = prefill_layout(m->cfg, m->L.qkv_rows, t).total;
  if (workspace_bytes < need) return QD_ERR_NOMEM;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (cudaMemcpyAsync(ws + prefill_layout(m->cfg, m->L.qkv_rows, t).tok, tokens, 4 * (size_t)t, cudaMemcpyDefault,
                      st) != cudaSuccess)
    return QD_ERR_CUDA;
  QD_TRY(enqueue_prefill(m, seq, t, flags, ws, st));
  if (cudaMemcpyAsync(out_token, m->s + m->L.tok_out + 4 * (size_t)seq, 4, cudaMemcpyDefault, st) != cudaSuccess)
    return QD_ERR_CUDA;
  if (logits_out && cudaMemcpyAsync(logits_out, m->f(m->L.logits) + (int64_t)seq * m->cfg.vocab,
                                    4 * (size_t)m->cfg.vocab, cudaMemcpyDefault, st) != cudaSuccess)
    return QD_ERR_CUDA;
  return QD_OK;
}

qd_status qd_model_reset(qd_model* m, qd_stream_t stream) {
  if (!m) return QD_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t cache = (size_t)m->cfg.layers * m->L.cache_layer_stride * (m->cfg.kv_f16 ? 2 : 4);
  QD_TRY(zero_region(m->s + m->L.kc, align_up(cache, 16), st));
  QD_TRY(zero_region(m->s + m->L.vc, align_up(cache, 16), st));
  QD_TRY(zero_region(m->s + m->L.pos, 16 * ((4 * m->cfg.max_batch + 15) / 16), st));
  QD_TRY(zero_region(m->s + m->L.err, 16, st));
  QD_TRY(zero_region(m->s + m->L.am_key, align_up(8 * (size_t)m->cfg.max_batch, 16), st));
  QD_TRY(zero_region(m->s + m->L.am_cnt, 16, st));
  return QD_OK;
}

qd_status qd_model_set_pos(qd_model* m, const int32_t* pos_host, int batch, qd_stream_t stream) {
  if (!m || !pos_host) return QD_ERR_INVALID_ARG;
  if (batch < 1 || batch > m->cfg.max_batch) return QD_ERR_SHAPE;
  for (int b = 0; b < batch; ++b)
    if (pos_host[b] < 0 || pos_host[b] >= m->cfg.max_ctx) return QD_ERR_SHAPE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(m->s + m->L.pos, pos_host, 4 * (size_t)batch, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return QD_ERR_CUDA;
  return QD_OK;
}

qd_status qd_model_pos(qd_model* m, int32_t* pos_host, int batch, qd_stream_t stream) {
  if (!m || !pos_host) return QD_ERR_INVALID_ARG;
  if (batch < 1 || batch > m->cfg.max_batch) return QD_ERR_SHAPE;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(pos_host, m->s + m->L.pos, 4 * (size_t)batch, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return QD_ERR_CUDA;
  return QD_OK;
}

qd_status qd_model_kv_cache(qd_model* m, void** k_cache, void** v_cache) {
  if (!m || !k_cache || !v_cache) return QD_ERR_INVALID_ARG;
  *k_cache = m->s + m->L.kc;
  *v_cache = m->s + m->L.vc;
  return QD_OK;
}

qd_status qd_model_act_q8_buffer(qd_model* m, void** buf, size_t* slot_bytes, int* slots) {
  if (!m || !buf || !slot_bytes || !slots) return QD_ERR_INVALID_ARG;
  const bool on = m->cfg.act_q8 != 0;
  *buf = on ? m->s + m->L.xq : nullptr;
  *slot_bytes = on ? m->L.xq_slot : 0;
  *slots = on ? 4 * m->cfg.layers + 1 : 0;
  return QD_OK;
}

qd_status qd_model_check(qd_model* m, qd_stream_t stream) {
  if (!m) return QD_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, m->s + m->L.err, 4, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return QD_ERR_CUDA;
  if (word) {
    QD_TRY(zero_region(m->s + m->L.err, 16, st));
    return QD_ERR_DEVICE_FLAG;
  }
  return QD_OK;
}

int qd_model_launches_per_step(const qd_model* m) { return m ? m->launches : 0; }

qd_status qd_model_set_step_path(qd_model* m, int path) {
  if (!m) return QD_ERR_INVALID_ARG;
  if (path != QD_STEP_AUTO && path != QD_STEP_KERNEL_CHAIN && path != QD_STEP_CLUSTER) return QD_ERR_INVALID_ARG;
  if (path == QD_STEP_CLUSTER && !m->cluster_ok) return QD_ERR_UNSUPPORTED;
  if (path != m->step_path) {
    for (auto& g : m->graph)
      if (g) {
        cudaGraphExecDestroy(g);
        g = nullptr;
      }
    m->step_path = path;
  }
  return QD_OK;
}

int qd_model_step_path(const qd_model* m) {
  if (!m) return -1;
  return m->cluster_ok && m->step_path == QD_STEP_CLUSTER ? QD_STEP_CLUSTER : QD_STEP_KERNEL_CHAIN;
}

int qd_model_cluster_available(const qd_model* m) { return m && m->cluster_ok ? 1 : 0; }

}  // extern "C"
