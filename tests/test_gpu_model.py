"""GPU parity of the whole decode step (qd_decode_step through the C ABI) against the oracle.

Greedy tokens are compared with teacher forcing: the oracle is always fed the token the GPU
chose, so both sides stay on one sequence.  A token may differ only at a near-tie: the
oracle's logit gap between its choice and the GPU's must be <= 1e-3 * max |oracle logit|.
"""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import TOL, assert_close, dev

pytestmark = pytest.mark.gpu


def build_model(qd, cfg, seed, max_ctx, max_batch, host=None, path=None):
    """path: None (the library's choice), or "chain" / "cluster" to force the step path."""
    host = qdsynth.model_tensors(cfg, seed) if host is None else host
    srcs = [None if t is None else dev(t.view(np.uint8) if t.dtype != np.float32 else t) for t in host]
    m = qd.Model(qd.make_config(cfg, max_ctx, max_batch), srcs)
    if path is not None:
        m.set_step_path(qd.STEP_CLUSTER if path == "cluster" else qd.STEP_KERNEL_CHAIN)
        assert m.step_path() == (qd.STEP_CLUSTER if path == "cluster" else qd.STEP_KERNEL_CHAIN)
    torch.cuda.synchronize()
    return m, host


def check_token(ora_logits, ora_tok, gpu_tok, tol=TOL):
    if gpu_tok == ora_tok:
        return 0
    gap = ora_logits[ora_tok] - ora_logits[gpu_tok]
    assert gap <= tol * np.abs(ora_logits).max(), f"token {gpu_tok} vs oracle {ora_tok}, gap {gap}"
    return 1


def run_teacher_forced(qd, cfg, seed, prompt, n_gen, batch=1, max_ctx=None, tol=TOL, path=None):
    """Feed `prompt` (batch x P ids) then n_gen greedy tokens; compare every step's logits
    (within `tol` of max |oracle|; near-tie tokens within the same gap)."""
    P = prompt.shape[1]
    max_ctx = max_ctx or (P + n_gen)
    m, host = build_model(qd, cfg, seed, max_ctx, batch, path=path)
    om = oracle.Model(dict(cfg, max_ctx=max_ctx), host)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    okc = [np.zeros(L * hk * max_ctx * hd, np.float32) for _ in range(batch)]
    ovc = [np.zeros_like(okc[0]) for _ in range(batch)]
    logits = torch.empty(batch, cfg["vocab"], device="cuda")
    out = torch.empty(batch, dtype=torch.int32)
    cur = prompt[:, 0].astype(np.int32)
    worst, near = 0.0, 0
    for step in range(P + n_gen - 1):
        m.decode_step(torch.from_numpy(cur.copy()), batch, out, logits)
        torch.cuda.synchronize()
        g = logits.cpu().numpy()
        gt = out.numpy().copy()
        assert m.check() == 0
        for b in range(batch):
            ol, ot = om.decode_step(okc[b], ovc[b], hk * max_ctx * hd, step, int(cur[b]))
            worst = max(worst, assert_close(g[b], ol, tol=tol, what=f"logits step {step} seq {b}"))
            assert gt[b] == int(np.argmax(g[b]))  # GPU argmax is exact on its own logits
            near += check_token(ol, ot, int(gt[b]), tol)
        cur = prompt[:, step + 1].astype(np.int32) if step + 1 < P else gt.astype(np.int32)
    assert m.pos(batch) == [P + n_gen - 1] * batch
    m.close()
    return worst, near


TINY = dict(layers=2, dim=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64, vocab=300, rope_theta=1e4, eps=1e-5,
            pairing="half", w_fmt="q4_0", emb_fmt="q8_0")


@pytest.mark.parametrize("w_fmt,emb_fmt,pairing,path", [
    ("q4_0", "q8_0", "half", "chain"), ("q8_0", "q8_0", "adjacent", "chain"), ("i8", "i8", "half", None),
    ("q4_k", "q4_0", "half", None), ("q4_0", "q8_0", "half", "cluster"), ("q8_0", "q8_0", "adjacent", "cluster"),
    ("q4_0", "q4_0", "adjacent", "cluster"), ("q8_0", "q8_0", "half", "cluster")])
def test_tiny_model_teacher_forced(qd, w_fmt, emb_fmt, pairing, path):
    """Both step paths (the kernel chain and the cluster kernel) on the same seeded models."""
    cfg = dict(TINY, w_fmt=w_fmt, emb_fmt=emb_fmt, pairing=pairing)
    prompt = qdsynth.tokens(9, "tiny.prompt", 3 * 5, cfg["vocab"]).reshape(3, 5)
    worst, near = run_teacher_forced(qd, cfg, 9, prompt, n_gen=6, batch=3, max_ctx=16, path=path)
    print(f"tiny {w_fmt}/{emb_fmt} {path}: worst rel err {worst:.2e}, near-tie tokens {near}")


@pytest.mark.parametrize("n_heads,n_kv,dim,ffn,max_ctx,batch", [(9, 3, 576, 1536, 40, 1), (8, 8, 512, 1024, 24, 2),
                                                                (16, 2, 256, 768, 70, 3), (6, 1, 320, 640, 33, 1)])
def test_cluster_step_shapes_teacher_forced(qd, n_heads, n_kv, dim, ffn, max_ctx, batch):
    """The cluster kernel over ragged splits: head groupings G = 3, 1, 8, 6, one kv head or
    as many as half the cluster, rows and positions that do not divide by the cluster, a
    context run to its end (max_ctx positions, so the last chunk holds the last slot)."""
    cfg = dict(layers=2, dim=dim, ffn=ffn, n_heads=n_heads, n_kv_heads=n_kv, head_dim=64, vocab=300,
               rope_theta=1e4, eps=1e-5, pairing="half", w_fmt="q4_0", emb_fmt="q8_0")
    P = max_ctx - 4
    prompt = qdsynth.tokens(27, "cl.prompt", batch * P, cfg["vocab"]).reshape(batch, P)
    worst, near = run_teacher_forced(qd, cfg, 27, prompt, n_gen=5, batch=batch, max_ctx=max_ctx, path="cluster")
    print(f"cluster G={n_heads // n_kv} n_kv={n_kv}: worst rel err {worst:.2e}, near-tie tokens {near}")


@pytest.mark.parametrize("mix,emb_fmt,batch", [
    (dict(w_fmt="q4_k", down_fmt="q6_k"), "q6_k", 1),  # Q4_K_M-like: Q4_K, Q6_K down and head
    (dict(qkv_fmt="q8_0", wo_fmt="q5_0", gate_up_fmt="q5_k", down_fmt="q6_k"), "q4_1", 3),
    (dict(w_fmt="q8_0", gate_up_fmt="f16", down_fmt="q4_1"), "q8_0", 2)])
def test_mixed_format_model_teacher_forced(qd, mix, emb_fmt, batch):
    """Models whose matrix classes take different formats (model files mix them by tensor):
    the streaming and tensor-core GEMVs for the formats they take, the register-path GEMV
    with a separate norm, QKV epilogue and argmax for the others, in one step."""
    cfg = dict(TINY, emb_fmt=emb_fmt, **mix)
    prompt = qdsynth.tokens(29, "mix.prompt", batch * 4, cfg["vocab"]).reshape(batch, 4)
    worst, near = run_teacher_forced(qd, cfg, 29, prompt, n_gen=4, batch=batch, max_ctx=12)
    print(f"mixed {mix} emb {emb_fmt} batch {batch}: worst rel err {worst:.2e}, near-tie tokens {near}")


@pytest.mark.parametrize("w_fmt,emb_fmt,batch", [("q4_0", "q8_0", 12), ("q8_0", "q4_0", 9)])
def test_wide_model_batch_over_8_row_passes(qd, w_fmt, emb_fmt, batch):
    """4096-wide activations at batch 9-16: 16 rows of x do not fit beside the weight ring,
    so the tensor-core GEMV runs two passes of up to 8 batch rows, each with its own x, y,
    positions, cache rows and argmax keys (the fused RMSNorm, the QKV epilogue, the
    residual adds and the head's argmax over both passes)."""
    cfg = dict(layers=1, dim=4096, ffn=512, n_heads=64, n_kv_heads=8, head_dim=64, vocab=300, rope_theta=1e4,
               eps=1e-5, pairing="half", w_fmt=w_fmt, emb_fmt=emb_fmt)
    prompt = qdsynth.tokens(30, "rowpass.prompt", batch * 3, cfg["vocab"]).reshape(batch, 3)
    worst, near = run_teacher_forced(qd, cfg, 30, prompt, n_gen=3, batch=batch, max_ctx=8)
    print(f"wide model {w_fmt} batch {batch}: worst rel err {worst:.2e}, near-tie tokens {near}")


@pytest.mark.parametrize("w_fmt,batch", [("q4_0", 6), ("q8_0", 8)])
def test_wide_ffn_model_column_ranges(qd, w_fmt, batch):
    """A 7B-wide FFN (11008) under a narrow model (dim 320, one stage and a partial one):
    at batch 6 and 8 the down projection's x is too wide for one launch, so it runs as
    column ranges that add into the residual, and the fused RMSNorm of the QKV and gate/up
    products spans a partial stage."""
    cfg = dict(layers=1, dim=320, ffn=11008, n_heads=5, n_kv_heads=1, head_dim=64, vocab=300, rope_theta=1e4,
               eps=1e-5, pairing="half", w_fmt=w_fmt, emb_fmt="q8_0")
    prompt = qdsynth.tokens(28, "wide.prompt", batch * 3, cfg["vocab"]).reshape(batch, 3)
    worst, near = run_teacher_forced(qd, cfg, 28, prompt, n_gen=3, batch=batch, max_ctx=8)
    print(f"wide ffn {w_fmt} batch {batch}: worst rel err {worst:.2e}, near-tie tokens {near}")


def test_step_path_choice(qd):
    """The kernel chain by default; the 135M shape can take the cluster path (two launches
    per token: the layers, then the head GEMV with the argmax), and switching back and
    forth gives the same tokens; modes the cluster kernel does not take refuse it."""
    m, _ = build_model(qd, dict(qdsynth.SMOL_135M, layers=2), 0, 256, 1)
    assert m.step_path() == qd.STEP_KERNEL_CHAIN and m.cluster_available()
    toks = {}
    for path in (qd.STEP_CLUSTER, qd.STEP_KERNEL_CHAIN):
        m.reset()
        m.set_step_path(path)
        assert m.step_path() == path
        out = torch.empty(1, dtype=torch.int32)
        seq = []
        cur = torch.tensor([3], dtype=torch.int32)
        for _ in range(4):
            m.decode_step(cur, 1, out)
            torch.cuda.synchronize()
            seq.append(int(out.item()))
            cur = out.clone()
        assert m.check() == 0
        assert m.launches_per_step() == (2 if path == qd.STEP_CLUSTER else 152 - 28 * 5)
        toks[path] = seq
    assert toks[qd.STEP_CLUSTER] == toks[qd.STEP_KERNEL_CHAIN]
    m.close()
    m, _ = build_model(qd, dict(TINY, kv_f16=True), 0, 16, 1)
    assert m.step_path() == qd.STEP_KERNEL_CHAIN and not m.cluster_available()
    with pytest.raises(qd.QDError):
        m.set_step_path(qd.STEP_CLUSTER)
    m.close()


@pytest.mark.parametrize("batch", [12, 16])
def test_tiny_int8_model_batch_over_8_tensor_cores(qd, batch):
    """INT8 rows at batch 9-16 take the tensor-core GEMV (store, accumulate and SwiGLU
    epilogues; separate RMSNorm, RoPE/KV-append and argmax kernels)."""
    cfg = dict(TINY, w_fmt="i8", emb_fmt="i8", pairing="half")
    prompt = qdsynth.tokens(10, "tiny.prompt16", batch * 3, cfg["vocab"]).reshape(batch, 3)
    worst, near = run_teacher_forced(qd, cfg, 10, prompt, n_gen=3, batch=batch, max_ctx=8)
    print(f"tiny i8 batch {batch}: worst rel err {worst:.2e}, near-tie tokens {near}")


def periodic_embedding(fmt, emb, vocab, dim, period):
    """The embedding table with row i replaced by row i % period (model-file layout), so the
    tied head's logits repeat with that period: every value, the largest included, is taken
    by about vocab / period indices."""
    e = emb.copy()
    if fmt == "i8":  # codes [vocab][dim], then f32 scales [vocab]
        codes = e[:vocab * dim].reshape(vocab, dim)
        scales = e[vocab * dim:].view(np.float32)
        for i in range(period, vocab):
            codes[i] = codes[i % period]
            scales[i] = scales[i % period]
        return e
    rows = e.reshape(vocab, -1)
    for i in range(period, vocab):
        rows[i] = rows[i % period]
    return e


@pytest.mark.parametrize("w_fmt,emb_fmt,batch,act_q8", [("q4_0", "q8_0", 1, False), ("q4_0", "q8_0", 3, False),
                                                        ("i8", "i8", 12, False), ("q8_0", "q4_0", 2, True)])
def test_argmax_first_index_on_tied_logits(qd, w_fmt, emb_fmt, batch, act_q8):
    """Exact ties at the largest logit: with embedding rows repeating with period 7, the tied
    head gives bit-identical logits to the rows of each class, so the maximum is shared by
    ~43 indices and the greedy token must be the first of them (go-llm index Argmax: ties
    go to the lowest index; dasLLAMA most_likely's strict '>').  Batch 1 and 3 take the
    head GEMV's fused 64-bit-key argmax; batch 12 (INT8 rows on the tensor cores) and the
    ggml-exact mode take the separate argmax kernel."""
    cfg = dict(TINY, w_fmt=w_fmt, emb_fmt=emb_fmt, act_q8=act_q8)
    host = qdsynth.model_tensors(cfg, 26)
    host[0] = periodic_embedding(emb_fmt, host[0], cfg["vocab"], cfg["dim"], 7)
    max_ctx, steps = 8, 4
    m, _ = build_model(qd, cfg, 26, max_ctx, batch, host=host)
    om = oracle.Model(dict(cfg, max_ctx=max_ctx), host)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    okc = [np.zeros(L * hk * max_ctx * hd, np.float32) for _ in range(batch)]
    ovc = [np.zeros_like(okc[0]) for _ in range(batch)]
    logits = torch.empty(batch, cfg["vocab"], device="cuda")
    out = torch.empty(batch, dtype=torch.int32)
    cur = qdsynth.tokens(26, "tie.prompt", batch, cfg["vocab"]).astype(np.int32)
    for step in range(steps):
        m.decode_step(torch.from_numpy(cur.copy()), batch, out, logits)
        torch.cuda.synchronize()
        assert m.check() == 0
        g = logits.cpu().numpy()
        gt = out.numpy().copy()
        for b in range(batch):
            top = np.flatnonzero(g[b] == g[b].max())
            assert top.size >= 40, top.size  # the maximum really is tied
            assert gt[b] == top[0] < 7, (gt[b], top[:3])
            ol, ot = om.decode_step(okc[b], ovc[b], hk * max_ctx * hd, step, int(cur[b]))
            assert ot < 7 and ol[ot] == ol[ot + 7]  # the oracle's own tie and first index
            assert_close(g[b], ol, what=f"tied logits step {step} seq {b}")
            check_token(ol, ot, int(gt[b]))
        cur = gt.astype(np.int32)
    m.close()


def test_model_reset_and_errors(qd):
    cfg = dict(TINY)
    m, _ = build_model(qd, cfg, 3, 4, 2)
    out = torch.empty(2, dtype=torch.int32)
    for _ in range(4):
        m.decode_step(torch.tensor([1, 2], dtype=torch.int32), 2, out)
    assert m.pos(2) == [4, 4]
    m.decode_step(torch.tensor([1, 2], dtype=torch.int32), 2, out)  # pos == max_ctx: flagged, no write
    assert m.check() == 7
    m.reset()
    assert m.pos(2) == [0, 0]
    m.decode_step(torch.tensor([1, 300], dtype=torch.int32), 2, out)  # token == vocab: flagged
    assert m.check() == 7
    assert m.check() == 0  # the word was cleared
    m.close()


@pytest.mark.slow
@pytest.mark.parametrize("path", ["cluster", "chain"])
def test_smol135m_prompt128_gen128_teacher_forced(qd, path):
    """135M-shaped model: 128 prompt ids ~U[0, 49152), then 128 greedy tokens, batch 1."""
    cfg = qdsynth.SMOL_135M
    prompt = qdsynth.tokens(0, "smol135m.prompt", 128, cfg["vocab"]).reshape(1, 128)
    worst, near = run_teacher_forced(qd, cfg, 0, prompt, n_gen=128, batch=1, max_ctx=256, path=path)
    print(f"135M {path}: worst rel err {worst:.2e}, near-tie tokens {near}/255")


def fill_cache_normal(m, cfg, seed, max_batch, max_ctx):
    """KV cache entries ~N(0,1), generated in (layer, sequence) slices straight into the
    model's cache (layout [layer][batch][kv_head][ctx][hd]); for a binary16 cache
    (cfg["kv_f16"]) the values rounded to binary16 (numpy's round-to-nearest-even cast)."""
    f16 = cfg.get("kv_f16", False)
    esz = 2 if f16 else 4
    kp, vp = m.kv_cache_ptrs()
    base = m.state.data_ptr()
    n = cfg["layers"] * max_batch * cfg["n_kv_heads"] * max_ctx * cfg["head_dim"]
    k = m.state[kp - base:kp - base + esz * n].view(torch.int16 if f16 else torch.float32)
    v = m.state[vp - base:vp - base + esz * n].view(torch.int16 if f16 else torch.float32)
    per = cfg["n_kv_heads"] * max_ctx * cfg["head_dim"]
    buf = np.empty(per, np.float32)
    host = torch.empty(per, dtype=torch.int16 if f16 else torch.float32).pin_memory()
    for name, dst in (("c5.kcache", k), ("c5.vcache", v)):
        for s in range(cfg["layers"] * max_batch):
            qdsynth.normal_f32(seed, name, per, offset=s * per, out=buf)
            host.numpy()[:] = buf.astype(np.float16).view(np.int16) if f16 else buf
            dst[s * per:(s + 1) * per].copy_(host, non_blocking=False)
    torch.cuda.synchronize()


def oracle_cache(cfg, seed, b, max_batch, max_ctx):
    per = cfg["n_kv_heads"] * max_ctx * cfg["head_dim"]
    L = cfg["layers"]
    k = np.empty(L * per, np.float32)
    v = np.empty(L * per, np.float32)
    for l in range(L):
        off = (l * max_batch + b) * per
        qdsynth.normal_f32(seed, "c5.kcache", per, offset=off, out=k[l * per:(l + 1) * per])
        qdsynth.normal_f32(seed, "c5.vcache", per, offset=off, out=v[l * per:(l + 1) * per])
    if cfg.get("kv_f16", False):  # the binary16 cache holds these values exactly
        k = k.astype(np.float16).astype(np.float32)
        v = v.astype(np.float16).astype(np.float32)
    return k, v


@pytest.mark.slow
@pytest.mark.parametrize("batch,check_seqs,kv_f16", [(1, [0], False), (16, [0, 9, 15], False), (1, [0], True)])
def test_smol1p7b_int8_ctx4096(qd, batch, check_seqs, kv_f16):
    """1.7B-shaped INT8 model, KV cache (f32, or binary16) holding 4095 N(0,1) positions;
    one step at pos 4095 (attending over 4096 entries), independent sequences."""
    cfg = dict(qdsynth.SMOL_1_7B, kv_f16=kv_f16)
    ctx = 4096
    m, host = build_model(qd, cfg, 0, ctx, batch)
    fill_cache_normal(m, cfg, 0, batch, ctx)
    m.set_pos([ctx - 1] * batch)
    toks = qdsynth.tokens(0, "c5.tokens", 16, cfg["vocab"])[:batch].astype(np.int32)
    logits = torch.empty(batch, cfg["vocab"], device="cuda")
    out = torch.empty(batch, dtype=torch.int32)
    m.decode_step(torch.from_numpy(toks.copy()), batch, out, logits)
    torch.cuda.synchronize()
    assert m.check() == 0
    g = logits.cpu().numpy()
    om = oracle.Model(dict(cfg, max_ctx=ctx), host)
    per = cfg["n_kv_heads"] * ctx * cfg["head_dim"]
    for b in check_seqs:
        kc, vc = oracle_cache(cfg, 0, b, batch, ctx)
        ol, ot = om.decode_step(kc, vc, per, ctx - 1, int(toks[b]))
        err = assert_close(g[b], ol, what=f"1.7B seq {b}")
        check_token(ol, ot, int(out[b]))
        print(f"1.7B batch {batch} seq {b}: rel err {err:.2e}")
    m.close()


def flat_cfg(n_heads, n_kv):
    """A 2-layer model whose f32 cache at batch 4 and context 2048 holds >= 8 MiB over all
    (sequence, kv head) pairs: the decode step takes the flat-split attention kernel."""
    return dict(layers=2, dim=512, ffn=1024, n_heads=n_heads, n_kv_heads=n_kv, head_dim=64, vocab=300,
                rope_theta=1e4, eps=1e-5, pairing="half", w_fmt="q8_0", emb_fmt="q8_0")


FLAT_CTX, FLAT_BATCH = 2048, 4


@pytest.mark.parametrize("n_heads,n_kv,kv_f16", [(8, 8, False), (8, 4, False), (12, 4, False), (16, 2, False),
                                                  (8, 8, True), (16, 2, True)])
def test_flat_attention_ragged_positions(qd, n_heads, n_kv, kv_f16):
    """Four sequences at ragged positions over an N(0,1) cache: one at the last position
    (2048 entries), one at position 0 (a single entry), one mid-context, one just past a
    64-position tile edge; two consecutive steps, every sequence checked against the oracle.
    On the second step the first sequence has run past the context: it is flagged and the
    others are unaffected.  With kv_f16 the cache holds binary16 values."""
    cfg = dict(flat_cfg(n_heads, n_kv), kv_f16=kv_f16)
    m, host = build_model(qd, cfg, 21, FLAT_CTX, FLAT_BATCH)
    fill_cache_normal(m, cfg, 21, FLAT_BATCH, FLAT_CTX)
    start = [FLAT_CTX - 1, 0, 700, 64]
    m.set_pos(start)
    om = oracle.Model(dict(cfg, max_ctx=FLAT_CTX), host)
    per = cfg["n_kv_heads"] * FLAT_CTX * cfg["head_dim"]
    caches = [oracle_cache(cfg, 21, b, FLAT_BATCH, FLAT_CTX) for b in range(FLAT_BATCH)]
    toks = qdsynth.tokens(21, "flat.tokens", 2 * FLAT_BATCH, cfg["vocab"]).astype(np.int32).reshape(2, FLAT_BATCH)
    logits = torch.empty(FLAT_BATCH, cfg["vocab"], device="cuda")
    out = torch.empty(FLAT_BATCH, dtype=torch.int32)
    for step in range(2):
        m.decode_step(torch.from_numpy(toks[step].copy()), FLAT_BATCH, out, logits)
        torch.cuda.synchronize()
        status = m.check()
        assert status == (0 if step == 0 else 7), status  # 7: QD_ERR_DEVICE_FLAG
        g = logits.cpu().numpy()
        for b in range(FLAT_BATCH):
            p = start[b] + step
            if p >= FLAT_CTX:
                continue
            ol, ot = om.decode_step(caches[b][0], caches[b][1], per, p, int(toks[step, b]))
            assert_close(g[b], ol, what=f"flat attention G={n_heads // n_kv} step {step} seq {b} pos {p}")
            check_token(ol, ot, int(out[b]))
    m.close()


def test_flat_attention_teacher_forced_from_empty_cache(qd):
    """The flat split from position 0 on (a handful of tiles over 152 CTAs: most CTAs idle,
    several CTAs per pair only later), batch 2 at context 2048 with 8 kv heads."""
    cfg = flat_cfg(8, 8)
    prompt = qdsynth.tokens(22, "flat.prompt", 2 * 6, cfg["vocab"]).reshape(2, 6)
    worst, near = run_teacher_forced(qd, cfg, 22, prompt, n_gen=4, batch=2, max_ctx=FLAT_CTX)
    print(f"flat split from an empty cache: worst rel err {worst:.2e}, near-tie tokens {near}")


@pytest.mark.parametrize("kv_f16", [False, True])
def test_flat_attention_many_short_pairs(qd, kv_f16):
    """96 kv heads x 16 sequences at positions < 64: 1536 one-tile pairs over 152 CTAs, so
    a CTA's run covers more pairs than it holds before settling them mid-run.  With the
    binary16 cache a tile spans 128 positions: the warps past position 63 see no live row."""
    cfg = dict(layers=1, dim=256, ffn=512, n_heads=96, n_kv_heads=96, head_dim=64, vocab=300, rope_theta=1e4,
               eps=1e-5, pairing="adjacent", w_fmt="q8_0", emb_fmt="q8_0", kv_f16=kv_f16)
    ctx, batch = 64, 16
    m, host = build_model(qd, cfg, 23, ctx, batch)
    fill_cache_normal(m, cfg, 23, batch, ctx)
    start = [int(v) for v in qdsynth.tokens(23, "flat.short.pos", batch, ctx)]
    m.set_pos(start)
    toks = qdsynth.tokens(23, "flat.short.tokens", batch, cfg["vocab"]).astype(np.int32)
    logits = torch.empty(batch, cfg["vocab"], device="cuda")
    out = torch.empty(batch, dtype=torch.int32)
    m.decode_step(torch.from_numpy(toks.copy()), batch, out, logits)
    torch.cuda.synchronize()
    assert m.check() == 0
    g = logits.cpu().numpy()
    om = oracle.Model(dict(cfg, max_ctx=ctx), host)
    per = cfg["n_kv_heads"] * ctx * cfg["head_dim"]
    for b in range(batch):
        kc, vc = oracle_cache(cfg, 23, b, batch, ctx)
        ol, ot = om.decode_step(kc, vc, per, start[b], int(toks[b]))
        assert_close(g[b], ol, what=f"short pairs seq {b} pos {start[b]}")
        check_token(ol, ot, int(out[b]))
    m.close()


@pytest.mark.parametrize("w_fmt,emb_fmt,pairing,batch", [("q4_0", "q8_0", "half", 1), ("i8", "i8", "adjacent", 3)])
def test_kv_f16_teacher_forced(qd, w_fmt, emb_fmt, pairing, batch):
    """Binary16 KV cache (go-llm's ggml-exact cache): k and v rounded through binary16 when
    appended, on both sides; the decode step takes the flat-split attention over it."""
    cfg = dict(TINY, w_fmt=w_fmt, emb_fmt=emb_fmt, pairing=pairing, kv_f16=True)
    prompt = qdsynth.tokens(24, "f16.prompt", batch * 5, cfg["vocab"]).reshape(batch, 5)
    worst, near = run_teacher_forced(qd, cfg, 24, prompt, n_gen=5, batch=batch, max_ctx=72)
    print(f"kv_f16 {w_fmt}: worst rel err {worst:.2e}, near-tie tokens {near}")


def _round_f16_vec(a):
    return np.array([oracle.round_f16(float(v)) for v in np.asarray(a, np.float32).reshape(-1)],
                    np.float32).reshape(np.shape(a))


def _cache_rows_at(m, cfg, max_batch, max_ctx, pos_list):
    """The GPU cache's k and v rows at each sequence's position, every layer, as f32:
    [batch][layers][2][n_kv * head_dim]."""
    f16 = cfg.get("kv_f16", False)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    esz = 2 if f16 else 4
    n = L * max_batch * hk * max_ctx * hd
    base = m.state.data_ptr()
    out = np.empty((len(pos_list), L, 2, hk * hd), np.float32)
    for j, ptr in enumerate(m.kv_cache_ptrs()):
        t = m.state[ptr - base:ptr - base + esz * n].view(torch.float16 if f16 else torch.float32)
        a = t.float().cpu().numpy().reshape(L, max_batch, hk, max_ctx, hd)
        for b, p in enumerate(pos_list):
            out[b, :, j] = a[:, b, :, p, :].reshape(L, hk * hd)
    return out


def _q8_inputs(m, cfg, batch):
    """Every quantised input of the GPU's last ggml-exact step (qd_model_act_q8_buffer), per
    sequence as the oracle's teacher-forcing slots take them: codes int8 [batch][slots][cols]
    and binary16 block scales as f32 [batch][slots][cols/32] (zero past each input's
    length), and the length of each slot's input."""
    ptr, slot_bytes, slots = m.act_q8_buffer()
    D, F, QD = cfg["dim"], cfg["ffn"], cfg["n_heads"] * cfg["head_dim"]
    width = [D, QD, D, F] * cfg["layers"] + [D]
    assert slots == len(width)
    cols = max(D, F, QD)
    base = m.state.data_ptr()
    raw = m.state[ptr - base:ptr - base + slot_bytes * slots].cpu().numpy().reshape(slots, slot_bytes)
    codes = np.zeros((batch, slots, cols), np.int8)
    d = np.zeros((batch, slots, cols // 32), np.float32)
    for k, n in enumerate(width):
        codes[:, k, :n] = raw[k, :batch * n].view(np.int8).reshape(batch, n)
        off = (batch * n + 15) // 16 * 16
        d[:, k, :n // 32] = raw[k, off:off + 2 * batch * (n // 32)].view(np.float16).astype(np.float32).reshape(
            batch, n // 32)
    return codes, d, width


# Teacher forcing at every quantised input leaves the GPU and the oracle apart only by the
# GPU's f32 arithmetic (summation order, its exp2-based softmax): EPS_F32 of a vector's
# magnitude bounds that with a wide margin (measured ~1e-7).  A code, a block scale or a
# binary16 cache value may differ from the oracle's own only where the oracle's value
# lies within that distance of a rounding boundary.
EPS_F32 = 1e-5


def check_cache_values(gpu, ora_f32, kv_f16):
    """The k, v values the GPU step appended against those the teacher-forced oracle formed
    (before any binary16 rounding): with the binary16 cache binary16 values (the rounding
    happened), each a correct rounding of a value within EPS_F32 of the oracle's (relative
    to the vector's largest |value|); with the f32 cache, that value itself.  Returns the
    number of values that differ from the oracle's own."""
    M = np.abs(ora_f32).max(axis=-1, keepdims=True)
    if not kv_f16:
        assert (np.abs(gpu - ora_f32) <= EPS_F32 * M).all(), "appended f32 value off the oracle's"
        return int((gpu != ora_f32).sum())
    assert np.array_equal(gpu, gpu.astype(np.float16).astype(np.float32)), "cache value not binary16"
    lo = _round_f16_vec((ora_f32 - EPS_F32 * M).astype(np.float32))
    hi = _round_f16_vec((ora_f32 + EPS_F32 * M).astype(np.float32))
    bad = ~((gpu >= lo) & (gpu <= hi))
    if bad.any():
        i = np.unravel_index(np.argmax(bad), bad.shape)
        raise AssertionError(f"binary16 cache value at {i}: gpu {gpu[i]!r}, oracle {ora_f32[i]!r} rounds to "
                             f"[{lo[i]!r}, {hi[i]!r}] ({int(bad.sum())} of {bad.size})")
    return int((gpu != _round_f16_vec(ora_f32)).sum())


def check_q8_input(codes, d, x_ora, what):
    """The GPU's Q8_0 quantisation (codes, binary16 d) of one product's input against the
    input x_ora the teacher-forced oracle formed: each block scale a binary16 rounding of
    (block max)/127 for a block max within EPS_F32 * M of the oracle's (M: the vector's
    largest |value|), each code within half a step of x / d, widened by that same
    distance.  Returns (codes, scales) differing from the oracle's own quantisation."""
    x = x_ora.astype(np.float64).reshape(-1, 32)
    M = float(np.abs(x).max())
    e = EPS_F32 * M
    m = np.abs(x).max(axis=1)
    dd = d.reshape(-1)
    assert np.abs(codes).max() <= 127
    dlo = _round_f16_vec(((m - e) / 127).astype(np.float32))
    dhi = _round_f16_vec(((m + e) / 127).astype(np.float32))
    badd = ~((dd >= dlo) & (dd <= dhi))
    if badd.any():
        j = int(np.argmax(badd))
        raise AssertionError(f"{what}: block scale {j} gpu {dd[j]!r}, oracle block max {m[j]!r}")
    live = m > 0
    df = np.where(live, m / 127, 1.0)[:, None]
    slack = 0.5 + e / df + 127 * e / np.where(live, m, 1.0)[:, None]
    over = (np.abs(codes.reshape(-1, 32) - x / df) > slack) & live[:, None]
    if over.any():
        i = np.unravel_index(np.argmax(over), over.shape)
        raise AssertionError(f"{what}: code at block {i[0]} element {i[1]}: gpu {codes.reshape(-1, 32)[i]}, "
                             f"oracle quotient {x[i] / df[i[0], 0]!r}")
    qo, do, _ = oracle.quantize_q8(x_ora[None, :])
    return int((qo.reshape(-1) != codes.reshape(-1)).sum()), int((do.reshape(-1) != dd).sum())


@pytest.mark.parametrize("w_fmt,emb_fmt,batch,kv_f16", [("q4_0", "q8_0", 1, True), ("q8_0", "q8_0", 3, True),
                                                        ("q4_0", "q8_0", 2, False)])
def test_ggml_exact_teacher_forced(qd, w_fmt, emb_fmt, batch, kv_f16):
    """go-llm's ggml-exact mode: every quantised product over Q8_0 activations in integers
    (act_q8), with and without the binary16 cache, against the oracle in the same mode,
    teacher-forced at every rounding the mode makes.  The two sides form their f32
    activations in different orders, so a value near a rounding boundary may take a Q8 code
    (or a binary16 cache value) one step away; one such step moves everything after it (a
    Q8_0 weight multiplies it by up to 127 d_w), so comparing free-running steps could only
    bound the drift.  Instead, after each GPU step the oracle is run from the GPU's own
    roundings: the binary16 (or f32) k, v the GPU appended, and the Q8 codes and scales of
    each of its quantised inputs (4 per layer and the head's).  Then every GPU rounding must
    be a correct rounding of the value the oracle formed, up to f32 arithmetic (EPS_F32),
    and the logits within 1e-3 of the oracle's."""
    cfg = dict(TINY, w_fmt=w_fmt, emb_fmt=emb_fmt, act_q8=True, kv_f16=kv_f16)
    max_ctx, n_gen, P = 72, 5, 5
    prompt = qdsynth.tokens(25, "q8.prompt", batch * P, cfg["vocab"]).reshape(batch, P)
    m, host = build_model(qd, cfg, 25, max_ctx, batch)
    om = oracle.Model(dict(cfg, max_ctx=max_ctx), host)
    L, hk, hd, V = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"], cfg["vocab"]
    per = hk * max_ctx * hd
    okc = [np.zeros(L * per, np.float32) for _ in range(batch)]
    ovc = [np.zeros_like(okc[0]) for _ in range(batch)]
    logits = torch.empty(batch, V, device="cuda")
    out = torch.empty(batch, dtype=torch.int32)
    cur = prompt[:, 0].astype(np.int32)
    worst = 0.0
    flips_cache = flips_code = flips_d = 0
    for step in range(P + n_gen - 1):
        m.decode_step(torch.from_numpy(cur.copy()), batch, out, logits)
        torch.cuda.synchronize()
        assert m.check() == 0
        g = logits.cpu().numpy()
        gt = out.numpy().copy()
        rows = _cache_rows_at(m, cfg, batch, max_ctx, [step] * batch)
        codes, dsc, width = _q8_inputs(m, cfg, batch)
        for b in range(batch):
            kc4 = okc[b].reshape(L, hk, max_ctx, hd)
            vc4 = ovc[b].reshape(L, hk, max_ctx, hd)
            kc4[:, :, step, :] = rows[b, :, 0].reshape(L, hk, hd)
            vc4[:, :, step, :] = rows[b, :, 1].reshape(L, hk, hd)
            ol, ot, kv, hx, xo = om.decode_step_tf(okc[b], ovc[b], per, step, int(cur[b]), kv_given=True,
                                                   q8_codes=codes[b], q8_d=dsc[b])
            flips_cache += check_cache_values(rows[b], kv, kv_f16)
            for k, n in enumerate(width):
                nc, nd = check_q8_input(codes[b, k, :n], dsc[b, k, :n // 32], xo[k, :n],
                                        f"step {step} seq {b} quantised input {k}")
                flips_code += nc
                flips_d += nd
            worst = max(worst, assert_close(g[b], ol, what=f"logits step {step} seq {b}"))
            assert gt[b] == int(np.argmax(g[b]))
            check_token(ol, ot, int(gt[b]))
        cur = prompt[:, step + 1].astype(np.int32) if step + 1 < P else gt.astype(np.int32)
    assert m.pos(batch) == [P + n_gen - 1] * batch
    m.close()
    print(f"ggml-exact {w_fmt} kv_f16={kv_f16}: worst rel err {worst:.2e}; roundings one step from the oracle's "
          f"own: cache values {flips_cache}, Q8 codes {flips_code}, Q8 scales {flips_d}")
