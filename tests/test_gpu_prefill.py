"""GPU parity of the batched prefill (qd_prefill through the C ABI) against the oracle.

The oracle runs the prompt as one decode step per token (the plain definition); qd_prefill
runs it as one t-row matrix per product.  Compared: the last token's logits (within 1e-3 of
max |oracle logit|), its greedy token (up to a near-tie, as in the decode-step tests), every
k and v row the prompt appended (within 1e-3 of each row's largest value), and the
position.  Both product paths are covered: the tensor-core GEMM (binary16 weights; flags 0,
t > 16) and the batched GEMV (QD_PREFILL_EXACT, or t <= 16, or a format the GEMM does not
take).
"""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import TOL, assert_close
from test_gpu_model import TINY, build_model, check_token

pytestmark = pytest.mark.gpu


def _gpu_cache(m, cfg, max_batch, max_ctx):
    """The GPU's k and v caches as f32 [layers][max_batch][n_kv][max_ctx][head_dim]."""
    f16 = cfg.get("kv_f16", False)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    esz = 2 if f16 else 4
    n = L * max_batch * hk * max_ctx * hd
    base = m.state.data_ptr()
    out = []
    for ptr in m.kv_cache_ptrs():
        t = m.state[ptr - base:ptr - base + esz * n].view(torch.float16 if f16 else torch.float32)
        out.append(t.float().cpu().numpy().reshape(L, max_batch, hk, max_ctx, hd))
    return out


def _oracle_prompt(om, cfg, max_ctx, tokens, kc=None, vc=None, p0=0):
    """The oracle over `tokens` at positions p0.. (one decode step each, the prompt fed in);
    returns the last step's (logits, token) and the caches."""
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    if kc is None:
        kc = np.zeros(L * hk * max_ctx * hd, np.float32)
        vc = np.zeros_like(kc)
    ol = ot = None
    for i, tok in enumerate(tokens):
        ol, ot = om.decode_step(kc, vc, hk * max_ctx * hd, p0 + i, int(tok))
    return ol, ot, kc, vc


def _check_cache(gpu, ora, cfg, max_ctx, seq, p0, p1, what):
    """Rows p0..p1-1 of sequence seq, every layer and kv head, k and v, within 1e-3 of each
    row's largest value.  With the binary16 cache both sides store a binary16 rounding of
    values that agree to that bound, and two such roundings may sit one binary16 step
    apart: at most 2^-10 of the value (2^-24 below the normal range) more is allowed."""
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    worst = 0.0
    for j, name in enumerate("kv"):
        o = ora[j].reshape(L, hk, max_ctx, hd)[:, :, p0:p1, :].reshape(-1, hd)
        g = gpu[j][:, seq, :, p0:p1, :].reshape(-1, hd)
        if not cfg.get("kv_f16", False):
            worst = max(worst, assert_close(g, o, what=f"{what} cache {name}"))
            continue
        assert np.array_equal(g, g.astype(np.float16).astype(np.float32)), "cache value not binary16"
        M = np.abs(o).max(axis=1, keepdims=True)
        bound = TOL * M + np.maximum(np.abs(o) * 2.0 ** -10, 2.0 ** -24)
        assert (np.abs(g - o) <= bound).all(), f"{what} cache {name}: beyond 1e-3 plus one binary16 step"
        worst = max(worst, float((np.abs(g - o) / M).max()))
    return worst


def _uses_gemm(cfg, t, flags):
    """The qd_prefill rule for the tensor-core GEMM."""
    qd_ = cfg["n_heads"] * cfg["head_dim"]
    return (flags == 0 and t > 16 and cfg["w_fmt"] in ("q4_0", "q8_0", "i8")
            and cfg["dim"] % 64 == 0 and qd_ % 64 == 0 and cfg["ffn"] % 64 == 0)


def _binary16_layer_weights(cfg, host):
    """The model's tensors with every layer matrix replaced by the binary16 rounding of its
    dequantised values (format f16): what the GEMM multiplies for Q4_0 / Q8_0 weights
    (d * q rounded to nearest binary16).  INT8 codes enter the GEMM exactly: unchanged."""
    if cfg["w_fmt"] == "i8":
        return cfg, host
    shapes = dict((n, (r, c)) for n, r, c in qdsynth.layer_shapes(cfg))
    out = list(host[:3])
    names = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")
    for l in range(cfg["layers"]):
        for j, name in enumerate(names):
            t = host[3 + 9 * l + j]
            if not name.endswith("norm"):
                r, c = shapes[name]
                t = oracle.dequant(cfg["w_fmt"], t, r, c).astype(np.float16).view(np.uint8).reshape(-1)
            out.append(t)
    return dict(cfg, w_fmt="f16"), out


def _prefill(qd, m, seq, tokens, flags, vocab):
    t = len(tokens)
    out = torch.empty(1, dtype=torch.int32)
    logits = torch.empty(vocab, device="cuda")
    m.prefill(seq, torch.from_numpy(np.asarray(tokens, np.int32).copy()), t, out, logits, flags=flags)
    torch.cuda.synchronize()
    assert m.check() == 0
    return int(out.item()), logits.cpu().numpy()


CASES = [
    # w_fmt, emb_fmt, kv_f16, flags, t, seq, max_batch
    ("q4_0", "q8_0", False, 0, 40, 0, 1),      # tensor-core GEMM
    ("q8_0", "q8_0", False, 1, 40, 2, 4),      # QD_PREFILL_EXACT, a later sequence
    ("i8", "i8", False, 0, 33, 1, 2),          # GEMM over INT8 rows, ragged token tile
    ("q4_0", "q8_0", True, 0, 37, 0, 1),       # binary16 cache (attention in chunks of 16)
    ("q4_k", "q4_0", False, 0, 20, 0, 1),      # a format the GEMM does not take: batched GEMV
    ("q4_0", "q8_0", False, 0, 5, 0, 1),       # t <= 16: batched GEMV
    ("mixed", "q6_k", False, 1, 24, 0, 1),     # a mixed-format model (Q4_K with Q6_K down), exact
]


def _check_prompt(m, cfg, host, max_ctx, max_batch, seq, prompt, flags, tok, logits, layers=None):
    """Last-position logits and token against the oracle's decode steps over the prompt (the
    model's own weights), and the appended cache rows (of `layers`, default all) against
    the same definition over the weights the products multiply: the model's own (batched
    GEMV, INT8 GEMM), or their binary16 roundings (Q4_0 / Q8_0 GEMM)."""
    t = len(prompt)
    om = oracle.Model(dict(cfg, max_ctx=max_ctx), host)
    ol, ot, kc, vc = _oracle_prompt(om, cfg, max_ctx, prompt)
    err = assert_close(logits, ol, what="prefill logits")
    assert tok == int(np.argmax(logits))
    check_token(ol, ot, tok)
    rcfg, rhost = _binary16_layer_weights(cfg, host) if _uses_gemm(cfg, t, flags) else (cfg, host)
    if rhost is not host:
        orf = oracle.Model(dict(rcfg, max_ctx=max_ctx), rhost)
        ol16, _, kc, vc = _oracle_prompt(orf, rcfg, max_ctx, prompt)
        assert_close(logits, ol16, what="prefill logits against binary16 layer weights")
    gpu = _gpu_cache(m, cfg, max_batch, max_ctx)
    L, hk, hd = cfg["layers"], cfg["n_kv_heads"], cfg["head_dim"]
    if layers is not None:
        keep = np.array(layers)
        gpu = [g[keep] for g in gpu]
        kc = kc.reshape(L, -1)[keep].reshape(-1)
        vc = vc.reshape(L, -1)[keep].reshape(-1)
        cfg = dict(cfg, layers=len(layers))
    cerr = _check_cache(gpu, (kc, vc), cfg, max_ctx, seq, 0, t, "prefill")
    return err, cerr


@pytest.mark.parametrize("w_fmt,emb_fmt,kv_f16,flags,t,seq,max_batch", CASES)
def test_prefill_matches_decode_steps(qd, w_fmt, emb_fmt, kv_f16, flags, t, seq, max_batch):
    mix = dict(w_fmt="q4_k", down_fmt="q6_k") if w_fmt == "mixed" else dict(w_fmt=w_fmt)
    cfg = dict(TINY, emb_fmt=emb_fmt, kv_f16=kv_f16, **mix)
    max_ctx = t + 8
    m, host = build_model(qd, cfg, 31, max_ctx, max_batch)
    prompt = qdsynth.tokens(31, f"pf.{w_fmt}.{t}", t, cfg["vocab"])
    tok, logits = _prefill(qd, m, seq, prompt, flags, cfg["vocab"])
    err, cerr = _check_prompt(m, cfg, host, max_ctx, max_batch, seq, prompt, flags, tok, logits)
    pos = m.pos(max_batch)
    assert pos[seq] == t and all(p == 0 for i, p in enumerate(pos) if i != seq)
    print(f"prefill {w_fmt} kv_f16={kv_f16} flags={flags} t={t}: logits {err:.2e}, cache {cerr:.2e}")
    m.close()


@pytest.mark.parametrize("flags", [0, 1])
def test_prefill_in_two_calls_then_decode(qd, flags):
    """A prompt prefilled in two calls (the second starts at position 24, so its causal
    attention also reads the first call's rows), then three greedy decode steps on the
    same cache; the oracle is teacher-forced with the GPU's tokens."""
    cfg = dict(TINY)
    max_ctx, t1, t2 = 64, 24, 19
    m, host = build_model(qd, cfg, 32, max_ctx, 1)
    om = oracle.Model(dict(cfg, max_ctx=max_ctx), host)
    prompt = qdsynth.tokens(32, "pf2.prompt", t1 + t2, cfg["vocab"])
    _prefill(qd, m, 0, prompt[:t1], flags, cfg["vocab"])
    tok, logits = _prefill(qd, m, 0, prompt[t1:], flags, cfg["vocab"])
    ol, ot, kc, vc = _oracle_prompt(om, cfg, max_ctx, prompt)
    assert_close(logits, ol, what="second prefill logits")
    check_token(ol, ot, tok)
    _check_cache(_gpu_cache(m, cfg, 1, max_ctx), (kc, vc), cfg, max_ctx, 0, 0, t1 + t2, "two prefills")
    out = torch.empty(1, dtype=torch.int32)
    g = torch.empty(1, cfg["vocab"], device="cuda")
    cur = tok
    for step in range(3):
        p = t1 + t2 + step
        m.decode_step(torch.tensor([cur], dtype=torch.int32), 1, out, g)
        torch.cuda.synchronize()
        ol, ot = om.decode_step(kc, vc, cfg["n_kv_heads"] * max_ctx * cfg["head_dim"], p, cur)
        assert_close(g.cpu().numpy()[0], ol, what=f"decode after prefill, step {step}")
        check_token(ol, ot, int(out.item()))
        cur = int(out.item())
    assert m.pos(1) == [t1 + t2 + 3]
    m.close()


@pytest.mark.parametrize("flags", [0, 1])
def test_prefill_smol135m_prompt128(qd, flags):
    """The 135M-shaped model's 128 prompt ids ~U[0, 49152) in one call: last-position
    logits and token against 128 oracle decode steps, and the appended rows of the first,
    a middle and the last layer (against the same steps over the binary16-rounded layer
    weights on the GEMM path: the rounding moves mid-network rows by ~1.4e-3 of their
    largest value over 15 layers, while the logits stay within 1e-3)."""
    cfg = qdsynth.SMOL_135M
    t, max_ctx = 128, 256
    m, host = build_model(qd, cfg, 0, max_ctx, 1)
    prompt = qdsynth.tokens(0, "smol135m.prompt", t, cfg["vocab"])
    tok, logits = _prefill(qd, m, 0, prompt, flags, cfg["vocab"])
    L = cfg["layers"]
    err, cerr = _check_prompt(m, cfg, host, max_ctx, 1, 0, prompt, flags, tok, logits, layers=[0, L // 2, L - 1])
    assert m.pos(1) == [t]
    print(f"135M prefill flags={flags}: logits {err:.2e}")
    m.close()


def test_prefill_refusals(qd):
    cfg = dict(TINY)
    m, _ = build_model(qd, cfg, 33, 16, 2)
    out = torch.empty(1, dtype=torch.int32)
    toks = torch.zeros(20, dtype=torch.int32)
    assert m.prefill_workspace(17) == 0  # t > max_ctx
    with pytest.raises(qd.QDError) as e:
        m.prefill(0, toks, 17, out)
    assert e.value.status == 2  # QD_ERR_SHAPE
    with pytest.raises(qd.QDError) as e:
        m.prefill(2, toks, 4, out)  # seq >= max_batch
    assert e.value.status == 2
    with pytest.raises(qd.QDError) as e:
        m.prefill(0, toks, 4, out, flags=2)
    assert e.value.status == 1  # QD_ERR_INVALID_ARG
    small = torch.empty(m.prefill_workspace(4) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(qd.QDError) as e:
        m.prefill(0, toks, 4, out, workspace=small)
    assert e.value.status == 6  # QD_ERR_NOMEM
    assert m.pos(2) == [0, 0]
    m.close()
    q8, _ = build_model(qd, dict(TINY, act_q8=True), 33, 16, 1)
    assert q8.prefill_workspace(4) == 0
    with pytest.raises(qd.QDError) as e:
        q8.prefill(0, toks, 4, out, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4  # QD_ERR_UNSUPPORTED
    q8.close()
