"""The oracle's decode step against a composition of its separately pinned operations.

The composition follows the block order of the llmoxide page (s7, "The block, and the
residual stream") and the dasLLAMA forward (8.7.1.6): pre-norm attention with RoPE and an
appended f32 KV cache, residual add, pre-norm SwiGLU feed-forward, residual add, final norm,
tied classifier, greedy argmax.  Activations are rounded to f32 between the composed calls,
so agreement is to ~1e-6; a wiring mistake (a dropped residual, swapped projections, a wrong
norm gain, a wrong cache slot) moves results by O(1).
"""
import numpy as np
import pytest

import oracle
import qdsynth

TINY = dict(layers=2, dim=64, ffn=96, n_heads=4, n_kv_heads=2, head_dim=16, vocab=100, max_ctx=8,
            rope_theta=1e4, eps=1e-5, pairing="half", w_fmt="q4_0", emb_fmt="q8_0")


def _composed_step(cfg, T, kc, vc, pos, tok):
    D, F, hd = cfg["dim"], cfg["ffn"], cfg["head_dim"]
    hq, hk, ctx = cfg["n_heads"], cfg["n_kv_heads"], cfg["max_ctx"]
    ef = cfg["emb_fmt"]
    # a mixed model names the format of each class of matrix; the others take w_fmt
    fq, fo = cfg.get("qkv_fmt", cfg["w_fmt"]), cfg.get("wo_fmt", cfg["w_fmt"])
    fg, fd = cfg.get("gate_up_fmt", cfg["w_fmt"]), cfg.get("down_fmt", cfg["w_fmt"])
    f32 = lambda a: np.asarray(a, dtype=np.float32)
    x = oracle.dequant(ef, T[0], cfg["vocab"], D, row0=tok, nrows=1)[0].astype(np.float64)
    for l in range(cfg["layers"]):
        an, wq, wk, wv, wo, fn, wg, wu, wd = T[3 + 9 * l:12 + 9 * l]
        xn = f32(oracle.rmsnorm(f32(x), an, cfg["eps"]))
        q = oracle.gemv(fq, wq, hq * hd, D, xn)[0]
        k = oracle.gemv(fq, wk, hk * hd, D, xn)[0]
        v = oracle.gemv(fq, wv, hk * hd, D, xn)[0]
        q = oracle.rope(f32(q), hq, hd, pos, cfg["pairing"], cfg["rope_theta"])
        k = oracle.rope(f32(k), hk, hd, pos, cfg["pairing"], cfg["rope_theta"])
        kc[l][:, pos, :] = f32(k).reshape(hk, hd)
        vc[l][:, pos, :] = f32(v).reshape(hk, hd)
        att = oracle.attention(f32(q), kc[l], vc[l], hq, hk, hd, pos + 1, ctx)
        x = x + oracle.gemv(fo, wo, D, hq * hd, f32(att))[0]
        xn = f32(oracle.rmsnorm(f32(x), fn, cfg["eps"]))
        g = oracle.gemv(fg, wg, F, D, xn)[0]
        u = oracle.gemv(fg, wu, F, D, xn)[0]
        a = oracle.swiglu(f32(g), f32(u))
        x = x + oracle.gemv(fd, wd, D, F, f32(a))[0]
    xn = f32(oracle.rmsnorm(f32(x), T[1], cfg["eps"]))
    logits = oracle.gemv(ef, T[0], cfg["vocab"], D, xn)[0]
    return logits


# mixed-format models (a Q4_K_M-like mix, and one with a different format in every class,
# so a matrix read in another class's format fails by O(1))
MIXED_A = dict(down_fmt="q6_k")  # with w_fmt q4_k
MIXED_B = dict(qkv_fmt="q8_0", wo_fmt="q5_0", gate_up_fmt="q5_k", down_fmt="q6_k")


@pytest.mark.parametrize("pairing,w_fmt,emb_fmt,mix", [("half", "q4_0", "q8_0", {}), ("adjacent", "q8_0", "q8_0", {}),
                                                       ("half", "i8", "i8", {}), ("half", "q4_k", "q8_0", {}),
                                                       ("half", "q4_k", "q6_k", MIXED_A),
                                                       ("adjacent", "q4_0", "q4_1", MIXED_B)])
def test_decode_step_equals_composition(pairing, w_fmt, emb_fmt, mix):
    cfg = dict(TINY, pairing=pairing, w_fmt=w_fmt, emb_fmt=emb_fmt, **mix)
    if "q4_k" in (w_fmt,) or mix:
        cfg.update(dim=256, ffn=512, n_heads=4, n_kv_heads=1, head_dim=64)
    T = qdsynth.model_tensors(cfg, seed=11)
    m = oracle.Model(cfg, T)
    L, hk, ctx, hd = cfg["layers"], cfg["n_kv_heads"], cfg["max_ctx"], cfg["head_dim"]
    kc = np.zeros((L, hk, ctx, hd), np.float32)
    vc = np.zeros_like(kc)
    kc2 = [np.zeros((hk, ctx, hd), np.float32) for _ in range(L)]
    vc2 = [np.zeros((hk, ctx, hd), np.float32) for _ in range(L)]
    toks = qdsynth.tokens(11, "prompt", 5, cfg["vocab"])
    for pos, tok in enumerate(toks):
        logits, nxt = m.decode_step(kc, vc, hk * ctx * hd, pos, int(tok))
        ref = _composed_step(cfg, T, kc2, vc2, pos, int(tok))
        scale = np.abs(ref).max()
        assert np.abs(logits - ref).max() <= 1e-5 * scale, (pos, np.abs(logits - ref).max(), scale)
        assert nxt == int(np.argmax(logits))
        for l in range(L):
            kmag = np.abs(kc2[l][:, pos]).max()
            assert np.abs(kc[l, :, pos] - kc2[l][:, pos]).max() <= 1e-5 * kmag
    # cache slots beyond the last position stay untouched
    assert np.all(kc[:, :, len(toks):] == 0) and np.all(vc[:, :, len(toks):] == 0)


def test_decode_step_position0_attends_only_to_itself():
    """At pos 0 the attention output of each head is its kv head's own v, so a cache filled
    with garbage beyond pos 0 must not change the result."""
    cfg = dict(TINY)
    T = qdsynth.model_tensors(cfg, seed=12)
    m = oracle.Model(cfg, T)
    L, hk, ctx, hd = cfg["layers"], cfg["n_kv_heads"], cfg["max_ctx"], cfg["head_dim"]
    kc = np.zeros((L, hk, ctx, hd), np.float32)
    vc = np.zeros_like(kc)
    la, _ = m.decode_step(kc, vc, hk * ctx * hd, 0, 7)
    kc2 = qdsynth.normal_f32(1, "junk", kc.size).reshape(kc.shape)
    vc2 = qdsynth.normal_f32(2, "junk", vc.size).reshape(vc.shape)
    lb, _ = m.decode_step(kc2, vc2, hk * ctx * hd, 0, 7)
    assert np.array_equal(la, lb)
    # ...while at pos 1 (another token, so v differs between positions) the keys at pos 0 matter
    kc2[:, :, 0] = qdsynth.normal_f32(3, "junk", L * hk * hd).reshape(L, hk, hd)
    lc, _ = m.decode_step(kc2, vc2, hk * ctx * hd, 1, 8)
    ld, _ = m.decode_step(kc, vc, hk * ctx * hd, 1, 8)
    assert not np.allclose(lc, ld)


def test_decode_step_rejects_bad_arguments():
    cfg = dict(TINY)
    m = oracle.Model(cfg, qdsynth.model_tensors(cfg, seed=1))
    kc = np.zeros((2, 2, 8, 16), np.float32)
    with pytest.raises(ValueError):
        m.decode_step(kc, kc.copy(), 2 * 8 * 16, 8, 1)  # pos == max_ctx
    with pytest.raises(ValueError):
        m.decode_step(kc, kc.copy(), 2 * 8 * 16, 0, 100)  # token == vocab
