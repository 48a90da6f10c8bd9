"""Pins of the oracle's ggml-exact activation path (go-llm type CPU, "ExactGGML": activations
quantised to Q8_0, Q8_1 for Q4_1 weights, before every quantised product).  The page prints
no quantisation rule; the reading (or_quantize_q8): per 32 values d = max|x| / 127 in f32,
q = x / d rounded to nearest with ties away from zero, d kept in binary16 (Q8_1 also
s = d * sum q in binary16).  Pinned by hand-worked blocks whose d is exact, and by the
identity with the already-pinned f32-activation product when x is exactly q * 2^-k."""
import numpy as np
import pytest

import oracle
import qdsynth


def test_quantize_hand_block_d_one():
    # max |x| = 127 -> d = 1 exactly; codes are x rounded, ties away from zero
    x = np.zeros(32, np.float32)
    x[:8] = [-127.0, 126.5, -0.5, 0.5, 2.5, -2.5, 1.49, -100.25]
    q, d, s = oracle.quantize_q8(x[None, :], with_sum=True)
    assert q[0, :8].tolist() == [-127, 127, -1, 1, 3, -3, 1, -100]
    assert (q[0, 8:] == 0).all()
    assert d[0, 0] == 1.0
    assert s[0, 0] == -99.0  # d * (-127 + 127 - 1 + 1 + 3 - 3 + 1 - 100)


def test_quantize_hand_block_d_half():
    # max |x| = 63.5 -> d = 0.5 exactly: 0.25 / 0.5 = 0.5 -> 1, -0.75 / 0.5 = -1.5 -> -2
    x = np.zeros(32, np.float32)
    x[0], x[1], x[2], x[31] = 63.5, 0.25, -0.75, -10.0
    q, d, _ = oracle.quantize_q8(x[None, :])
    assert (q[0, 0], q[0, 1], q[0, 2], q[0, 31]) == (127, 1, -2, -20)
    assert d[0, 0] == 0.5


def test_quantize_zero_and_non_finite_blocks():
    x = np.zeros((1, 96), np.float32)
    x[0, 40] = np.nan
    x[0, 64:] = 3.0
    q, d, s = oracle.quantize_q8(x, with_sum=True)
    assert d[0, 0] == 0.0 and s[0, 0] == 0.0 and (q[0, :32] == 0).all()       # zero block
    assert np.isnan(d[0, 1]) and np.isnan(s[0, 1]) and (q[0, 32:64] == 0).all()  # NaN block
    assert (q[0, 64:] == 127).all() and d[0, 2] == np.float32(np.float16(3.0 / 127))


def test_product_hand_block():
    # W: one Q8_0 block, d_w = 0.25, code 4 at element 0; x: 127 at element 0 (d_x = 1)
    blk = np.zeros(34, np.uint8)
    blk[0:2] = np.array([0.25], np.float16).view(np.uint8)
    blk[2] = 4
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0
    q, d, _ = oracle.quantize_q8(x)
    assert oracle.gemv_q8act("q8_0", blk, 1, 32, q, d)[0, 0] == 127.0  # 0.25 * 1 * 4 * 127


def _exact_x(seed, batch, cols, k):
    """x = q * 2^-k with every block's largest |q| = 127: the quantiser returns q and
    d = 2^-k exactly."""
    q = qdsynth.ints_i32(seed, "xq", batch * cols, -20, 20).reshape(batch, cols)
    q[:, ::32] = 127
    return (q * 2.0 ** -k).astype(np.float32), q


def test_product_equals_f32_product_for_exact_x():
    for fmt in ("q8_0", "q4_0"):
        rows, cols = 9, 256
        w = qdsynth.weight_src(fmt, 11, "w" + fmt, rows, cols)
        x, qx = _exact_x(11, 3, cols, 6)
        q, d, _ = oracle.quantize_q8(x)
        assert np.array_equal(q, qx) and (d == 2.0 ** -6).all()
        np.testing.assert_allclose(oracle.gemv_q8act(fmt, w, rows, cols, q, d), oracle.gemv(fmt, w, rows, cols, x),
                                   rtol=1e-12, atol=0)


def test_q4_1_product_uses_the_block_sum():
    # Q4_1: sum (d q_w + m) x = d d_x sum q_w q_x + m * (d_x sum q_x); with x exact and the
    # block sums small, s = d_x sum q_x is exact in binary16 and the two products agree
    rows, cols = 7, 128
    w = qdsynth.weight_src("q4_1", 12, "w41", rows, cols)
    x, qx = _exact_x(12, 2, cols, 5)
    q, d, s = oracle.quantize_q8(x, with_sum=True)
    assert np.array_equal(s, (qx.reshape(2, -1, 32).sum(axis=2) * 2.0 ** -5).astype(np.float32))
    np.testing.assert_allclose(oracle.gemv_q8act("q4_1", w, rows, cols, q, d, s),
                               oracle.gemv("q4_1", w, rows, cols, x), rtol=1e-12, atol=0)


TINY_Q8 = dict(layers=2, dim=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64, vocab=300, rope_theta=1e4,
               eps=1e-5, pairing="half", w_fmt="q4_0", emb_fmt="q8_0", max_ctx=16)


def _round_f16_vec(a):
    return np.array([oracle.round_f16(float(v)) for v in np.asarray(a, np.float32)], np.float32)


def _composed_mode_step(cfg, T, kc, vc, pos, tok, act_q8, kv_f16):
    """One decode step rebuilt from separately pinned operations, in the step's own precision
    (x and every intermediate vector double).  act_q8: every quantised product takes its
    input rounded to f32 and quantised to Q8_0 -- Q8_1 for Q4_1 weights -- after the norm
    gains, and multiplies in integers (go-llm "ExactGGML"); kv_f16: the appended k and v,
    rounded to f32, go through binary16 (go-llm RoundF16).  The head's input is quantised
    once."""
    D, F, hd = cfg["dim"], cfg["ffn"], cfg["head_dim"]
    hq, hk, ctx = cfg["n_heads"], cfg["n_kv_heads"], cfg["max_ctx"]
    wf, ef = cfg["w_fmt"], cfg["emb_fmt"]

    def prod(fmt, w, rows, cols, xd):
        if not act_q8:
            return oracle.gemv_xd(fmt, w, rows, cols, xd)[0]
        q, d, s = oracle.quantize_q8(np.asarray(xd, np.float32)[None, :], with_sum=fmt == "q4_1")
        return oracle.gemv_q8act(fmt, w, rows, cols, q, d, s)[0]

    x = oracle.dequant(ef, T[0], cfg["vocab"], D, row0=tok, nrows=1)[0].astype(np.float64)
    for l in range(cfg["layers"]):
        an, wq, wk, wv, wo, fn, wg, wu, wd = T[3 + 9 * l:12 + 9 * l]
        xn = oracle.rmsnorm_d(x, an, cfg["eps"])
        q = oracle.rope_d(prod(wf, wq, hq * hd, D, xn), hq, hd, pos, cfg["pairing"], cfg["rope_theta"])
        k = oracle.rope_d(prod(wf, wk, hk * hd, D, xn), hk, hd, pos, cfg["pairing"], cfg["rope_theta"])
        v = prod(wf, wv, hk * hd, D, xn)
        kf, vf = k.astype(np.float32), v.astype(np.float32)
        if kv_f16:
            kf, vf = _round_f16_vec(kf), _round_f16_vec(vf)
        kc[l][:, pos, :] = kf.reshape(hk, hd)
        vc[l][:, pos, :] = vf.reshape(hk, hd)
        att = oracle.attention_d(q, kc[l], vc[l], hq, hk, hd, pos + 1, ctx)
        x = x + prod(wf, wo, D, hq * hd, att)
        xn = oracle.rmsnorm_d(x, fn, cfg["eps"])
        g = prod(wf, wg, F, D, xn)
        u = prod(wf, wu, F, D, xn)
        a = np.array([oracle.silu(float(gi)) for gi in g]) * u
        x = x + prod(wf, wd, D, F, a)
    xn = oracle.rmsnorm_d(x, T[1], cfg["eps"])
    return prod(ef, T[0] if T[2] is None else T[2], cfg["vocab"], D, xn)


@pytest.mark.parametrize("w_fmt", ["q4_0", "q8_0", "q4_1"])
def test_decode_step_modes_equal_composition(w_fmt):
    """The oracle's decode step in each of its modes (Q8 activations and / or the binary16
    cache) equals, bit for bit, the step rebuilt from the separately pinned quantiser,
    integer product, binary16 rounding, norm, RoPE, attention and SwiGLU.  A wiring mistake
    (a product left in f32, Q8_0 where Q4_1 needs Q8_1, quantising before the gains, the
    head's input quantised twice, v or k not rounded through binary16) changes bits."""
    cfg = dict(TINY_Q8, w_fmt=w_fmt)
    host = qdsynth.model_tensors(cfg, 3)
    L, hk, ctx, hd = cfg["layers"], cfg["n_kv_heads"], cfg["max_ctx"], cfg["head_dim"]
    per = hk * ctx * hd
    last = {}
    for act_q8, kv_f16 in ((0, 0), (1, 0), (0, 1), (1, 1)):
        if w_fmt == "q4_1" and not act_q8:
            continue
        om = oracle.Model(dict(cfg, act_q8=act_q8, kv_f16=kv_f16), host)
        kc = np.zeros(L * per, np.float32)
        vc = np.zeros_like(kc)
        kc2 = [np.zeros((hk, ctx, hd), np.float32) for _ in range(L)]
        vc2 = [np.zeros((hk, ctx, hd), np.float32) for _ in range(L)]
        for p, tok in enumerate([5, 17, 200, 33]):
            lg, nxt = om.decode_step(kc, vc, per, p, tok)
            ref = _composed_mode_step(cfg, host, kc2, vc2, p, tok, act_q8, kv_f16)
            assert np.array_equal(lg, ref), (act_q8, kv_f16, p, np.abs(lg - ref).max())
            assert nxt == int(np.argmax(ref))
            for l in range(L):
                assert np.array_equal(kc.reshape(L, hk, ctx, hd)[l, :, p], kc2[l][:, p])
                assert np.array_equal(vc.reshape(L, hk, ctx, hd)[l, :, p], vc2[l][:, p])
        if kv_f16:  # the cache holds binary16 values
            assert np.array_equal(kc, kc.astype(np.float16).astype(np.float32))
        last[(act_q8, kv_f16)] = lg
    # each mode changes the result (so the composition above is not vacuous)
    keys = list(last)
    for i in range(len(keys)):
        for j in range(i + 1, len(keys)):
            assert not np.array_equal(last[keys[i]], last[keys[j]]), (keys[i], keys[j])


def test_decode_step_ggml_exact_mode_close_to_f32():
    """Q8 activations and a binary16 cache stay within the activation quantisation's reach of
    the f32 step (each value moves by at most 1/254 of its block's largest |x|)."""
    cfg = dict(TINY_Q8)
    host = qdsynth.model_tensors(cfg, 3)
    out = {}
    for exact in (False, True):
        om = oracle.Model(dict(cfg, act_q8=exact, kv_f16=exact), host)
        kc = np.zeros(2 * 2 * 16 * 64, np.float32)
        vc = np.zeros_like(kc)
        for p, tok in enumerate([5, 17, 200]):
            lg, _ = om.decode_step(kc, vc, 2 * 16 * 64, p, tok)
        out[exact] = lg
    diff = np.abs(out[True] - out[False]).max() / np.abs(out[False]).max()
    assert 0 < diff < 2e-2


@pytest.mark.parametrize("act_q8,kv_f16", [(0, 0), (1, 1)])
def test_teacher_forcing_hooks(act_q8, kv_f16):
    """or_decode_step_tf: without kv_given it is the step itself; kv_out holds the k and v the
    step appends (before their binary16 rounding); head_x is the head's input; with
    kv_given the step reads the cache at pos as given and leaves it unwritten."""
    cfg = dict(TINY_Q8, act_q8=act_q8, kv_f16=kv_f16)
    host = qdsynth.model_tensors(cfg, 4)
    om = oracle.Model(cfg, host)
    L, hk, ctx, hd = cfg["layers"], cfg["n_kv_heads"], cfg["max_ctx"], cfg["head_dim"]
    per = hk * ctx * hd
    kc, vc = np.zeros(L * per, np.float32), np.zeros(L * per, np.float32)
    kc2, vc2 = kc.copy(), vc.copy()
    for p, tok in enumerate([9, 250, 1]):
        lg, nxt = om.decode_step(kc, vc, per, p, tok)
        lg2, nxt2, kv, hx, xo = om.decode_step_tf(kc2, vc2, per, p, tok, kv_given=False)
        assert np.array_equal(lg, lg2) and nxt == nxt2
        assert np.array_equal(kc, kc2) and np.array_equal(vc, vc2)
        rnd = _round_f16_vec if kv_f16 else (lambda a: a)
        for l in range(L):
            assert np.array_equal(rnd(kv[l, 0]), kc.reshape(L, hk, ctx, hd)[l, :, p].reshape(-1))
            assert np.array_equal(rnd(kv[l, 1]), vc.reshape(L, hk, ctx, hd)[l, :, p].reshape(-1))
        head = host[0] if host[2] is None else host[2]
        if act_q8:
            q, d, _ = oracle.quantize_q8(hx[None, :])
            assert np.array_equal(lg, oracle.gemv_q8act(cfg["emb_fmt"], head, cfg["vocab"], cfg["dim"], q, d)[0])
        else:
            np.testing.assert_allclose(lg, oracle.gemv(cfg["emb_fmt"], head, cfg["vocab"], cfg["dim"], hx)[0],
                                       rtol=0, atol=1e-5 * np.abs(lg).max())
        if act_q8:
            # every product's f32 input: the head's is head_x; feeding back each slot's own
            # quantisation reproduces the step bit for bit
            slots, cols = om.q8_slots()
            assert np.array_equal(xo[slots - 1, :cfg["dim"]], hx)
            qs = np.zeros((slots, cols), np.int8)
            ds = np.zeros((slots, cols // 32), np.float32)
            width = [cfg["dim"], cfg["n_heads"] * cfg["head_dim"], cfg["dim"], cfg["ffn"]] * L + [cfg["dim"]]
            for k in range(slots):
                q, d, _ = oracle.quantize_q8(xo[k, :width[k]][None, :])
                qs[k, :width[k]], ds[k, :width[k] // 32] = q[0], d[0]
            k5, v5 = kc.copy(), vc.copy()
            lg5, _, _, _, xo5 = om.decode_step_tf(k5, v5, per, p, tok, kv_given=True, q8_codes=qs, q8_d=ds)
            assert np.array_equal(lg5, lg) and np.array_equal(xo5, xo)
            # a given code changed in the first layer's attention-output slot: that product uses
            # it, so the inputs formed after it move (the logits depend on the head's slot only)
            q1 = qs.copy()
            q1[1, 3] = q1[1, 3] + (1 if q1[1, 3] < 127 else -1)
            lg6, _, _, _, xo6 = om.decode_step_tf(kc.copy(), vc.copy(), per, p, tok, kv_given=True, q8_codes=q1,
                                                  q8_d=ds)
            assert np.array_equal(xo6[:2], xo[:2]) and not np.array_equal(xo6[2], xo[2])
            assert np.array_equal(lg6, lg)
            q8 = qs.copy()
            q8[slots - 1, 3] = q8[slots - 1, 3] + (1 if q8[slots - 1, 3] < 127 else -1)
            lg7, _, _, _, _ = om.decode_step_tf(kc.copy(), vc.copy(), per, p, tok, kv_given=True, q8_codes=q8, q8_d=ds)
            assert not np.array_equal(lg7, lg)
    # kv_given: the same cache gives the same step; other values at pos are read, not replaced
    p, tok = 3, 42
    base_k, base_v = kc.copy(), vc.copy()
    lg, _ = om.decode_step(kc, vc, per, p, tok)
    k3, v3 = kc.copy(), vc.copy()
    lg3, _, _, _, _ = om.decode_step_tf(k3, v3, per, p, tok, kv_given=True)
    assert np.array_equal(lg, lg3) and np.array_equal(k3, kc)
    k4, v4 = kc.copy(), vc.copy()
    k4.reshape(L, hk, ctx, hd)[:, :, p] *= 2.0
    lg4, _, kv4, _, _ = om.decode_step_tf(k4, v4, per, p, tok, kv_given=True)
    assert not np.array_equal(lg4, lg)
    assert np.array_equal(k4.reshape(L, hk, ctx, hd)[:, :, p], 2.0 * kc.reshape(L, hk, ctx, hd)[:, :, p])
    assert np.array_equal(base_k.reshape(L, hk, ctx, hd)[:, :, :p], k4.reshape(L, hk, ctx, hd)[:, :, :p])


def test_quantize_error_bound_and_extreme_code():
    """Every value lies within half a step of its code times the f32 scale m / 127 (the
    binary16 d differs from it by at most 2^-11 relative, times |q| <= 127), and each
    block's largest |x| takes the code +-127."""
    x = qdsynth.activations(13, "q8bound", 4, 4096)
    q, d, _ = oracle.quantize_q8(x)
    xb = x.reshape(4, -1, 32).astype(np.float64)
    qb = q.reshape(4, -1, 32).astype(np.float64)
    m = np.abs(xb).max(axis=2, keepdims=True)
    step = (m.astype(np.float32) / np.float32(127)).astype(np.float64)
    assert (np.abs(xb - qb * step) <= step * (0.5 + 1e-5)).all()
    d16 = d.reshape(4, -1, 1).astype(np.float64)
    assert (np.abs(d16 - step) <= step * 2.0 ** -11).all()
    assert (np.abs(qb).max(axis=2) == 127).all()
