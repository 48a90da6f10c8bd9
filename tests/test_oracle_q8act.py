"""Pins of the oracle's ggml-exact activation path (go-llm type CPU, "ExactGGML": activations
quantised to Q8_0, Q8_1 for Q4_1 weights, before every quantised product).  The page prints
no quantisation rule; the reading (or_quantize_q8): per 32 values d = max|x| / 127 in f32,
q = x / d rounded to nearest with ties away from zero, d kept in binary16 (Q8_1 also
s = d * sum q in binary16).  Pinned by hand-worked blocks whose d is exact, and by the
identity with the already-pinned f32-activation product when x is exactly q * 2^-k."""
import numpy as np

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


def test_decode_step_ggml_exact_mode_close_to_f32():
    """The decode step with every product over Q8 activations and a binary16 cache stays
    within the activation quantisation's reach of the f32 step (each value moves by at most
    1/254 of its block's largest |x|): 2e-2 of the largest logit over three steps."""
    cfg = dict(layers=2, dim=256, ffn=512, n_heads=4, n_kv_heads=2, head_dim=64, vocab=300, rope_theta=1e4,
               eps=1e-5, pairing="half", w_fmt="q4_0", emb_fmt="q8_0", max_ctx=16)
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
