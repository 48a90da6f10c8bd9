"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test checks the oracle against something other than itself: hand-worked blocks from
``tests/golden``, closed forms, invariants, special cases that reduce to a library routine,
or brute force on tiny inputs.  Together they are chosen so that a dropped term, a wrong sign
or index, or a transposed operand anywhere in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import qdsynth
from conftest import golden_rows

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------- scalar formats

def test_f16_all_patterns_vs_torch():
    """binary16 decode of all 65,536 patterns equals torch's float16 -> float32 conversion."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16).float().numpy()
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits], dtype=np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan].astype(np.float64))
    arr = oracle.f16_to_f32_array(bits)
    assert np.array_equal(arr.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])
    # float16 -> float32 is exact, so the double must already be an f32 value
    assert np.array_equal(got[~nan].astype(np.float32).astype(np.float64), got[~nan])


def test_bf16_all_patterns_zero_extension():
    """BF16 -> F32 is the zero-extension bits << 16 (minillm-cpp README, "Loader"),
    bit-exact against both the shift and torch's bfloat16 -> float32."""
    bits = np.arange(65536, dtype=np.uint32)
    shifted = (bits << 16).astype(np.uint32).view(np.float32)
    tref = torch.from_numpy(bits.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = oracle.bf16_to_f32_array(bits.astype(np.uint16))
    assert oracle.bf16_to_f32(0x3F80) == 1.0 and oracle.bf16_to_f32(0xC000) == -2.0
    assert np.array_equal(got.view(np.uint32), shifted.view(np.uint32))
    assert np.array_equal(got.view(np.uint32), tref.view(np.uint32))


# --------------------------------------------------------------------------- Q4_0

def _hand_q4_0():
    rows = golden_rows("q4_0_hand_blocks.txt")
    out = []
    for r in rows:
        d = int(r[0], 16)
        qs = bytes.fromhex(r[1])
        vals = np.array([float(v) for v in r[2:34]])
        total = float(r[34])
        blk = np.frombuffer(bytes([d & 0xFF, d >> 8]) + qs, dtype=np.uint8)
        out.append((blk, vals, total))
    return out


def test_q4_0_hand_blocks():
    for blk, vals, total in _hand_q4_0():
        deq = oracle.dequant("q4_0", blk, 1, 32)[0]
        assert np.array_equal(deq.astype(np.float64), vals)
        y = oracle.gemv("q4_0", blk, 1, 32, np.ones((1, 32), np.float32))
        assert y[0, 0] == total


def test_q4_0_ones_row_sums_closed_form():
    """All-ones x: row r sums to sum_b d_b (sum of the 32 codes - 256)."""
    rows, cols = 7, 256
    w = qdsynth.q4_0_blocks(3, "w", rows, cols)
    d = w[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qs = w[:, :, 2:].astype(np.int64)
    code_sum = (qs & 0xF).sum(-1) + (qs >> 4).sum(-1)
    expect = (d * (code_sum - 256)).sum(-1)
    y = oracle.gemv("q4_0", w, rows, cols, np.ones((1, cols), np.float32))[0]
    assert np.allclose(y, expect, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- Q8_0

def test_q8_0_block_values_and_ones():
    rows, cols = 5, 128
    w = qdsynth.q8_0_blocks(4, "w", rows, cols)
    d = w[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    q = w[:, :, 2:].view(np.int8).astype(np.int64)
    # hand case: d = 1.0 -> values are the codes
    blk = np.concatenate([np.array([0x00, 0x3C], np.uint8), np.arange(-16, 16, dtype=np.int8).view(np.uint8)])
    assert np.array_equal(oracle.dequant("q8_0", blk, 1, 32)[0], np.arange(-16, 16, dtype=np.float32))
    y = oracle.gemv("q8_0", w, rows, cols, np.ones((1, cols), np.float32))[0]
    assert np.allclose(y, (d * q.sum(-1)).sum(-1), rtol=0, atol=1e-12)
    assert np.all(np.abs(q) <= 127)


# --------------------------------------------------------------------------- Q4_K

def test_q4_k_scale_min_hand_cases():
    for r in golden_rows("q4_k_scale_min.txt"):
        q12 = np.frombuffer(bytes.fromhex(r[0]), dtype=np.uint8)
        want = [int(v) for v in r[1:17]]
        got = []
        for j in range(8):
            got += list(oracle.get_scale_min_k4(j, q12))
        assert got == want, r[0]


def _pack_scale_min(sc, m):
    """Pack eight 6-bit (scale, min) pairs as the Q4_K field is described in words."""
    q = [0] * 12
    for j in range(4):
        q[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        q[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        q[j + 8] = (sc[j + 4] & 0xF) | ((m[j + 4] & 0xF) << 4)
    return np.array(q, dtype=np.uint8)


def test_q4_k_scale_min_round_trip():
    rng = np.random.default_rng(0)
    for _ in range(500):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        q = _pack_scale_min(sc, m)
        for j in range(8):
            assert oracle.get_scale_min_k4(j, q) == (sc[j], m[j])


def test_q4_k_element_order_and_formula():
    """A super-block whose value at each element identifies that element's code position."""
    sc = [1, 2, 3, 4, 5, 6, 7, 8]
    m = [0, 1, 0, 2, 0, 3, 0, 4]
    scales = _pack_scale_min(sc, m)
    qs = np.array([(l % 16) | (((l + c) % 16) << 4) for c in range(4) for l in range(32)], dtype=np.uint8)
    d, dmin = 0x3C00, 0x3800  # 1.0, 0.5
    blk = np.concatenate([np.array([d & 0xFF, d >> 8, dmin & 0xFF, dmin >> 8], np.uint8), scales, qs])
    deq = oracle.dequant("q4_k", blk, 1, 256)[0].astype(np.float64)
    for c in range(4):
        for l in range(32):
            lo, hi = l % 16, (l + c) % 16
            assert deq[64 * c + l] == 1.0 * sc[2 * c] * lo - 0.5 * m[2 * c]
            assert deq[64 * c + 32 + l] == 1.0 * sc[2 * c + 1] * hi - 0.5 * m[2 * c + 1]
    # zero scale bytes -> every value is 0
    blk0 = blk.copy()
    blk0[4:16] = 0
    assert np.all(oracle.dequant("q4_k", blk0, 1, 256) == 0)


def test_q4_k_ones_row_sums_closed_form():
    rows, cols = 3, 512
    w = qdsynth.q4_k_blocks(5, "w", rows, cols)
    expect = np.zeros(rows)
    for r in range(rows):
        for s in range(cols // 256):
            b = w[r, s]
            d = float(b[0:2].copy().view(np.float16)[0])
            dm = float(b[2:4].copy().view(np.float16)[0])
            qs = b[16:].astype(np.int64)
            for j in range(8):
                scj, mj = oracle.get_scale_min_k4(j, b[4:16])
                c, hi = divmod(j, 2)
                codes = (qs[32 * c:32 * c + 32] >> 4) if hi else (qs[32 * c:32 * c + 32] & 0xF)
                expect[r] += d * scj * codes.sum() - 32 * dm * mj
    y = oracle.gemv("q4_k", w, rows, cols, np.ones((1, cols), np.float32))[0]
    # each element is rounded to f32 before the sum; the closed form is exact
    assert np.allclose(y, expect, rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------- INT8 per row

def test_i8_row_values():
    rows, cols = 4, 48
    q, s = qdsynth.i8_row(6, "w", rows, cols)
    src = np.concatenate([q.reshape(-1).view(np.uint8), s.view(np.uint8)])
    deq = oracle.dequant("i8", src, rows, cols)
    assert np.array_equal(deq, (q.astype(np.float64) * s.astype(np.float64)[:, None]).astype(np.float32))
    y = oracle.gemv("i8", src, rows, cols, np.ones((1, cols), np.float32))[0]
    assert np.allclose(y, s.astype(np.float64) * q.astype(np.int64).sum(1), rtol=1e-6)


# --------------------------------------------------------------------------- GEMV

@pytest.mark.parametrize("fmt,cols", [("q4_0", 96), ("q8_0", 96), ("q4_k", 256), ("i8", 80)])
def test_gemv_unit_vectors_give_columns(fmt, cols):
    """W . e_c is column c of the dequantised matrix (catches a transposed operand)."""
    rows = 6
    w = qdsynth.weight_src(fmt, 7, "w", rows, cols)
    deq = oracle.dequant(fmt, w, rows, cols).astype(np.float64)
    eye = np.eye(cols, dtype=np.float32)
    y = oracle.gemv(fmt, w, rows, cols, eye)  # [cols][rows]
    assert np.array_equal(y, deq.T)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "i8"])
def test_gemv_exact_integer_case(fmt):
    """d = 2^-k and integer x: every partial sum is exact, so the result equals integer math."""
    rows, cols, k = 9, 192, 3
    if fmt == "i8":
        q, _ = qdsynth.i8_row(8, "w", rows, cols)
        s = np.full(rows, 2.0 ** -k, np.float32)
        w = np.concatenate([q.reshape(-1).view(np.uint8), s.view(np.uint8)])
        codes = q.astype(np.int64)
    else:
        w = qdsynth.weight_src(fmt, 8, "w", rows, cols).reshape(rows, cols // 32, -1).copy()
        w[:, :, 0:2] = np.array([2.0 ** -k], np.float16).view(np.uint8)
        if fmt == "q4_0":
            qs = w[:, :, 2:].astype(np.int64)
            codes = np.concatenate([(qs & 0xF), (qs >> 4)], axis=-1) - 8
        else:
            codes = w[:, :, 2:].view(np.int8).astype(np.int64)
        codes = codes.reshape(rows, cols)
        w = w.reshape(-1)
    x = qdsynth.ints_i32(8, "x", 2 * cols, -4, 4).reshape(2, cols)
    want = (x.astype(np.int64) @ codes.T).astype(np.float64) * 2.0 ** -k
    y = oracle.gemv(fmt, w, rows, cols, x.astype(np.float32))
    assert np.array_equal(y, want)


@pytest.mark.parametrize("fmt,rows,cols", [("q4_0", 576, 1536), ("q8_0", 33, 640), ("q4_k", 17, 1024),
                                           ("i8", 40, 2048)])
def test_gemv_vs_library_matmul(fmt, rows, cols):
    """The oracle's loop equals torch's float64 matmul of its own dequantised matrix."""
    w = qdsynth.weight_src(fmt, 0, "w", rows, cols)
    x = qdsynth.activations(0, "x", 3, cols)
    deq = torch.from_numpy(oracle.dequant(fmt, w, rows, cols)).double()
    ref = (torch.from_numpy(x).double() @ deq.T).numpy()
    y = oracle.gemv(fmt, w, rows, cols, x)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # row slicing returns the same rows
    ys = oracle.gemv(fmt, w, rows, cols, x, row0=rows // 3, nrows=5)
    assert np.array_equal(ys, y[:, rows // 3:rows // 3 + 5])


# --------------------------------------------------------------------------- RMSNorm

def test_rmsnorm_unit_rms_and_scale_invariance():
    x = qdsynth.activations(1, "x", 2, 576)
    g = np.ones(576, np.float32)
    out = oracle.rmsnorm(x, g, 0.0)
    assert np.allclose(np.sqrt((out ** 2).mean(-1)), 1.0, rtol=1e-12)
    out2 = oracle.rmsnorm(x * np.float32(4.0), g, 0.0)
    assert np.allclose(out, out2, rtol=1e-12)
    gg = qdsynth.norm_gains(1, "g", 576)
    assert np.allclose(oracle.rmsnorm(x, gg, 0.0), out * gg, rtol=1e-12)


def test_rmsnorm_eps_inside_root():
    """For a constant vector c: out = c g / sqrt(c^2 + eps) (eps under the square root)."""
    for c, eps in [(0.01, 1e-5), (2.0, 1e-5), (0.0, 1e-5), (3e-3, 1e-2)]:
        x = np.full((1, 64), c, np.float32)
        g = np.linspace(0.5, 1.5, 64).astype(np.float32)
        out = oracle.rmsnorm(x, g, eps)[0]
        cf = float(np.float32(c))
        assert np.allclose(out, cf * g.astype(np.float64) / math.sqrt(cf * cf + eps), rtol=1e-12, atol=0)


# --------------------------------------------------------------------------- RoPE

def test_rope_hand_angles():
    # hd = 2, pos = 1: one pair turned by exactly 1 rad (theta^0 = 1)
    v = np.array([1.0, 2.0], np.float32)
    out = oracle.rope(v, 1, 2, 1, "adjacent", 1e4)
    assert np.allclose(out, [math.cos(1) - 2 * math.sin(1), math.sin(1) + 2 * math.cos(1)], rtol=1e-14)
    # hd = 4, theta = 1e4, pos = 100: pair 1 turns by 100 * 1e4^(-1/2) = 1 rad, pair 0 by 100 rad
    v = np.array([1.0, 0.0, 0.0, 1.0], np.float32)  # adjacent pairs: (x0,x1)=(1,0), (x2,x3)=(0,1)
    out = oracle.rope(v, 1, 4, 100, "adjacent", 1e4)
    assert np.allclose(out, [math.cos(100), math.sin(100), -math.sin(1), math.cos(1)], rtol=1e-12)
    # the same numbers with half pairing: pairs (0,2) and (1,3)
    v = np.array([1.0, 0.0, 0.0, 1.0], np.float32)
    out = oracle.rope(v, 1, 4, 100, "half", 1e4)
    assert np.allclose(out, [math.cos(100), -math.sin(1), math.sin(100), math.cos(1)], rtol=1e-12)


def test_rope_identity_norms_relative_and_permutation():
    hd, H = 64, 3
    v = qdsynth.activations(2, "v", 1, H * hd)[0]
    w = qdsynth.activations(2, "w", 1, H * hd)[0]
    for pairing in ("adjacent", "half"):
        assert np.array_equal(oracle.rope(v, H, hd, 0, pairing, 1e5), v.astype(np.float64))
        out = oracle.rope(v, H, hd, 37, pairing, 1e5).reshape(H, hd)
        vv = v.astype(np.float64).reshape(H, hd)
        if pairing == "adjacent":
            n_in, n_out = vv[:, 0::2] ** 2 + vv[:, 1::2] ** 2, out[:, 0::2] ** 2 + out[:, 1::2] ** 2
        else:
            n_in, n_out = vv[:, :32] ** 2 + vv[:, 32:] ** 2, out[:, :32] ** 2 + out[:, 32:] ** 2
        assert np.allclose(n_in, n_out, rtol=1e-12)
        # relative position: rope(q, m) . rope(k, n) depends on m - n only
        a = oracle.rope(v, H, hd, 10, pairing, 1e5) @ oracle.rope(w, H, hd, 3, pairing, 1e5)
        b = oracle.rope(v, H, hd, 110, pairing, 1e5) @ oracle.rope(w, H, hd, 103, pairing, 1e5)
        assert abs(a - b) < 1e-9 * max(1.0, abs(a))
    # permutation: half pairing on P v equals P applied to adjacent pairing of v
    perm = np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])  # (2i,2i+1) -> (i, i+hd/2)
    vh = v.reshape(H, hd)[:, perm].reshape(-1)
    adj = oracle.rope(v, H, hd, 77, "adjacent", 1e5).reshape(H, hd)[:, perm].reshape(-1)
    assert np.allclose(oracle.rope(vh, H, hd, 77, "half", 1e5), adj, rtol=0, atol=1e-12)


def test_rope_table_matches_angles():
    hd, ctx, theta = 64, 50, 1e5
    t = oracle.rope_table(theta, hd, ctx)
    p = np.arange(ctx)[:, None].astype(np.float64)
    ang = p * theta ** (-2.0 * np.arange(hd // 2)[None, :] / hd)
    assert np.allclose(t[..., 0], np.cos(ang), rtol=0, atol=1e-7)
    assert np.allclose(t[..., 1], np.sin(ang), rtol=0, atol=1e-7)
    assert np.array_equal(t[0, :, 0], np.ones(hd // 2, np.float32))
    assert np.array_equal(t[0, :, 1], np.zeros(hd // 2, np.float32))


# --------------------------------------------------------------------------- attention

def test_attention_two_token_brute_force():
    hq = hk = 1
    hd, ctx = 8, 4
    q = qdsynth.activations(3, "q", 1, hd)[0]
    k = qdsynth.activations(3, "k", 1, ctx * hd)[0]
    v = qdsynth.activations(3, "v", 1, ctx * hd)[0]
    out = oracle.attention(q, k, v, hq, hk, hd, 2, ctx)
    qd, kd, vd = q.astype(np.float64), k.astype(np.float64).reshape(ctx, hd), v.astype(np.float64).reshape(ctx, hd)
    s0, s1 = qd @ kd[0] / math.sqrt(hd), qd @ kd[1] / math.sqrt(hd)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert np.allclose(out, w0 * vd[0] + (1 - w0) * vd[1], rtol=1e-12, atol=1e-14)
    # a single position returns its value row exactly
    assert np.array_equal(oracle.attention(q, k, v, hq, hk, hd, 1, ctx), vd[0])


def test_attention_gqa_head_mapping_and_uniform_keys():
    hq, hk, hd, ctx, n = 6, 2, 4, 8, 5
    q = qdsynth.activations(4, "q", 1, hq * hd)[0]
    k = np.zeros((hk, ctx, hd), np.float32)  # equal keys -> uniform weights
    v = np.zeros((hk, ctx, hd), np.float32)
    for j in range(hk):
        v[j, :n] = (j + 1) * 10 + np.arange(n)[:, None]
    out = oracle.attention(q, k, v, hq, hk, hd, n, ctx).reshape(hq, hd)
    for h in range(hq):
        j = h // (hq // hk)  # heads 0-2 share kv head 0, heads 3-5 kv head 1
        assert np.allclose(out[h], v[j, :n].astype(np.float64).mean(0), rtol=1e-14)


# --------------------------------------------------------------------------- SwiGLU / argmax

def test_silu_and_swiglu():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    g = np.array([0.0, 1.0, -2.0, 3.0], np.float32)
    u = np.array([5.0, 2.0, 1.0, -1.0], np.float32)
    want = [0.0, 2.0 / (1 + math.exp(-1)), -2.0 / (1 + math.exp(2)), -3.0 / (1 + math.exp(-3))]
    assert np.allclose(oracle.swiglu(g, u), want, rtol=1e-15)


def test_argmax_first_index_on_ties():
    v = np.array([1.0, 3.0, 2.0, 3.0, 3.0], np.float32)
    assert oracle.argmax(v) == 1
    assert oracle.argmax(np.full(10, 7.0, np.float32)) == 0
    assert oracle.argmax(np.array([-5.0, -1.0, -1.0], np.float64)) == 1
    x = qdsynth.activations(9, "l", 1, 49152)[0]
    assert oracle.argmax(x) == int(np.argmax(x))  # numpy also returns the first maximum


def test_double_input_forms_equal_their_f32_forms():
    """The decode step's double-input forms of the product, RMSNorm, RoPE and attention (the
    forms the step composes) give the same bits as the pinned f32-input forms above when the
    double input holds f32 values, and differ when it does not (they read all 53 bits)."""
    rows, cols = 40, 128
    w = qdsynth.weight_src("q4_0", 31, "dform.w", rows, cols)
    x = qdsynth.activations(31, "dform.x", 2, cols)
    assert np.array_equal(oracle.gemv_xd("q4_0", w, rows, cols, x.astype(np.float64)),
                          oracle.gemv("q4_0", w, rows, cols, x))
    g = qdsynth.uniform_f32(31, "dform.g", cols, 0.9, 1.1)
    assert np.array_equal(oracle.rmsnorm_d(x[0].astype(np.float64), g, 1e-5), oracle.rmsnorm(x[0], g, 1e-5)[0])
    hd = 64
    v = x.reshape(-1)[:2 * hd]
    for pairing in ("adjacent", "half"):
        assert np.array_equal(oracle.rope_d(v.astype(np.float64), 2, hd, 7, pairing, 1e4),
                              oracle.rope(v, 2, hd, 7, pairing, 1e4))
    ctx = 8
    kc = qdsynth.normal_f32(31, "dform.k", 2 * ctx * hd)
    vc = qdsynth.normal_f32(31, "dform.v", 2 * ctx * hd)
    q = qdsynth.normal_f32(31, "dform.q", 4 * hd)
    assert np.array_equal(oracle.attention_d(q.astype(np.float64), kc, vc, 4, 2, hd, 5, ctx),
                          oracle.attention(q, kc, vc, 4, 2, hd, 5, ctx))
    # a double input off the f32 grid changes the result: nothing rounds it to f32 first
    xd = x[0].astype(np.float64) * (1.0 + 2.0 ** -40)
    assert not np.array_equal(oracle.gemv_xd("q4_0", w, rows, cols, xd), oracle.gemv("q4_0", w, rows, cols, x[0]))
