"""Pins for the oracle's per-row INT8 quantiser of BF16 weights (minillm-cpp README,
"Direct INT8 loading" and "Quantization": symmetric, one scale per output row; the rule
s = max|w| / 127, q = round(w / s) with ties away from zero is the reading taken where
the page prints none).  Checked against hand-worked rows, a brute-force nearest-code
search, and properties any correct symmetric per-row quantiser has."""
import numpy as np

import oracle
import qdsynth


def bf16(v) -> np.ndarray:
    """f32 values that are exact in bf16 -> bf16 bit patterns (truncation is exact here)."""
    a = np.asarray(v, np.float32)
    bits = (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(((bits.astype(np.uint32)) << 16).view(np.float32), a), "value not exact in bf16"
    return bits


def random_bf16(seed: int, name: str, rows: int, cols: int) -> np.ndarray:
    """N(0,1) values rounded to bf16 (round to nearest even on the f32 bit pattern)."""
    x = qdsynth.activations(seed, name, rows, cols).astype(np.float32).reshape(-1)
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r.reshape(rows, cols)


def as_f32(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_hand_worked_row_with_unit_scale():
    # max |w| = 127 -> s = 1 exactly, so the codes are the values rounded, ties away from 0
    w = bf16([127, 2.5, -2.5, 0.5, -0.5, 1.5, 3.75, -126.5, 0, 1, -1, 63.25, -0.25, 0.75, 100, -100])
    q, s = oracle.quantize_i8_rows(w, 1, 16)
    assert s[0] == 1.0
    assert q[0].tolist() == [127, 3, -3, 1, -1, 2, 4, -127, 0, 1, -1, 63, 0, 1, 100, -100]


def test_hand_worked_row_with_fractional_scale():
    # max |w| = 0.5 -> s = 0.5/127; w = 0.25 is 63.5 s up to rounding of s and of the
    # quotient: it must land on 63 or 64; the extremes on +-127; zero on 0
    w = bf16([0.5, -0.5, 0.25, 0.0] + [0.0] * 12)
    q, s = oracle.quantize_i8_rows(w, 1, 16)
    assert s[0] == np.float32(np.float32(0.5) / np.float32(127.0))
    assert q[0, 0] == 127 and q[0, 1] == -127 and q[0, 2] in (63, 64) and q[0, 3] == 0


def test_codes_are_the_nearest_code_by_brute_force():
    rows, cols = 24, 96
    w = random_bf16(41, "quant.bf", rows, cols)
    q, s = oracle.quantize_i8_rows(w, rows, cols)
    wf = as_f32(w).astype(np.float64)
    cand = np.arange(-127, 128, dtype=np.float64)
    mism = 0
    for r in range(rows):
        sd = float(s[r])
        assert sd == np.float32(np.abs(as_f32(w[r])).max() / np.float32(127.0))
        for c in range(cols):
            err = np.abs(cand * sd - wf[r, c])
            best = cand[err == err.min()]
            pick = best[np.argmax(np.abs(best))]  # a tie goes away from zero
            if q[r, c] != pick:
                # only where the exact quotient sits within f32 rounding of a half-way point
                t = wf[r, c] / sd
                assert abs(abs(t - np.trunc(t)) - 0.5) < 1e-5, (r, c, q[r, c], pick, t)
                mism += 1
    assert mism <= 2


def test_error_bound_and_full_range():
    rows, cols = 32, 160
    w = random_bf16(42, "quant.bf2", rows, cols)
    q, s = oracle.quantize_i8_rows(w, rows, cols)
    wf = as_f32(w).astype(np.float64)
    recon = q.astype(np.float64) * s.astype(np.float64)[:, None]
    # half a step, plus the f32 rounding of the quotient w / s (|w / s| <= 127: 127 * 2^-24)
    assert np.all(np.abs(recon - wf) <= s.astype(np.float64)[:, None] * (0.5 + 2e-5))
    assert np.all(np.abs(q).max(axis=1) == 127)
    for r in range(rows):
        assert abs(int(q[r, np.argmax(np.abs(wf[r]))])) == 127


def test_sign_symmetry_and_power_of_two_invariance():
    rows, cols = 16, 64
    w = random_bf16(43, "quant.bf3", rows, cols)
    q, s = oracle.quantize_i8_rows(w, rows, cols)
    qn, sn = oracle.quantize_i8_rows(w ^ np.uint16(0x8000), rows, cols)  # flip every sign bit
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    w4 = bf16(as_f32(w) * np.float32(4.0))  # exponent + 2: exact
    q4, s4 = oracle.quantize_i8_rows(w4, rows, cols)
    assert np.array_equal(q4, q) and np.array_equal(s4, s * np.float32(4.0))


def test_zero_and_non_finite_rows():
    w = np.zeros((3, 16), np.uint16)
    w[1, :] = bf16(np.ones(16, np.float32))
    w[2, 5] = 0x7FC0  # bf16 NaN
    w[2, 6] = bf16([3.0])[0]
    q, s = oracle.quantize_i8_rows(w, 3, 16)
    assert s[0] == 0.0 and not q[0].any()
    assert s[1] == np.float32(1.0 / 127.0) and np.all(q[1] == 127)
    assert np.isnan(s[2]) and not q[2].any()
    w[2, 5] = 0x7F80  # +inf
    q, s = oracle.quantize_i8_rows(w, 3, 16)
    assert np.isnan(s[2]) and not q[2].any()


def test_round_f16_worked_values():
    """RoundF16 (go-llm index: what an f16 KV cache stores): nearest binary16, ties to even."""
    r = oracle.round_f16
    assert r(1.0) == 1.0 and r(-2.5) == -2.5
    assert r(1.0 / 3.0) == 0.333251953125                       # 1/3 -> 0x3555
    assert r(65504.0) == 65504.0 and r(65519.0) == 65504.0      # largest finite
    assert r(65520.0) == np.inf and r(-70000.0) == -np.inf      # the tie at 65520 rounds up to inf
    assert r(1.0 + 2.0 ** -11) == 1.0                           # tie, even significand below
    assert r(1.0 + 3 * 2.0 ** -11) == 1.0 + 2.0 ** -9           # tie, even significand above
    assert r(2.0 ** -24) == 2.0 ** -24 and r(2.0 ** -25) == 0.0  # smallest subnormal; tie to 0
    assert r(3 * 2.0 ** -26) == 2.0 ** -24
    assert np.isnan(r(np.nan))
    assert np.signbit(r(-0.0)) and r(-0.0) == 0.0


def test_round_f16_matches_numpy_binary16_on_random_values():
    # numpy's float32 -> float16 cast is round-to-nearest-even: an independent implementation
    x = np.concatenate([qdsynth.activations(44, "f16.rt", 1, 4000).reshape(-1) * 3.0,
                        qdsynth.activations(45, "f16.rt2", 1, 2000).reshape(-1) * 1e-5,
                        qdsynth.activations(46, "f16.rt3", 1, 2000).reshape(-1) * 3e4]).astype(np.float32)
    got = np.array([oracle.round_f16(v) for v in x], np.float32)
    with np.errstate(over="ignore"):  # values past 65504 become infinity, as intended
        want = x.astype(np.float16).astype(np.float32)
    assert np.array_equal(got, want)
