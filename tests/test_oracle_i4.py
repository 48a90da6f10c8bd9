"""Pins of the oracle's per-row INT4 path (minillm "Quantization": symmetric per-channel INT8
and INT4, one scale per output row; the rule read from it: s = max|w| / 7, codes w / s
rounded to nearest with ties away from zero, clamped to +-7).  Hand-worked rows with an
exact scale, the zero and non-finite rows, and the half-step error bound."""
import numpy as np

import oracle
import qdsynth


def _bf16(vals) -> np.ndarray:
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _codes(packed, cols):
    nib = np.stack([packed & 0x0F, packed >> 4], axis=-1).reshape(-1, cols).astype(np.int16)
    return np.where(nib >= 8, nib - 16, nib)


def test_hand_row_exact_scale():
    # max |w| = 7 -> s = 1; 3.5 -> 4 and -3.5 -> -4 (ties away), 0.5 -> 1, 1.25 -> 1, bf16(6.4)
    # = 6.40625 -> 6
    w = _bf16([[7.0, -7.0, 3.5, -3.5, 0.5, 1.25, 0.0, 6.4]])
    codes, s = oracle.quantize_i4_rows(w, 1, 8)
    assert s[0] == 1.0
    assert _codes(codes, 8).tolist() == [[7, -7, 4, -4, 1, 1, 0, 6]]
    assert codes[0, 0] == 0x97  # element 0 (7) in the low nibble, element 1 (-7 = 0x9) in the high one
    src = np.concatenate([codes.reshape(-1), s.view(np.uint8)])
    assert oracle.dequant("i4", src, 1, 8)[0].tolist() == [7.0, -7.0, 4.0, -4.0, 1.0, 1.0, 0.0, 6.0]


def test_zero_and_non_finite_rows():
    w = np.zeros((3, 4), np.float32)
    w[1, 2] = np.inf
    w[2] = [1.0, -2.0, 0.5, 0.25]
    codes, s = oracle.quantize_i4_rows(_bf16(w), 3, 4)
    assert s[0] == 0.0 and (codes[0] == 0).all()
    assert np.isnan(s[1]) and (codes[1] == 0).all()
    assert s[2] == np.float32(2.0) / np.float32(7.0)
    # s = 2/7 in f32; the quotients in f32 are 3.4999998, -6.9999995, 1.7499999, 0.87499994
    # (below the ties in exact arithmetic), so the codes are 3, -7, 2, 1: the decision is
    # taken in f32, as the rule states
    assert _codes(codes[2:], 4).tolist() == [[3, -7, 2, 1]]


def test_error_bound_and_extreme_code():
    rows, cols = 16, 256
    w = _bf16(qdsynth.activations(61, "i4w", rows, cols))
    codes, s = oracle.quantize_i4_rows(w, rows, cols)
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    q = _codes(codes, cols).astype(np.float64)
    assert (np.abs(wf - q * s[:, None].astype(np.float64)) <= s[:, None] * (0.5 + 1e-5)).all()
    assert (np.abs(q).max(axis=1) == 7).all()
