"""GPU parity of the batched prefill product (qd_q_gemm, tensor cores) against the oracle,
through the C ABI: the contract bound (1e-3 of max |oracle| per token row), a tight bound
against the oracle's dequantised weights rounded to binary16 (the kernel's stated weight
arithmetic), bit-exact power-of-two cases, ragged rows and tokens, several tiles per CTA,
full-size shapes on sampled rows, non-finite x rows."""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import assert_close, dev, packed, weights

pytestmark = pytest.mark.gpu

FMTS = ["q4_0", "q8_0", "i8"]


def _gemm(qd, fmt, p, rows, cols, x):
    t = x.shape[0]
    ws = torch.empty(qd.q_gemm_workspace(fmt, rows, cols, t), dtype=torch.uint8, device="cuda")
    y = torch.full((t, rows), float("nan"), dtype=torch.float32, device="cuda")
    qd.q_gemm(fmt, p, rows, cols, dev(x), y, t, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _binary16_weights_ref(fmt, src, rows, cols, x, row0=0, nrows=None):
    """y with each Q4_0 / Q8_0 weight rounded to binary16 (numpy's round-to-nearest-even
    cast of the oracle's exact f32 value d * q); INT8 rows unchanged.  Double matmul."""
    w = oracle.dequant(fmt, src, rows, cols, row0, nrows).astype(np.float64)
    if fmt != "i8":
        w = oracle.dequant(fmt, src, rows, cols, row0, nrows).astype(np.float16).astype(np.float64)
    return x.astype(np.float64) @ w.T


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols,t", [(584, 576, 1), (584, 576, 64), (100, 1024, 100), (584, 576, 200)])
def test_q_gemm_parity(qd, fmt, rows, cols, t):
    """Three 256-row tiles (the last ragged) or one partial tile; one to four 64-token tiles
    (ragged last); 9-16 stages of 64 columns."""
    src, p = weights(qd, fmt, 31, f"gm{rows}x{cols}", rows, cols)
    x = qdsynth.activations(31, f"gmx{t}x{cols}", t, cols)
    got = _gemm(qd, fmt, p, rows, cols, x)
    err = assert_close(got, oracle.gemv(fmt, src, rows, cols, x), what=f"{fmt} {rows}x{cols} t{t}")
    # the stated arithmetic: binary16 weights (Q4_0 / Q8_0), x to ~2^-22, f32 sums
    tight = assert_close(got, _binary16_weights_ref(fmt, src, rows, cols, x), tol=2e-5,
                         what=f"{fmt} {rows}x{cols} t{t} against binary16 weights")
    print(f"{fmt} {rows}x{cols} t{t}: rel err vs oracle {err:.2e}, vs binary16 weights {tight:.2e}")


@pytest.mark.parametrize("fmt", FMTS)
def test_q_gemm_exact_case_bit_exact(qd, fmt):
    """Power-of-two scales and small integer x: d * q is exact in binary16, x's high parts
    exact and low parts zero, every product and partial sum exact in f32 -> bit-exact."""
    rows, cols, t = 300, 2048, 70
    src = qdsynth.weight_src(fmt, 32, "gmex", rows, cols).copy()
    if fmt in ("q4_0", "q8_0"):
        blk = src.reshape(rows, cols // 32, -1)
        blk[:, :, 0:2] = np.array([2.0 ** -3], np.float16).view(np.uint8)
    else:
        src[rows * cols:] = np.full(rows, 2.0 ** -5, np.float32).view(np.uint8)
    p = packed(qd, fmt, src, rows, cols)
    x = qdsynth.ints_i32(32, "gmxi", t * cols, -4, 4).reshape(t, cols).astype(np.float32)
    got = _gemm(qd, fmt, p, rows, cols, x)
    assert np.array_equal(got.astype(np.float64), oracle.gemv(fmt, src, rows, cols, x))


def _sampled_rows(rows, n=48, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 255, 256, rows - 1], rng.integers(0, rows, n)]))


def test_q_gemm_several_tiles_per_cta(qd):
    """10 row tiles x 48 token tiles = 480 tiles over at most 152 persistent CTAs: each CTA
    walks 3-4 tiles, reusing both accumulator sets; sampled rows, every token."""
    fmt, rows, cols, t = "q8_0", 2560, 576, 3072
    src, p = weights(qd, fmt, 33, "gmmany", rows, cols)
    x = qdsynth.activations(33, "gmmanyx", t, cols)
    got = _gemm(qd, fmt, p, rows, cols, x)
    for r in _sampled_rows(rows):
        want = oracle.gemv(fmt, src, rows, cols, x, int(r), 1)[:, 0]
        assert_close(got[:, r][None, :], want[None, :], what=f"row {r}")


@pytest.mark.parametrize("fmt,shape", [("q4_0", (14336, 4096)), ("q8_0", (4096, 11008)), ("i8", (8192, 2048))])
def test_q_gemm_full_size_sampled(qd, fmt, shape):
    """Full-size prefill shapes at t = 512 (the bench's launch), sampled rows, every token."""
    rows, cols = shape
    t = 512
    src, p = weights(qd, fmt, 34, f"gmfull{rows}x{cols}", rows, cols)
    x = qdsynth.activations(34, f"gmfullx{cols}", t, cols)
    got = _gemm(qd, fmt, p, rows, cols, x)
    rs = _sampled_rows(rows, 24)
    want = np.stack([oracle.gemv(fmt, src, rows, cols, x, int(r), 1)[:, 0] for r in rs], axis=1)
    assert_close(got[:, rs], want, what=f"{fmt} {rows}x{cols} t{t}")


def test_q_gemm_non_finite_rows(qd):
    rows, cols, t = 300, 512, 80
    src, p = weights(qd, "q4_0", 35, "gmnf", rows, cols)
    x = qdsynth.activations(35, "gmnfx", t, cols)
    x[3, 17] = np.nan
    x[70, 500] = np.inf
    got = _gemm(qd, "q4_0", p, rows, cols, x)
    for n in range(t):
        assert (not np.isfinite(got[n]).any()) if n in (3, 70) else np.isfinite(got[n]).all(), n


def test_q_gemm_matches_q_gemv_within_tolerance(qd):
    """The same 16 tokens through the decode product and the prefill product agree."""
    rows, cols, t = 1536, 576, 16
    src, p = weights(qd, "i8", 36, "gmgv", rows, cols)
    x = qdsynth.activations(36, "gmgvx", t, cols)
    got = _gemm(qd, "i8", p, rows, cols, x)
    y = torch.empty(t, rows, dtype=torch.float32, device="cuda")
    qd.q_gemv("i8", p, rows, cols, dev(x), y, t)
    torch.cuda.synchronize()
    assert_close(got, y.cpu().numpy(), tol=2e-5, what="gemm vs gemv")
