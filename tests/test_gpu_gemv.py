"""GPU parity of the repacker, the dequantiser and the q_gemv family against the oracle,
through the C ABI.  Bit-exact where the result is integer/byte work or exactly representable;
within 1e-3 of max |oracle| per output vector otherwise."""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import TOL, assert_close, dev, packed, weights

pytestmark = pytest.mark.gpu

FMTS = ["q4_0", "q8_0", "q4_k", "i8"]
SMALL = {"q4_0": [(1, 32), (7, 96), (67, 1056), (130, 4128)], "q8_0": [(1, 32), (9, 160), (67, 1056), (33, 4128)],
         "q4_k": [(1, 256), (5, 512), (37, 2304), (19, 4352)], "i8": [(1, 16), (5, 48), (67, 1040), (41, 4112)]}


@pytest.mark.parametrize("fmt", FMTS)
def test_repack_unpack_round_trip_bit_exact(qd, fmt):
    for rows, cols in SMALL[fmt]:
        src = qdsynth.weight_src(fmt, 1, f"rt{rows}", rows, cols)
        p = packed(qd, fmt, src, rows, cols)
        back = torch.zeros(qd.src_bytes(fmt, rows, cols), dtype=torch.uint8, device="cuda")
        qd.unpack(fmt, p, rows, cols, back)
        torch.cuda.synchronize()
        assert np.array_equal(back.cpu().numpy(), src.reshape(-1).view(np.uint8)), (rows, cols)


@pytest.mark.parametrize("fmt", FMTS)
def test_dequant_block_values_bit_exact(qd, fmt):
    for rows, cols in SMALL[fmt]:
        src, p = weights(qd, fmt, 2, f"dq{rows}", rows, cols)
        out = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
        qd.dequant(fmt, p, rows, cols, out)
        want = oracle.dequant(fmt, src, rows, cols)
        assert np.array_equal(out.cpu().numpy().reshape(rows, cols).view(np.uint32), want.view(np.uint32))


def test_hand_worked_q4_0_blocks_on_gpu(qd):
    from test_oracle_pins import _hand_q4_0

    for blk, vals, total in _hand_q4_0():
        p = packed(qd, "q4_0", blk, 1, 32)
        out = torch.empty(32, dtype=torch.float32, device="cuda")
        qd.dequant("q4_0", p, 1, 32, out)
        assert np.array_equal(out.cpu().numpy().astype(np.float64), vals)
        y = torch.empty(1, dtype=torch.float32, device="cuda")
        qd.q_gemv("q4_0", p, 1, 32, torch.ones(32, device="cuda"), y, 1)
        assert y.item() == total


def test_f16_bf16_all_patterns_bit_exact(qd):
    bits = np.arange(65536, dtype=np.uint16)
    inp = dev(bits.view(np.int16))
    out = torch.empty(65536, dtype=torch.float32, device="cuda")
    qd.f16_to_f32(inp, out)
    want = oracle.f16_to_f32_array(bits)
    got = out.cpu().numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got.view(np.uint32)[~nan], want.view(np.uint32)[~nan])
    qd.bf16_to_f32(inp, out)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), oracle.bf16_to_f32_array(bits).view(np.uint32))


def _gemv(qd, fmt, p, rows, cols, x):
    batch = x.shape[0]
    y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
    qd.q_gemv(fmt, p, rows, cols, dev(x), y, batch)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8, 13, 16])
def test_q_gemv_small_ragged_shapes(qd, fmt, batch):
    for rows, cols in SMALL[fmt]:
        src, p = weights(qd, fmt, 3, f"g{rows}x{cols}", rows, cols)
        x = qdsynth.activations(3, f"x{cols}", batch, cols)
        got = _gemv(qd, fmt, p, rows, cols, x)
        assert_close(got, oracle.gemv(fmt, src, rows, cols, x), what=f"{fmt} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "i8", "q4_k"])
@pytest.mark.parametrize("batch", [3, 8])
def test_q_gemv_exact_case_bit_exact(qd, fmt, batch):
    """Power-of-two scales and integer x: every partial sum is exact in f32, so the GPU must
    equal the oracle exactly whatever its summation order (batch 3 and 8 take the tensor-core
    kernel for Q4_0, Q8_0 and INT8 rows)."""
    rows, cols = 70, 2048
    src = qdsynth.weight_src(fmt, 4, "ex", rows, cols).copy()
    if fmt in ("q4_0", "q8_0"):
        blk = src.reshape(rows, cols // 32, -1)
        blk[:, :, 0:2] = np.array([2.0 ** -3], np.float16).view(np.uint8)
    elif fmt == "q4_k":
        blk = src.reshape(rows, cols // 256, 144)
        blk[:, :, 0:2] = np.array([2.0 ** -3], np.float16).view(np.uint8)
        blk[:, :, 2:4] = np.array([2.0 ** -4], np.float16).view(np.uint8)
    else:
        src[rows * cols:] = np.full(rows, 2.0 ** -3, np.float32).view(np.uint8)
    p = packed(qd, fmt, src, rows, cols)
    x = qdsynth.ints_i32(4, "xi", batch * cols, -4, 4).reshape(batch, cols).astype(np.float32)
    got = _gemv(qd, fmt, p, rows, cols, x)
    want = oracle.gemv(fmt, src, rows, cols, x)
    assert np.array_equal(got.astype(np.float64), want)


def test_q_gemv_config1_full(qd):
    """Q4_0 576 x 1536, batch 1, seed 0 (the single-GEMV configuration), every output."""
    rows, cols = 576, 1536
    src, p = weights(qd, "q4_0", 0, "W", rows, cols)
    x = qdsynth.activations(0, "x", 1, cols)
    got = _gemv(qd, "q4_0", p, rows, cols, x)
    err = assert_close(got, oracle.gemv("q4_0", src, rows, cols, x), what="C1")
    print(f"C1 max rel err {err:.2e}")


SWEEP = [(4096, 4096), (11008, 4096), (4096, 11008), (14336, 4096)]


def _sampled_rows(rows, n=64, seed=0):
    rng = np.random.default_rng(seed)
    r = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, n)]))
    return r


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
@pytest.mark.parametrize("shape", SWEEP)
def test_q_gemv_7b_sweep_sampled(qd, fmt, shape):
    """The 7B-like sweep at full size, batch 1/2/4/8, on sampled output rows."""
    rows, cols = shape
    src, p = weights(qd, fmt, 0, f"sweep.{fmt}.{rows}x{cols}", rows, cols)
    rs = _sampled_rows(rows)
    for batch in (1, 2, 4, 8):
        x = qdsynth.activations(0, f"sweep.x{cols}", batch, cols)
        got = _gemv(qd, fmt, p, rows, cols, x)
        assert np.all(np.isfinite(got))
        want = np.concatenate([oracle.gemv(fmt, src, rows, cols, x, row0=int(r), nrows=1) for r in rs], axis=1)
        assert_close(got[:, rs], want, what=f"{fmt} {shape} b{batch}")


@pytest.mark.parametrize("shape", [(2048, 2048), (5632, 2048), (2048, 5632), (32000, 2048)])
def test_q_gemv_q4k_tinyllama_sampled(qd, shape):
    rows, cols = shape
    src, p = weights(qd, "q4_k", 0, f"tl.{rows}x{cols}", rows, cols)
    x = qdsynth.activations(0, f"tl.x{cols}", 1, cols)
    got = _gemv(qd, "q4_k", p, rows, cols, x)
    rs = _sampled_rows(rows)
    want = np.concatenate([oracle.gemv("q4_k", src, rows, cols, x, row0=int(r), nrows=1) for r in rs], axis=1)
    assert_close(got[:, rs], want, what=f"q4_k {shape}")


@pytest.mark.parametrize("shape", [(6144, 2048), (2048, 2048), (16384, 2048), (2048, 8192), (49152, 2048)])
@pytest.mark.parametrize("batch", [1, 16])
def test_q_gemv_i8_1p7b_sampled(qd, shape, batch):
    rows, cols = shape
    src, p = weights(qd, "i8", 0, f"i8.{rows}x{cols}", rows, cols)
    x = qdsynth.activations(0, f"i8.x{cols}", batch, cols)
    got = _gemv(qd, "i8", p, rows, cols, x)
    rs = _sampled_rows(rows, 32)
    want = np.concatenate([oracle.gemv("i8", src, rows, cols, x, row0=int(r), nrows=1) for r in rs], axis=1)
    assert_close(got[:, rs], want, what=f"i8 {shape} b{batch}")


def test_q_gemv_is_deterministic(qd):
    rows, cols = 4096, 4096
    src, p = weights(qd, "q4_0", 5, "det", rows, cols)
    x = qdsynth.activations(5, "xd", 4, cols)
    a = _gemv(qd, "q4_0", p, rows, cols, x)
    b = _gemv(qd, "q4_0", p, rows, cols, x)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt,rows,cols,batch", [("q4_0", 1024, 3072, 2), ("q4_0", 2048, 8192, 2),
                                                 ("q8_0", 2048, 8192, 1), ("i8", 2048, 8192, 1), ("i8", 2048, 8192, 2),
                                                 ("q4_k", 1024, 4096, 2), ("q8_0", 1042, 4160, 2)])
def test_q_gemv_split_k_tall_thin(qd, fmt, rows, cols, batch):
    """Tall-and-thin products (1024 rows or more, at least twice as many columns) at batch
    2, or with 8-bit weights, split their columns over a cluster of two CTAs whose partial
    row sums meet in the first one and are added in CTA order: every row against the
    oracle, and two runs give the same bits (1042x4160: ragged row groups and an odd
    number of 32-unit steps)."""
    src, p = weights(qd, fmt, 15, f"sk.{fmt}.{rows}x{cols}", rows, cols)
    x = qdsynth.activations(15, f"sk.x{cols}", batch, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} {rows}x{cols} b{batch}")
    again = _gemv(qd, fmt, p, rows, cols, x)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch", [1, 2, 8])
def test_q_gemv_activation_planes_precision(qd, fmt, batch):
    """The streaming kernel holds x as 24-bit integers with a power-of-two scale per
    32-element unit; its error stays near f32 rounding, far inside the 1e-3 bound."""
    rows, cols = 96, 4096
    src, p = weights(qd, fmt, 5, "prec", rows, cols)
    x = qdsynth.activations(5, "xprec", batch, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} b{batch}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("batch", [2, 5])
def test_q_gemv_non_finite_x_propagates(qd, fmt, batch):
    """A non-finite x value makes its batch row's outputs non-finite; the other rows stay
    finite and correct."""
    rows, cols = 40, 512
    src, p = weights(qd, fmt, 6, "nf", rows, cols)
    x = qdsynth.activations(6, "xnf", batch, cols)
    x[0, 37] = np.inf
    x[1, 300] = np.nan
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert not np.isfinite(got[:2]).any()
    if batch > 2:
        assert_close(got[2:], oracle.gemv(fmt, src, rows, cols, x[2:]), what=f"{fmt} finite rows")


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "i8"])
@pytest.mark.parametrize("batch", [3, 4, 6, 8, 9, 13, 16])
def test_q_gemv_tensor_core_batches_full(qd, fmt, batch):
    """Batch 3-16 on the tensor-core kernel: 16-row tiles with a ragged last tile (rows 1000
    = 62 tiles + 8), every output row, the 2e-5 bound of the integer planes."""
    rows, cols = 1000, 1536
    src, p = weights(qd, fmt, 12, f"tcb.{fmt}", rows, cols)
    x = qdsynth.activations(12, "tcb.x", batch, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} b{batch}")


@pytest.mark.parametrize("fmt,cols", [("q4_0", 1600), ("q8_0", 1600), ("i8", 1504)])
@pytest.mark.parametrize("batch", [3, 7, 11])
def test_q_gemv_tensor_core_partial_stage(qd, fmt, cols, batch):
    """Rows whose last 256-column stage is partial (1600 = 6 stages + 2 units; INT8 1504 =
    5 stages + 7 units, an odd count): the stage loop's run-time tail and the x scale of a
    short stage, every output row."""
    rows = 1000
    src, p = weights(qd, fmt, 13, f"tcp.{fmt}", rows, cols)
    x = qdsynth.activations(13, "tcp.x", batch, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} {cols} b{batch}")


@pytest.mark.parametrize("fmt,cols,batch", [(f, c, b) for f, c in [("q4_0", 11008), ("q8_0", 11008), ("i8", 11040)]
                                            for b in (5, 8, 16)]
                         + [("q4_0", 8192, 16), ("i8", 8192, 9), ("q8_0", 8192, 12), ("i8", 8192, 16)])
def test_q_gemv_tensor_core_column_split(qd, fmt, cols, batch):
    """x rows too wide for the shared memory beside the weight ring (11008 columns at batch
    5 or 8: over 220 KB of x) and few enough tiles for one per warp group: the columns
    split over a cluster's CTAs (whole 256-column x groups; INT8 11040 = 345 units leaves
    the last CTA a partial group), the first CTA adding the others' tile sums in CTA
    order.  8192 columns at batch 9-16: one split launch with two blocks of 8 columns
    (one buffer of per-warp partial sums: each warp group takes a single tile).
    Batch 16 at 11008 columns runs two passes of 8 rows, each split (INT8: the tcgen05
    kernel).  Every output row against the oracle, and two runs give the same bits."""
    rows = 300
    src, p = weights(qd, fmt, 15, f"tcs.{fmt}", rows, cols)
    x = qdsynth.activations(15, "tcs.x", batch, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} {cols} b{batch}")
    again = _gemv(qd, fmt, p, rows, cols, x)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))


@pytest.mark.parametrize("fmt,cols,batch", [("q4_0", 11008, 5), ("q4_0", 11008, 8), ("q8_0", 8192, 8),
                                            ("i8", 11040, 8)])
def test_q_gemv_tensor_core_column_ranges(qd, fmt, cols, batch):
    """x rows too wide for the shared memory and more tiles than a split grid gives its
    warp groups (12288 rows = 768 tiles) run as consecutive launches over column ranges,
    the first storing and the rest adding; INT8 11040 = 345 units leaves an odd, partial
    last range.  Every output row against the oracle, and two runs give the same bits."""
    rows = 12288
    src, p = weights(qd, fmt, 14, f"tcr.{fmt}", rows, cols)
    x = qdsynth.activations(14, "tcr.x", batch, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} {cols} b{batch}")
    again = _gemv(qd, fmt, p, rows, cols, x)
    assert np.array_equal(got.view(np.uint32), again.view(np.uint32))


def test_q_gemv_overlap_chain_matches_plain_launches(qd):
    """QD_GEMV_OVERLAP (weights streamed while the previous kernel finishes) must not change
    any result: a chain y1 = W1 x, y2 = W2 y1, y3 = W3 y2 gives the same bits either way."""
    shapes = [("q4_0", 576, 1536), ("q8_0", 1536, 576), ("q4_k", 256, 1536)]
    ws = [weights(qd, f, 8, f"ov{i}", r, c)[1] for i, (f, r, c) in enumerate(shapes)]
    x = dev(qdsynth.activations(8, "xov", 2, 1536))
    outs = []
    for flags in (qd.GEMV_OVERLAP, 0):
        ys = [torch.empty(2, r, device="cuda") for (_, r, _) in shapes]
        src = x
        for (f, r, c), w, y in zip(shapes, ws, ys):
            qd.q_gemv_ex(f, w, r, c, src, y, 2, flags)
            src = y
        torch.cuda.synchronize()
        outs.append([y.cpu().numpy() for y in ys])
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# Batch 9-16 per-row INT8 runs on the tensor cores (tcgen05, f16 hi/lo split of x, split-K
# over a cluster); shapes chosen to hit ragged row tiles and cluster sizes 1-8.
TC_SHAPES = [(1, 128), (129, 256), (200, 2048), (300, 1024), (2048, 2048), (640, 8192)]


@pytest.mark.parametrize("batch", [9, 13, 16])
def test_q_gemv_int8_tensor_core_batches(qd, batch):
    for rows, cols in TC_SHAPES:
        src, p = weights(qd, "i8", 11, f"tc{rows}x{cols}", rows, cols)
        x = qdsynth.activations(11, f"xtc{cols}", batch, cols)
        got = _gemv(qd, "i8", p, rows, cols, x)
        assert_close(got, oracle.gemv("i8", src, rows, cols, x), tol=2e-5, what=f"i8 tc {rows}x{cols} b{batch}")


def test_q_gemv_int8_tensor_core_exact_case(qd):
    """Power-of-two row scales and small integer x: the f16 high parts are exact, the low parts
    zero, every product and partial sum an integer below 2^24 -> bit-exact."""
    rows, cols, batch = 260, 2048, 16
    src = qdsynth.weight_src("i8", 12, "tcex", rows, cols).copy()
    src[rows * cols:] = np.full(rows, 2.0 ** -5, np.float32).view(np.uint8)
    p = packed(qd, "i8", src, rows, cols)
    x = qdsynth.ints_i32(12, "tcxi", batch * cols, -3, 3).reshape(batch, cols).astype(np.float32)
    got = _gemv(qd, "i8", p, rows, cols, x)
    assert np.array_equal(got.astype(np.float64), oracle.gemv("i8", src, rows, cols, x))


def test_q_gemv_int8_tensor_core_non_finite(qd):
    rows, cols, batch = 130, 1024, 12
    src, p = weights(qd, "i8", 13, "tcnf", rows, cols)
    x = qdsynth.activations(13, "xtcnf", batch, cols)
    x[3, 17] = np.nan
    x[7, 900] = np.inf
    got = _gemv(qd, "i8", p, rows, cols, x)
    bad = {3, 7}
    for b in range(batch):
        assert (not np.isfinite(got[b]).any()) if b in bad else np.isfinite(got[b]).all(), b
