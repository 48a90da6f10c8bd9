"""GPU parity of the load-time per-row INT8 quantiser (qd_quantize_i8_rows through the C
ABI) against the oracle: codes and scales bit-exact (the f32 decisions are the same on
both sides), then the quantised matrix fed through qd_repack and qd_q_gemv."""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import assert_close, dev
from test_oracle_quant import bf16, random_bf16

pytestmark = pytest.mark.gpu


def gpu_quantize(qd, w_bits: np.ndarray, rows: int, cols: int):
    w = torch.from_numpy(np.ascontiguousarray(w_bits).view(np.int16)).cuda()
    out = torch.empty(qd.src_bytes("i8", rows, cols), dtype=torch.uint8, device="cuda")
    qd.quantize_i8_rows(w, rows, cols, out)
    torch.cuda.synchronize()
    raw = out.cpu().numpy()
    codes = raw[: rows * cols].view(np.int8).reshape(rows, cols)
    scales = raw[rows * cols: rows * cols + 4 * rows].view(np.float32)
    return codes, scales, out


def special_rows(cols: int) -> np.ndarray:
    """Rows that exercise the rule's corners: zeros, exact half-way codes (max 127 gives
    scale 1), a NaN, an infinity, the largest magnitude last, negative extremes, a row
    whose scale is subnormal (max |w| ~ 1e-37) and a row of subnormal bf16 values."""
    rows = np.zeros((8, cols), np.uint16)
    ties = np.zeros(cols, np.float32)
    ties[:8] = [127, 2.5, -2.5, 0.5, -0.5, -126.5, 1.5, 63.5]
    rows[1] = bf16(ties)
    rows[2] = bf16(np.ones(cols, np.float32))
    rows[2, 3] = 0x7FC0
    rows[3] = bf16(np.full(cols, -1.0, np.float32))
    rows[3, 1] = 0xFF80  # -inf
    ramp = ((np.arange(cols) % 256 - 128) / 8).astype(np.float32)  # exact in bf16
    rows[4] = bf16(ramp)
    rows[5] = bf16(-np.abs(ramp) - 1)
    tiny = (ramp * np.float32(2.0 ** -126)).astype(np.float32)  # |w| <= 16 * 2^-126: subnormal scale
    rows[6] = bf16(tiny)
    rows[7] = (np.arange(cols) % 120 + 1).astype(np.uint16)  # positive bf16 subnormals
    return rows


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (9, 128), (257, 2048), (40, 8192)])
def test_quantize_matches_oracle_bit_exact(qd, rows, cols):
    w = random_bf16(51, f"gq{rows}x{cols}", rows, cols)
    if rows >= 9:
        w[: 8] = special_rows(cols)
    q, s, _ = gpu_quantize(qd, w, rows, cols)
    oq, os_ = oracle.quantize_i8_rows(w, rows, cols)
    assert np.array_equal(q, oq)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))  # NaN scales included


@pytest.mark.parametrize("batch", [1, 16])
def test_quantized_matrix_feeds_the_int8_gemv(qd, batch):
    rows, cols = 512, 2048
    w = random_bf16(52, "gq.gemv", rows, cols)
    _, _, src = gpu_quantize(qd, w, rows, cols)
    packed = torch.empty(qd.packed_bytes("i8", rows, cols), dtype=torch.uint8, device="cuda")
    qd.repack("i8", src, rows, cols, packed)
    x = qdsynth.activations(52, "gq.x", batch, cols)
    y = torch.empty(batch, rows, device="cuda")
    qd.q_gemv("i8", packed, rows, cols, torch.from_numpy(x).cuda(), y, batch)
    torch.cuda.synchronize()
    ref = oracle.gemv("i8", src.cpu().numpy(), rows, cols, x)
    assert_close(y.cpu().numpy(), ref, tol=2e-5, what=f"quantised INT8 gemv b{batch}")
    # and the quantised matrix approximates the bf16 one: |q s - w| <= s / 2 per weight
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    oq, os_ = oracle.quantize_i8_rows(w, rows, cols)
    assert np.all(np.abs(oq * os_[:, None].astype(np.float64) - wf) <= os_[:, None] * (0.5 + 2e-5))


def test_quantize_full_1p7b_head_sampled_rows(qd):
    """The 1.7B head shape (49152 x 2048, 201 MB of bf16) in one launch; 64 sampled rows
    checked against the oracle bit-exactly."""
    rows, cols = 49152, 2048
    g = torch.Generator(device="cuda").manual_seed(53)
    wf = torch.randn(rows, cols, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty(qd.src_bytes("i8", rows, cols), dtype=torch.uint8, device="cuda")
    qd.quantize_i8_rows(wf.view(torch.int16), rows, cols, out)
    torch.cuda.synchronize()
    pick = np.random.default_rng(53).choice(rows, 64, replace=False)
    bits = wf.view(torch.int16)[torch.from_numpy(pick).cuda()].cpu().numpy().view(np.uint16)
    oq, os_ = oracle.quantize_i8_rows(bits, 64, cols)
    codes = out[: rows * cols].view(rows, cols)[torch.from_numpy(pick).cuda()].cpu().numpy().view(np.int8)
    scales = out[rows * cols:].view(torch.float32)[torch.from_numpy(pick).cuda()].cpu().numpy()
    assert np.array_equal(codes, oq) and np.array_equal(scales, os_)


def test_quantize_i4_rows_bit_exact(qd):
    """Per-row INT4 (s = max|w| / 7, codes rounded ties away, +-7): codes and scales bit-exact
    against the oracle, including a zero row, a non-finite row and rows whose quotients sit
    at the ties; the result feeds the INT4 q_gemv."""
    rows, cols = 70, 1024
    w = qdsynth.normal_f32(71, "i4q", rows * cols).reshape(rows, cols)
    w[3] = 0.0
    w[5, 17] = np.inf
    w[8] = (np.arange(cols) % 15 - 7) * 0.5  # multiples of s / 2: the ties
    wb = (w.view(np.uint32) >> 16).astype(np.uint16)
    out = torch.zeros(qd.src_bytes("i4", rows, cols), dtype=torch.uint8, device="cuda")
    qd.quantize_i4_rows(dev(wb.view(np.int16)), rows, cols, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    codes, scales = oracle.quantize_i4_rows(wb, rows, cols)
    assert np.array_equal(got[:rows * cols // 2], codes.reshape(-1))
    gs = got[rows * cols // 2:].view(np.float32)
    assert np.array_equal(np.isnan(gs), np.isnan(scales))
    assert np.array_equal(gs[~np.isnan(gs)].view(np.uint32), scales[~np.isnan(scales)].view(np.uint32))
