"""GPU parity of the ggml-exact activation path (qd_quantize_q8, qd_q_gemv_q8) against the
oracle through the C ABI: codes, d and s bit-exact (seeded rows, exact-d rows with ties,
zero and non-finite blocks); the integer product within 1e-5 of max |oracle| per output
vector (the integer sums are exact, only the f32 scaled sum differs from the double one),
at batch 1-16 over several row tiles and at the 7B-like shape on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import assert_close, dev, weights

pytestmark = pytest.mark.gpu


def _quantize(qd, x, with_sum):
    batch, cols = x.shape
    nbytes = qd.q8_bytes(batch, cols, with_sum)
    out = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    qd.quantize_q8(dev(x), batch, cols, out, with_sum)
    torch.cuda.synchronize()
    return out


def _split(buf, batch, cols, with_sum):
    b = buf.cpu().numpy()
    nb = cols // 32
    q = b[:batch * cols].view(np.int8).reshape(batch, cols)
    d_off = (batch * cols + 15) // 16 * 16
    d = b[d_off:d_off + 2 * batch * nb].view(np.float16).reshape(batch, nb)
    s = None
    if with_sum:
        s_off = d_off + (2 * batch * nb + 15) // 16 * 16
        s = b[s_off:s_off + 2 * batch * nb].view(np.float16).reshape(batch, nb)
    return q, d, s


def _same_f16(gpu_f16, ora_f32):
    want = ora_f32.astype(np.float16)
    return np.array_equal(gpu_f16.view(np.uint16)[~np.isnan(want)], want.view(np.uint16)[~np.isnan(want)]) and \
        np.array_equal(np.isnan(gpu_f16), np.isnan(want))


@pytest.mark.parametrize("with_sum", [False, True])
def test_quantize_bit_exact(qd, with_sum):
    batch, cols = 5, 4096
    x = qdsynth.activations(51, "q8x", batch, cols)
    x[1, :32] = 0.0                                   # zero block
    x[2, 40] = np.nan                                 # non-finite block
    x[3, 64:96] = np.arange(32, dtype=np.float32) - 15.5  # values on ties of the rounding
    x[4, :32] = 127.0 * (np.arange(32) % 3 - 1) + 0.5 * (np.arange(32) % 2)  # d = 1, half-way codes
    q, d, s = _split(_quantize(qd, x, with_sum), batch, cols, with_sum)
    oq, od, os_ = oracle.quantize_q8(x, with_sum)
    assert np.array_equal(q, oq)
    assert _same_f16(d, od)
    if with_sum:
        assert _same_f16(s, os_)


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0", "q4_1"])
@pytest.mark.parametrize("batch", [1, 3, 8, 16])
def test_q_gemv_q8_parity(qd, fmt, batch):
    with_sum = fmt == "q4_1"
    for rows, cols in ((67, 1056), (300, 4096)):
        src, p = weights(qd, fmt, 52, f"q8w{rows}", rows, cols)
        x = qdsynth.activations(52, f"q8gx{cols}", batch, cols)
        xq = _quantize(qd, x, with_sum)
        y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
        qd.q_gemv_q8(fmt, p, rows, cols, xq, y, batch)
        torch.cuda.synchronize()
        oq, od, os_ = oracle.quantize_q8(x, with_sum)
        want = oracle.gemv_q8act(fmt, src, rows, cols, oq, od, os_)
        assert_close(y.cpu().numpy(), want, tol=1e-5, what=f"{fmt} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("fmt", ["q4_0", "q8_0"])
def test_q_gemv_q8_full_size_sampled(qd, fmt):
    rows, cols, batch = 14336, 4096, 4
    src, p = weights(qd, fmt, 53, "q8full", rows, cols)
    x = qdsynth.activations(53, "q8fullx", batch, cols)
    xq = _quantize(qd, x, False)
    y = torch.empty(batch, rows, dtype=torch.float32, device="cuda")
    qd.q_gemv_q8(fmt, p, rows, cols, xq, y, batch)
    torch.cuda.synchronize()
    oq, od, _ = oracle.quantize_q8(x)
    rng = np.random.default_rng(2)
    rs = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, 40)]))
    want = np.stack([oracle.gemv_q8act(fmt, src, rows, cols, oq, od, None, int(r), 1)[:, 0] for r in rs], axis=1)
    assert_close(y.cpu().numpy()[:, rs], want, tol=1e-5, what=f"{fmt} full")


def test_q8_product_close_to_f32_product(qd):
    """The ggml-exact product differs from the f32-activation product by the activation
    quantisation (about 1/254 of each block's largest |x| per value): within 1e-2 of max |y|."""
    rows, cols = 576, 1536
    src, p = weights(qd, "q4_0", 54, "q8vs", rows, cols)
    x = qdsynth.activations(54, "q8vsx", 1, cols)
    xq = _quantize(qd, x, False)
    y = torch.empty(1, rows, dtype=torch.float32, device="cuda")
    qd.q_gemv_q8("q4_0", p, rows, cols, xq, y, 1)
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), oracle.gemv("q4_0", src, rows, cols, x), tol=1e-2, what="q8 vs f32")
