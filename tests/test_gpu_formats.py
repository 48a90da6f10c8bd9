"""GPU parity for the formats a Q4_K_M-class file mixes in (Q4_1, Q5_0, Q5_K, Q6_K, F16) and
per-row INT4
through the C ABI: the repack round trip and the dequantiser bit-exact against the oracle,
the embedding row bit-exact, q_gemv within 1e-3 of max |oracle| per output vector at batch
1-16 (several row tiles, ragged rows), and the 7B-like shapes at full size on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import assert_close, dev, packed, weights

pytestmark = pytest.mark.gpu

NEW = ["q4_1", "q5_0", "q5_k", "q6_k", "f16", "i4"]
SHAPES = {"q4_1": [(1, 32), (67, 1056), (130, 4128)], "q5_0": [(1, 32), (67, 1056), (33, 4128), (67, 1024), (33, 4160)],
          "q5_k": [(1, 256), (37, 2304), (19, 4352)], "q6_k": [(1, 256), (37, 2304), (19, 4352), (37, 2048), (19, 3584)],
          "f16": [(1, 32), (67, 1056), (41, 4128)], "i4": [(1, 32), (67, 1056), (41, 4128)]}


@pytest.mark.parametrize("fmt", NEW)
def test_repack_round_trip_bit_exact(qd, fmt):
    for rows, cols in SHAPES[fmt]:
        src = qdsynth.weight_src(fmt, 41, f"rt{rows}", rows, cols)
        p = packed(qd, fmt, src, rows, cols)
        back = torch.zeros(qd.src_bytes(fmt, rows, cols), dtype=torch.uint8, device="cuda")
        qd.unpack(fmt, p, rows, cols, back)
        torch.cuda.synchronize()
        assert np.array_equal(back.cpu().numpy(), src.reshape(-1).view(np.uint8)), (fmt, rows, cols)


@pytest.mark.parametrize("fmt", NEW)
def test_dequant_bit_exact(qd, fmt):
    for rows, cols in SHAPES[fmt]:
        src, p = weights(qd, fmt, 42, f"dq{rows}", rows, cols)
        out = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
        qd.dequant(fmt, p, rows, cols, out)
        want = oracle.dequant(fmt, src, rows, cols)
        assert np.array_equal(out.cpu().numpy().reshape(rows, cols).view(np.uint32), want.view(np.uint32)), fmt


@pytest.mark.parametrize("fmt", NEW)
def test_embed_bit_exact(qd, fmt):
    vocab, dim = 300, 512
    src, p = weights(qd, fmt, 43, "emb", vocab, dim)
    toks = np.array([0, 299, 17, 150], np.int32)
    x = torch.empty(4, dim, dtype=torch.float32, device="cuda")
    qd.embed(fmt, p, vocab, dim, dev(toks), 4, x)
    torch.cuda.synchronize()
    want = oracle.dequant(fmt, src, vocab, dim)[toks]
    assert np.array_equal(x.cpu().numpy().view(np.uint32), want.view(np.uint32))


def _gemv(qd, fmt, p, rows, cols, x):
    b = x.shape[0]
    y = torch.full((b, rows), float("nan"), dtype=torch.float32, device="cuda")
    qd.q_gemv(fmt, p, rows, cols, dev(x), y, b)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt", NEW)
@pytest.mark.parametrize("batch", [1, 3, 8, 16])
def test_q_gemv_parity(qd, fmt, batch):
    for rows, cols in SHAPES[fmt][1:]:
        src, p = weights(qd, fmt, 44, f"gv{rows}", rows, cols)
        x = qdsynth.activations(44, f"gvx{cols}", batch, cols)
        got = _gemv(qd, fmt, p, rows, cols, x)
        assert_close(got, oracle.gemv(fmt, src, rows, cols, x), what=f"{fmt} {rows}x{cols} b{batch}")


STREAMED = {"q6_k": [(37, 2048), (19, 3584), (300, 7168)],   # even super-block counts
            "q5_k": [(37, 2304), (19, 4352), (300, 7168)],
            "q5_0": [(67, 1024), (33, 4160), (300, 7168)]}     # even block counts


@pytest.mark.parametrize("fmt", ["q6_k", "q5_k", "q5_0"])
def test_q_gemv_streaming_integer_precision(qd, fmt):
    """Q6_K, Q5_K and Q5_0 on the streaming kernel's integer dot (Q6_K and Q5_0 as signed
    codes, Q5_K as Q4_K's unsigned codes with the fifth bit) against x's 24-bit planes: at
    batch 1, 2, 5 and 8, over full and short last steps, every row within 2e-5 of the
    oracle (the planes' bound), not just 1e-3."""
    for rows, cols in STREAMED[fmt]:
        src, p = weights(qd, fmt, 46, f"st{fmt}{rows}", rows, cols)
        for batch in (1, 2, 5, 8):
            x = qdsynth.activations(46, f"stx{cols}", batch, cols)
            got = _gemv(qd, fmt, p, rows, cols, x)
            assert_close(got, oracle.gemv(fmt, src, rows, cols, x), tol=2e-5, what=f"{fmt} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("fmt", NEW)
def test_q_gemv_full_size_sampled(qd, fmt):
    rows, cols = 4096, 4096
    src, p = weights(qd, fmt, 45, "gvfull", rows, cols)
    x = qdsynth.activations(45, "gvfullx", 1, cols)
    got = _gemv(qd, fmt, p, rows, cols, x)
    rng = np.random.default_rng(1)
    rs = np.unique(np.concatenate([[0, rows - 1], rng.integers(0, rows, 48)]))
    want = np.stack([oracle.gemv(fmt, src, rows, cols, x, int(r), 1)[0, 0] for r in rs])
    assert_close(got[:, rs], want[None, :], what=f"{fmt} full")
