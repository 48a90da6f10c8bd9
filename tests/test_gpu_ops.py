"""GPU parity of the decode-step operations (RMSNorm, RoPE, KV append, attention, SwiGLU,
argmax, embedding) against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import assert_close, dev, weights

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n,batch", [(576, 1), (576, 3), (2048, 16), (1, 1), (4097, 2)])
def test_rmsnorm(qd, n, batch):
    x = qdsynth.activations(1, f"x{n}", batch, n)
    g = qdsynth.norm_gains(1, f"g{n}", n)
    out = torch.empty(batch, n, dtype=torch.float32, device="cuda")
    qd.rmsnorm(dev(x), dev(g), out, n, batch, 1e-5)
    assert_close(out.cpu().numpy(), oracle.rmsnorm(x, g, 1e-5), tol=1e-5, what="rmsnorm")


def _table(theta, hd, ctx):
    t = np.empty((ctx, hd // 2, 2), np.float32)
    import quantized_decode_gemv_gb300 as q

    q.rope_table(theta, hd, ctx, t.ctypes.data)
    return t


@pytest.mark.parametrize("pairing", ["adjacent", "half"])
def test_rope(qd, pairing):
    H, hd, ctx, batch, stride = 12, 64, 4096, 4, 960
    tab = dev(_table(1e5, hd, ctx))
    v = qdsynth.activations(2, "v", batch, stride)
    pos = np.array([0, 1, 777, 4095], np.int32)
    vd = dev(v)
    qd.rope(vd, H, hd, stride, dev(pos), pairing, tab, ctx, batch)
    got = vd.cpu().numpy()
    for b in range(batch):
        want = oracle.rope(v[b, :H * hd], H, hd, int(pos[b]), pairing, 1e5)
        assert_close(got[b, :H * hd], want, tol=1e-5, what=f"rope b{b}")
        assert np.array_equal(got[b, H * hd:], v[b, H * hd:])  # beyond the heads: untouched
    # a position outside [0, max_ctx) leaves the row unchanged
    vd = dev(v)
    qd.rope(vd, H, hd, stride, dev(np.array([4096, -1, 0, 0], np.int32)), pairing, tab, ctx, batch)
    assert np.array_equal(vd.cpu().numpy()[:2], v[:2])


def test_kv_append_bit_exact(qd):
    hk, hd, ctx, batch, stride = 3, 64, 32, 3, 960
    src = qdsynth.activations(3, "kv", batch, stride)
    kc = torch.zeros(batch, hk, ctx, hd, device="cuda")
    vc = torch.zeros_like(kc)
    pos = np.array([0, 31, 5], np.int32)
    s = dev(src)
    qd.kv_append(s[:, 576:], s[:, 768:], stride, kc, vc, hk, hd, dev(pos), ctx, batch)
    k, v = kc.cpu().numpy(), vc.cpu().numpy()
    for b in range(batch):
        assert np.array_equal(k[b, :, pos[b]], src[b, 576:768].reshape(hk, hd))
        assert np.array_equal(v[b, :, pos[b]], src[b, 768:960].reshape(hk, hd))
        mask = np.ones(ctx, bool)
        mask[pos[b]] = False
        assert np.all(k[b][:, mask] == 0) and np.all(v[b][:, mask] == 0)


@pytest.mark.parametrize("hq,hk,ctx,positions", [(9, 3, 256, [0, 1, 63, 64, 200, 255]),
                                                 (32, 32, 4096, [0, 127, 128, 2500, 4095]),
                                                 (8, 1, 300, [299, 0, 150]), (4, 2, 70, [69])])
def test_gqa_decode_attention(qd, hq, hk, ctx, positions):
    hd = 64
    batch = len(positions)
    kc = qdsynth.normal_f32(4, "k", batch * hk * ctx * hd).reshape(batch, hk, ctx, hd)
    vc = qdsynth.normal_f32(4, "v", batch * hk * ctx * hd).reshape(batch, hk, ctx, hd)
    qs = hq * hd + 32  # a row stride larger than the heads, as inside the fused qkv buffer
    q = qdsynth.activations(4, "q", batch, qs)
    ws_bytes = qd.gqa_decode_attn_workspace(hq, hd, ctx, batch)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((batch, hq * hd), float("nan"), device="cuda")
    pos = np.array(positions, np.int32)
    qd.gqa_decode_attn(dev(q), qs, dev(kc), dev(vc), out, hq, hk, hd, dev(pos), ctx, batch, ws, ws_bytes)
    got = out.cpu().numpy()
    for b, p in enumerate(positions):
        want = oracle.attention(q[b, :hq * hd], kc[b], vc[b], hq, hk, hd, p + 1, ctx)
        assert_close(got[b], want, tol=1e-5, what=f"attn b{b} pos{p}")
        if p == 0:  # a single position returns its value rows
            assert np.allclose(got[b].reshape(hq, hd), np.repeat(vc[b, :, 0], hq // hk, axis=0), rtol=0, atol=1e-6)


def test_attention_out_of_range_position_gives_zeros(qd):
    hq, hk, hd, ctx = 4, 2, 64, 16
    kc = torch.randn(1, hk, ctx, hd, device="cuda")
    q = torch.randn(1, hq * hd, device="cuda")
    ws_bytes = qd.gqa_decode_attn_workspace(hq, hd, ctx, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((1, hq * hd), 5.0, device="cuda")
    qd.gqa_decode_attn(q, hq * hd, kc, kc, out, hq, hk, hd, dev(np.array([16], np.int32)), ctx, 1, ws, ws_bytes)
    assert torch.all(out == 0).item()


def test_swiglu(qd):
    n, batch = 1536, 3
    g = qdsynth.activations(5, "g", batch, n) * np.float32(4.0)
    u = qdsynth.activations(5, "u", batch, n)
    out = torch.empty(batch, n, device="cuda")
    qd.swiglu(dev(g), dev(u), out, n, batch)
    want = oracle.swiglu(g.reshape(-1), u.reshape(-1)).reshape(batch, n)
    assert_close(out.cpu().numpy(), want, tol=1e-5, what="swiglu")


def test_argmax_bit_exact_and_ties(qd):
    n = 49152
    logits = qdsynth.activations(6, "l", 4, n)
    logits[1, 100] = logits[1, 40000] = logits[1].max() + 1.0  # tie: first index wins
    logits[2, :] = 0.5                                         # all equal: index 0
    logits[3, n - 1] = 50.0                                    # last element
    out = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    qd.argmax(dev(logits), n, 4, out)
    got = out.cpu().numpy()
    want = [oracle.argmax(logits[b]) for b in range(4)]
    assert list(got) == want
    assert want[1] == 100 and want[2] == 0 and want[3] == n - 1


@pytest.mark.parametrize("fmt,dim", [("q8_0", 576), ("i8", 2048), ("q4_0", 576), ("q4_k", 512)])
def test_embedding_bit_exact(qd, fmt, dim):
    vocab = 1000
    src, p = weights(qd, fmt, 7, "emb", vocab, dim)
    toks = np.array([0, 999, 17, 500], np.int32)
    x = torch.empty(4, dim, device="cuda")
    qd.embed(fmt, p, vocab, dim, dev(toks), 4, x)
    got = x.cpu().numpy()
    for b, t in enumerate(toks):
        want = oracle.dequant(fmt, src, vocab, dim, row0=int(t), nrows=1)[0]
        assert np.array_equal(got[b].view(np.uint32), want.view(np.uint32))
