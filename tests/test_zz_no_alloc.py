"""The allocation-free attention entry point.

Some callers of this library cannot allocate device memory for a workspace: a serving
loop that must never call cudaMalloc (it can synchronise the device), or code running
under a fixed memory budget that another allocator already owns.  For them
qd_gqa_decode_attn_noalloc keeps its partial results in a fixed device array inside the
library.  This test calls it through the C ABI twice in a row, with different inputs, and
checks each result against qd_gqa_decode_attn with a caller-provided workspace and against
the oracle's attention, within the tolerance the other parity tests use; it also runs a
request just under the array's size limit and checks that one just over it is refused.  The
file sorts last so that a run stopping at the first failure has already run every other
test.
"""
import numpy as np
import pytest
import torch

import oracle
import qdsynth
from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu


SCRATCH_BYTES = 8 << 20  # the fixed array's size, as qdecode.h states it


def _host_case(seed, hq, hk, ctx, positions):
    hd = 64
    batch = len(positions)
    kc = qdsynth.normal_f32(seed, "na.k", batch * hk * ctx * hd).reshape(batch, hk, ctx, hd)
    vc = qdsynth.normal_f32(seed, "na.v", batch * hk * ctx * hd).reshape(batch, hk, ctx, hd)
    q = qdsynth.activations(seed, "na.q", batch, hq * hd)
    return q, kc, vc


def _case(seed, hq, hk, ctx, positions):
    q, kc, vc = _host_case(seed, hq, hk, ctx, positions)
    return dev(q), dev(kc), dev(vc), dev(np.array(positions, np.int32))


def _check_oracle(got, seed, hq, hk, ctx, positions, seqs):
    """The allocation-free result against the oracle's attention for the listed sequences."""
    q, kc, vc = _host_case(seed, hq, hk, ctx, positions)
    for b in seqs:
        ref = oracle.attention(q[b], kc[b], vc[b], hq, hk, 64, positions[b] + 1, ctx)
        assert_close(got[b].reshape(hq, 64), ref.reshape(hq, 64), what=f"noalloc vs oracle seq {b}")


def test_noalloc_attention_matches_workspace_attention_twice(qd):
    hq, hk, hd, ctx = 32, 32, 64, 4096
    for seed, positions in ((1, [4095, 17, 2048]), (2, [0, 1000, 4095])):
        q, kc, vc, pos = _case(seed, hq, hk, ctx, positions)
        batch = len(positions)
        ws_bytes = qd.gqa_decode_attn_workspace(hq, hd, ctx, batch)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        want = torch.empty(batch, hq * hd, device="cuda")
        qd.gqa_decode_attn(q, hq * hd, kc, vc, want, hq, hk, hd, pos, ctx, batch, ws, ws_bytes)
        got = torch.full((batch, hq * hd), float("nan"), device="cuda")
        qd.gqa_decode_attn_noalloc(q, hq * hd, kc, vc, got, hq, hk, hd, pos, ctx, batch)
        torch.cuda.synchronize()
        g = got.cpu().numpy()
        assert_close(g, want.cpu().numpy(), what=f"noalloc call seed {seed}")
        _check_oracle(g, seed, hq, hk, ctx, positions, range(batch))


def test_noalloc_attention_gqa_groups(qd):
    hq, hk, hd, ctx = 9, 3, 64, 256
    q, kc, vc, pos = _case(3, hq, hk, ctx, [255, 0, 100, 64])
    ws_bytes = qd.gqa_decode_attn_workspace(hq, hd, ctx, 4)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    want = torch.empty(4, hq * hd, device="cuda")
    got = torch.empty(4, hq * hd, device="cuda")
    qd.gqa_decode_attn(q, hq * hd, kc, vc, want, hq, hk, hd, pos, ctx, 4, ws, ws_bytes)
    qd.gqa_decode_attn_noalloc(q, hq * hd, kc, vc, got, hq, hk, hd, pos, ctx, 4)
    torch.cuda.synchronize()
    g = got.cpu().numpy()
    assert_close(g, want.cpu().numpy(), what="noalloc gqa")
    _check_oracle(g, 3, hq, hk, ctx, [255, 0, 100, 64], range(4))


def _near_cap(hq, batch):
    """The largest context (in steps of 64 from 7680) whose workspace fits the array, and
    the next one, which does not."""
    import quantized_decode_gemv_gb300 as qd

    ctx = 7680
    assert qd.gqa_decode_attn_workspace(hq, 64, ctx, batch) <= SCRATCH_BYTES
    while qd.gqa_decode_attn_workspace(hq, 64, ctx + 64, batch) <= SCRATCH_BYTES:
        ctx += 64
    return ctx, ctx + 64


def test_noalloc_attention_just_under_the_size_limit(qd):
    """32 heads, batch 16, at the largest context whose partials still fit the array (over
    96 % of it): the last partial slots sit at the array's end, so a layout or offset
    mistake there would write past it or read garbage; checked against the workspace entry
    point for every sequence and against the oracle for three."""
    hq, hk, hd, batch = 32, 4, 64, 16
    ctx, _ = _near_cap(hq, batch)
    assert qd.gqa_decode_attn_workspace(hq, hd, ctx, batch) > 0.96 * SCRATCH_BYTES
    positions = [ctx - 1 - 37 * b for b in range(batch)]
    q, kc, vc, pos = _case(4, hq, hk, ctx, positions)
    ws_bytes = qd.gqa_decode_attn_workspace(hq, hd, ctx, batch)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    want = torch.empty(batch, hq * hd, device="cuda")
    qd.gqa_decode_attn(q, hq * hd, kc, vc, want, hq, hk, hd, pos, ctx, batch, ws, ws_bytes)
    got = torch.full((batch, hq * hd), float("nan"), device="cuda")
    qd.gqa_decode_attn_noalloc(q, hq * hd, kc, vc, got, hq, hk, hd, pos, ctx, batch)
    torch.cuda.synchronize()
    g = got.cpu().numpy()
    assert_close(g, want.cpu().numpy(), what="noalloc near the size limit")
    del kc, vc
    _check_oracle(g, 4, hq, hk, ctx, positions, [0, 7, 15])


def test_noalloc_attention_rejects_oversized_requests(qd):
    # just over the limit (one context step past the largest that fits) and far over it
    # (context 65536: ~68 MB of partials): refused with QD_ERR_NOMEM, nothing runs
    hq, hd, batch = 32, 64, 16
    _, over = _near_cap(hq, batch)
    t = torch.zeros(16, device="cuda")
    for ctx in (over, 65536):
        assert qd.gqa_decode_attn_workspace(hq, hd, ctx, batch) > SCRATCH_BYTES
        with pytest.raises(qd.QDError) as e:
            qd.gqa_decode_attn_noalloc(t, hq * hd, t, t, t, hq, hq, hd, t, ctx, batch)
        assert e.value.status == 6  # QD_ERR_NOMEM
