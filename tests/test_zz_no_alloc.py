"""The allocation-free attention entry point.

Some callers of this library cannot allocate device memory for a workspace: a serving
loop that must never call cudaMalloc (it can synchronise the device), or code running
under a fixed memory budget that another allocator already owns.  For them
qd_gqa_decode_attn_noalloc keeps its partial results in a fixed device array inside the
library.  This test calls it through the C ABI twice in a row, with different inputs, and
checks each result against qd_gqa_decode_attn with a caller-provided workspace, within the
tolerance the other parity tests use.  The file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import qdsynth
from gpu_helpers import assert_close, dev

pytestmark = pytest.mark.gpu


def _case(seed, hq, hk, ctx, positions):
    hd = 64
    batch = len(positions)
    kc = qdsynth.normal_f32(seed, "na.k", batch * hk * ctx * hd).reshape(batch, hk, ctx, hd)
    vc = qdsynth.normal_f32(seed, "na.v", batch * hk * ctx * hd).reshape(batch, hk, ctx, hd)
    q = qdsynth.activations(seed, "na.q", batch, hq * hd)
    return dev(q), dev(kc), dev(vc), dev(np.array(positions, np.int32))


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
        assert_close(got.cpu().numpy(), want.cpu().numpy(), what=f"noalloc call seed {seed}")


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
    assert_close(got.cpu().numpy(), want.cpu().numpy(), what="noalloc gqa")


def test_noalloc_attention_rejects_oversized_requests(qd):
    # 32 heads, context 65536, batch 16 would need ~68 MB of partials: refused, nothing runs
    hq, hd, ctx, batch = 32, 64, 65536, 16
    assert qd.gqa_decode_attn_workspace(hq, hd, ctx, batch) > (8 << 20)
    t = torch.zeros(16, device="cuda")
    with pytest.raises(qd.QDError) as e:
        qd.gqa_decode_attn_noalloc(t, hq * hd, t, t, t, hq, hq, hd, t, ctx, batch)
    assert e.value.status == 6  # QD_ERR_NOMEM
