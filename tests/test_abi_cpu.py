"""The C-ABI library without a GPU: it loads, exports every declared symbol, sizes layouts,
and refuses bad arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import quantized_decode_gemv_gb300 as qd
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qdecode.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(qd.LIB_PATH):
        qd.build()
    return qd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qd_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(qd.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert qd.status_str(0) == "ok"
    for s in range(1, 8):
        assert qd.status_str(s) != "unknown status"
    assert lib.qd_abi_version() == 4


@pytest.mark.parametrize("fmt,rows,cols,src,packed", [
    ("q4_0", 576, 1536, 576 * 48 * 18, 576 * 48 * 16 + 576 * 48 * 2),
    ("q8_0", 3, 64, 3 * 2 * 34, 3 * 2 * 32 + 16),
    ("q4_k", 2, 512, 2 * 2 * 144, 2 * 2 * 128 + 2 * 2 * 16),
    ("i8", 5, 48, 5 * 48 + 20, 5 * 48 + 32),
    # Q4_1 / Q5_0: 16 code bytes per block, then 4 (d, m) / 6 (d, qh) scale bytes per block
    ("q4_1", 3, 64, 3 * 2 * 20, 3 * 2 * 16 + 32),
    ("q5_0", 3, 64, 3 * 2 * 22, 3 * 2 * 16 + 48),
    # Q5_K: 160 code bytes (qh, nibbles) + 16 header bytes; Q6_K: 192 + 18 (padded to 16)
    ("q5_k", 2, 512, 2 * 2 * 176, 2 * 2 * 160 + 2 * 2 * 16),
    ("q6_k", 3, 256, 3 * 210, 3 * 192 + 64),
    ("f16", 3, 32, 3 * 32 * 2, 3 * 32 * 2),
    ("i4", 3, 64, 3 * 32 + 12, 3 * 32 + 16),
])
def test_layout_sizes(lib, fmt, rows, cols, src, packed):
    assert qd.src_bytes(fmt, rows, cols) == src
    assert qd.packed_bytes(fmt, rows, cols) == packed


@pytest.mark.parametrize("fmt,rows,cols", [("q4_0", 4, 48), ("q8_0", 0, 64), ("q4_k", 2, 128), ("i8", 3, 40),
                                           ("q4_0", -1, 64), ("q4_1", 2, 48), ("q5_0", 2, 80), ("q5_k", 2, 384),
                                           ("q6_k", 1, 128), ("f16", 2, 48), ("i4", 2, 48)])
def test_layout_sizes_reject_bad_shapes(lib, fmt, rows, cols):
    assert qd.src_bytes(fmt, rows, cols) == 0
    assert qd.packed_bytes(fmt, rows, cols) == 0


def test_gemv_validation_before_any_device_work(lib):
    good = 4096  # a fake 16-byte-aligned "device" address: never dereferenced on these paths
    f = lib.qd_q_gemv
    assert f(99, good, 8, 64, good, good, 1, None, 0, None) == 4           # unknown format
    assert f(0, None, 8, 64, good, good, 1, None, 0, None) == 1            # null W
    assert f(0, good, 8, 64, good, good, 0, None, 0, None) == 2            # batch 0
    assert f(0, good, 8, 64, good, good, 17, None, 0, None) == 2           # batch > 16
    assert f(0, good, 8, 48, good, good, 1, None, 0, None) == 2            # cols % 32
    assert f(2, good, 8, 128, good, good, 1, None, 0, None) == 2           # Q4_K cols % 256
    assert f(0, good + 4, 8, 64, good, good, 1, None, 0, None) == 3        # misaligned W
    assert f(0, good, 8, 64, good, good + 8, 1, None, 0, None) == 3        # misaligned y
    g = lib.qd_q_gemv_ex
    assert g(0, good, 8, 64, good, good, 1, 2, None) == 1                  # unknown flag bit
    assert g(0, good, 8, 48, good, good, 1, qd.GEMV_OVERLAP, None) == 2    # cols % 32
    assert g(99, good, 8, 64, good, good, 1, 0, None) == 4                 # unknown format


def test_gemm_validation_before_any_device_work(lib):
    good = 4096
    f, w = lib.qd_q_gemm, lib.qd_q_gemm_workspace
    need = w(0, 300, 512, 80)
    # B images: 2 token tiles x 8 stages x 16 KB, then 128 f32 unscale factors
    assert need == 2 * 8 * 16384 + 128 * 4
    assert w(1, 300, 512, 80) == need and w(3, 300, 512, 80) == need
    assert w(2, 300, 512, 80) == 0 and w(0, 300, 480, 80) == 0 and w(0, 300, 512, 0) == 0
    assert w(0, 300, 512, 65537) == 0
    assert f(2, good, 300, 512, good, good, 80, good, need, None) == 4      # Q4_K: no prefill kernel
    assert f(99, good, 300, 512, good, good, 80, good, need, None) == 4     # unknown format
    assert f(0, None, 300, 512, good, good, 80, good, need, None) == 1      # null W
    assert f(0, good, 300, 512, good, good, 80, None, need, None) == 1      # null workspace
    assert f(0, good, 300, 480, good, good, 80, good, need, None) == 2      # cols % 64
    assert f(0, good, 300, 512, good, good, 0, good, need, None) == 2       # t = 0
    assert f(0, good, 300, 512, good, good, 65537, good, need, None) == 2   # t too large
    assert f(0, good, 0, 512, good, good, 80, good, need, None) == 2        # no rows
    assert f(0, good, 300, 512, good, good, 80, good, need - 1, None) == 6  # workspace too small: NOMEM
    assert f(0, good + 4, 300, 512, good, good, 80, good, need, None) == 3  # misaligned W
    assert f(0, good, 300, 512, good, good, 80, good + 8, need, None) == 3  # misaligned workspace


def test_q8_activation_validation(lib):
    good = 4096
    assert lib.qd_q8_bytes(3, 64, 0) == 3 * 64 + 16             # codes, then 3 x 2 f16 d (padded)
    assert lib.qd_q8_bytes(3, 64, 1) == 3 * 64 + 16 + 16        # ... then 3 x 2 f16 s
    assert lib.qd_q8_bytes(0, 64, 0) == 0 and lib.qd_q8_bytes(17, 64, 0) == 0 and lib.qd_q8_bytes(3, 48, 0) == 0
    assert lib.qd_q8_bytes(3, 64, 2) == 0
    q = lib.qd_quantize_q8
    assert q(None, 3, 64, 0, good, 4096, None) == 1              # null x
    assert q(good, 3, 48, 0, good, 4096, None) == 2              # cols % 32
    assert q(good, 3, 64, 0, good + 4, 4096, None) == 3          # misaligned out
    assert q(good, 3, 64, 0, good, 100, None) == 6               # out too small
    g = lib.qd_q_gemv_q8
    assert g(2, good, 8, 256, good, 4096, good, 1, None) == 4    # Q4_K: no integer product here
    assert g(0, good, 8, 48, good, 4096, good, 1, None) == 2     # cols % 32
    assert g(4, good, 8, 64, good, lib.qd_q8_bytes(1, 64, 0), good, 1, None) == 6  # Q4_1 needs the sums


def test_other_entry_points_validate(lib):
    good = 4096
    assert lib.qd_repack(0, good, 8, 64, good, 10, None) == 6              # dst too small
    assert lib.qd_repack(0, good, 8, 64, good + 2, 1 << 20, None) == 3
    assert lib.qd_rmsnorm(good, good, good, 0, 1, 1e-5, None) == 2
    assert lib.qd_rmsnorm(good, good, good, 64, 1, -1.0, None) == 1
    assert lib.qd_rope(good, 3, 63, 0, good, 1, good, 8, 1, None) == 2     # odd head_dim
    assert lib.qd_rope(good, 3, 64, 192, good, 7, good, 8, 1, None) == 4   # unknown pairing
    assert lib.qd_gqa_decode_attn(good, 576, good, good, good, 9, 3, 32, good, 8, 1, good, 1 << 20, None) == 4
    assert lib.qd_gqa_decode_attn(good, 576, good, good, good, 9, 2, 64, good, 8, 1, good, 1 << 20, None) == 2
    assert lib.qd_gqa_decode_attn(good, 576, good, good, good, 9, 3, 64, good, 8, 1, good, 1, None) == 6
    assert lib.qd_argmax(good, 0, 1, good, None) == 2
    assert lib.qd_embed(1, good, 100, 576, good, 1, good + 4, None) == 3
    assert lib.qd_swiglu(None, good, good, 10, 1, None) == 1
    assert lib.qd_decode_step(None, good, 1, good, None, None) == 1
    q = lib.qd_quantize_i8_rows
    assert q(None, 8, 64, good, 1 << 20, None) == 1                        # null weights
    assert q(good, 8, 40, good, 1 << 20, None) == 2                        # cols % 16
    assert q(good, 0, 64, good, 1 << 20, None) == 2                        # no rows
    assert q(good + 2, 8, 64, good, 1 << 20, None) == 3                    # misaligned weights
    assert q(good, 8, 64, good + 4, 1 << 20, None) == 3                    # misaligned output
    assert q(good, 8, 64, good, 8 * 64 + 8 * 4 - 1, None) == 6             # output one byte short
    q4 = lib.qd_quantize_i4_rows
    assert q4(None, 8, 64, good, 1 << 20, None) == 1                       # null weights
    assert q4(good, 8, 48, good, 1 << 20, None) == 2                       # INT4 rows need cols % 32
    assert q4(good, 0, 64, good, 1 << 20, None) == 2                       # no rows
    assert q4(good, 8, 64, good + 8, 1 << 20, None) == 3                   # misaligned output
    assert q4(good, 8, 64, good, 8 * 32 + 8 * 4 - 1, None) == 6            # output one byte short


def test_model_sizes_and_config_refusals(lib):
    import qdsynth

    c = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=1)
    wb = lib.qd_model_weight_bytes(ctypes.byref(c))
    sb = lib.qd_model_state_bytes(ctypes.byref(c))
    src = qdsynth.model_weight_src_bytes(qdsynth.SMOL_135M)
    assert src <= wb <= src + 4096 * (3 + 9 * 30)  # same bytes as the source plus alignment padding
    kv = 2 * 30 * 3 * 256 * 64 * 4
    assert kv < sb < kv + (64 << 20)
    bad = qd.make_config(dict(qdsynth.SMOL_135M, n_kv_heads=2), max_ctx=256, max_batch=1)  # 9 % 2
    assert lib.qd_model_weight_bytes(ctypes.byref(bad)) == 0
    bad = qd.make_config(dict(qdsynth.SMOL_135M, head_dim=32), max_ctx=256, max_batch=1)
    assert lib.qd_model_state_bytes(ctypes.byref(bad)) == 0
    bad = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=17)
    assert lib.qd_model_state_bytes(ctypes.byref(bad)) == 0
    bad = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=1)
    bad.kv_f16 = 2
    assert lib.qd_model_state_bytes(ctypes.byref(bad)) == 0
    # the decode step takes every format but per-row INT4, where its block fits the shapes:
    # 576 columns take the 32-wide blocks, not the 256-wide K super-blocks
    for f in ("q4_1", "q5_0", "f16"):
        ok = qd.make_config(dict(qdsynth.SMOL_135M, w_fmt=f), max_ctx=256, max_batch=1)
        assert lib.qd_model_weight_bytes(ctypes.byref(ok)) > 0, f
        ok = qd.make_config(dict(qdsynth.SMOL_135M, emb_fmt=f), max_ctx=256, max_batch=1)
        assert lib.qd_model_state_bytes(ctypes.byref(ok)) > 0, f
    for f in ("q5_k", "q6_k", "q4_k"):
        bad = qd.make_config(dict(qdsynth.SMOL_135M, w_fmt=f), max_ctx=256, max_batch=1)
        assert lib.qd_model_weight_bytes(ctypes.byref(bad)) == 0, f
    bad = qd.make_config(dict(qdsynth.SMOL_135M, w_fmt="i4"), max_ctx=256, max_batch=1)
    assert lib.qd_model_weight_bytes(ctypes.byref(bad)) == 0
    # per-class formats: each class checked on its own shapes; sizes follow the classes
    wide = dict(qdsynth.SMOL_135M, dim=512, ffn=1024, n_heads=8, n_kv_heads=4)  # 256-divisible widths
    uni = qd.make_config(dict(wide, w_fmt="q4_k"), max_ctx=256, max_batch=1)
    mix = qd.make_config(dict(wide, w_fmt="q4_k", down_fmt="q6_k"), max_ctx=256, max_batch=1)
    assert mix.mixed_fmt == 1 and uni.mixed_fmt == 0
    wu, wm = lib.qd_model_weight_bytes(ctypes.byref(uni)), lib.qd_model_weight_bytes(ctypes.byref(mix))
    # Q6_K in place of Q4_K for wd (512 x 1024) in each of 30 layers, regions 256-aligned
    r256 = lambda n: (n + 255) // 256 * 256
    pb = lambda f: lib.qd_packed_bytes(qd.FMT[f], 512, 1024)
    assert wm - wu == 30 * (r256(pb("q6_k")) - r256(pb("q4_k"))) > 0
    bad = qd.make_config(dict(qdsynth.SMOL_135M, down_fmt="q6_k"), max_ctx=256, max_batch=1)  # 1536 ok, 576 rows
    assert lib.qd_model_weight_bytes(ctypes.byref(bad)) > 0  # wd is 576 x 1536: 1536 = 6 x 256 columns
    bad = qd.make_config(dict(qdsynth.SMOL_135M, wo_fmt="q6_k"), max_ctx=256, max_batch=1)  # 576 columns
    assert lib.qd_model_weight_bytes(ctypes.byref(bad)) == 0
    bad = qd.make_config(dict(qdsynth.SMOL_135M, down_fmt="q4_k"), max_ctx=256, max_batch=1, act_q8=True)
    assert lib.qd_model_state_bytes(ctypes.byref(bad)) == 0  # ggml-exact products: Q4_0 / Q8_0 only
    bad = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=1)
    bad.mixed_fmt = 2
    assert lib.qd_model_weight_bytes(ctypes.byref(bad)) == 0
    # ggml-exact products take Q4_0 / Q8_0 weights only, and act_q8 is a flag
    ok = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=1, act_q8=True)
    assert lib.qd_model_state_bytes(ctypes.byref(ok)) > sb  # plus the quantised-activation buffer
    bad = qd.make_config(dict(qdsynth.SMOL_135M, w_fmt="q4_k"), max_ctx=256, max_batch=1, act_q8=True)
    assert lib.qd_model_state_bytes(ctypes.byref(bad)) == 0
    bad = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=1)
    bad.act_q8 = 2
    assert lib.qd_model_state_bytes(ctypes.byref(bad)) == 0
    # a binary16 cache takes half the bytes (the state also gains the flat attention's workspace)
    h = qd.make_config(qdsynth.SMOL_135M, max_ctx=256, max_batch=1, kv_f16=True)
    sh = lib.qd_model_state_bytes(ctypes.byref(h))
    assert kv // 2 < sh < sb - kv // 2 + (1 << 20)


def test_rope_table_host_matches_oracle(lib):
    """The library's host table and the oracle's both round double cos/sin of
    p * theta^(-2i/hd) to f32; they must agree exactly."""
    hd, ctx, theta = 64, 300, 1e5
    got = np.empty((ctx, hd // 2, 2), np.float32)
    qd.rope_table(theta, hd, ctx, got.ctypes.data)
    want = oracle.rope_table(theta, hd, ctx)
    assert np.array_equal(got, want)


def test_prefill_workspace_sizes(lib):
    """qd_prefill_workspace: host arithmetic only (no device work); 0 where qd_prefill refuses."""
    import qdsynth

    cfg = qdsynth.SMOL_135M
    c = qd.make_config(cfg, max_ctx=256, max_batch=1)
    w128 = lib.qd_prefill_workspace(ctypes.byref(c), 128)
    w16 = lib.qd_prefill_workspace(ctypes.byref(c), 16)
    # at least the t-row activations: x, xn (dim), qkv (dim + 2 kv), q and attention out, act (ffn)
    per_tok = 4 * (2 * 576 + (576 + 2 * 192) + 2 * 576 + 1536)
    assert w128 >= 128 * per_tok and w16 >= 16 * per_tok and w128 > w16
    assert lib.qd_prefill_workspace(ctypes.byref(c), 0) == 0
    assert lib.qd_prefill_workspace(ctypes.byref(c), 257) == 0  # beyond max_ctx
    q8 = qd.make_config(cfg, max_ctx=256, max_batch=1, act_q8=True)
    assert lib.qd_prefill_workspace(ctypes.byref(q8), 16) == 0  # ggml-exact models: refused
    h = qd.make_config(cfg, max_ctx=256, max_batch=1, kv_f16=True)
    assert lib.qd_prefill_workspace(ctypes.byref(h), 128) >= 128 * per_tok
