"""Python binding of libqdecode (argument marshalling only).

Every function here forwards to the C entry point of the same name in ``include/qdecode.h``
(without the ``qd_`` prefix): device tensors are passed as ``data_ptr()`` and the stream as
``torch.cuda.current_stream().cuda_stream`` unless given.  All arithmetic runs in the CUDA
library.  There is no fallback: if ``libqdecode.so`` is missing or does not load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqdecode.so")
_lib = None

FMT = {"q4_0": 0, "q8_0": 1, "q4_k": 2, "i8": 3, "q4_1": 4, "q5_0": 5, "q5_k": 6, "q6_k": 7, "f16": 8, "i4": 9}
PAIRING = {"adjacent": 0, "half": 1}
MAX_BATCH = 16
STATUS = {0: "QD_OK", 1: "QD_ERR_INVALID_ARG", 2: "QD_ERR_SHAPE", 3: "QD_ERR_ALIGN", 4: "QD_ERR_UNSUPPORTED",
          5: "QD_ERR_CUDA", 6: "QD_ERR_NOMEM", 7: "QD_ERR_DEVICE_FLAG"}

# Every symbol include/qdecode.h declares (checked by the CPU test suite).
EXPORTS = ["qd_status_str", "qd_abi_version", "qd_f16_to_f32", "qd_bf16_to_f32", "qd_src_bytes", "qd_packed_bytes",
           "qd_repack", "qd_unpack", "qd_dequant", "qd_quantize_i8_rows", "qd_quantize_i4_rows",
           "qd_q_gemv_workspace", "qd_q_gemv",
           "qd_q_gemv_ex", "qd_read_ceiling", "qd_q_gemm_workspace", "qd_q_gemm", "qd_q8_bytes",
           "qd_quantize_q8", "qd_q_gemv_q8", "qd_rmsnorm",
           "qd_rope_table", "qd_rope", "qd_kv_append", "qd_gqa_decode_attn_workspace", "qd_gqa_decode_attn",
           "qd_gqa_decode_attn_noalloc",
           "qd_swiglu", "qd_argmax", "qd_embed", "qd_model_weight_bytes", "qd_model_state_bytes",
           "qd_model_create", "qd_model_destroy", "qd_decode_step", "qd_prefill_workspace", "qd_prefill",
           "qd_model_reset", "qd_model_set_pos",
           "qd_model_pos", "qd_model_kv_cache", "qd_model_act_q8_buffer", "qd_model_check",
           "qd_model_launches_per_step", "qd_model_set_step_path", "qd_model_step_path",
           "qd_model_cluster_available"]
STEP_AUTO, STEP_KERNEL_CHAIN, STEP_CLUSTER = 0, 1, 2
PREFILL_EXACT = 1


class QDError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


class Config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("vocab", ctypes.c_int), ("max_ctx", ctypes.c_int), ("max_batch", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("eps", ctypes.c_float), ("pairing", ctypes.c_int),
                ("w_fmt", ctypes.c_int), ("emb_fmt", ctypes.c_int), ("tied", ctypes.c_int),
                ("kv_f16", ctypes.c_int), ("act_q8", ctypes.c_int), ("mixed_fmt", ctypes.c_int),
                ("qkv_fmt", ctypes.c_int), ("wo_fmt", ctypes.c_int), ("gate_up_fmt", ctypes.c_int),
                ("down_fmt", ctypes.c_int)]


def build(force: bool = False) -> str:
    from . import builder as _b

    return _b.build(force=force)


def load():
    """Load libqdecode.so (built in-tree by ``build()``); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libqdecode.so not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    p, i64, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    sig = {
        "qd_status_str": ([i32], ctypes.c_char_p),
        "qd_abi_version": ([], i32),
        "qd_f16_to_f32": ([p, p, i64, p], i32),
        "qd_bf16_to_f32": ([p, p, i64, p], i32),
        "qd_src_bytes": ([i32, i64, i64], sz),
        "qd_packed_bytes": ([i32, i64, i64], sz),
        "qd_repack": ([i32, p, i64, i64, p, sz, p], i32),
        "qd_unpack": ([i32, p, i64, i64, p, sz, p], i32),
        "qd_dequant": ([i32, p, i64, i64, p, p], i32),
        "qd_quantize_i8_rows": ([p, i64, i64, p, sz, p], i32),
        "qd_quantize_i4_rows": ([p, i64, i64, p, sz, p], i32),
        "qd_q_gemv_workspace": ([i32, i64, i64, i32], sz),
        "qd_q_gemv": ([i32, p, i64, i64, p, p, i32, p, sz, p], i32),
        "qd_q_gemv_ex": ([i32, p, i64, i64, p, p, i32, ctypes.c_uint, p], i32),
        "qd_read_ceiling": ([p, sz, i32, i32, ctypes.c_uint, p, p], i32),
        "qd_q_gemm_workspace": ([i32, i64, i64, i32], sz),
        "qd_q_gemm": ([i32, p, i64, i64, p, p, i32, p, sz, p], i32),
        "qd_q8_bytes": ([i32, i64, i32], sz),
        "qd_quantize_q8": ([p, i32, i64, i32, p, sz, p], i32),
        "qd_q_gemv_q8": ([i32, p, i64, i64, p, sz, p, i32, p], i32),
        "qd_rmsnorm": ([p, p, p, i32, i32, f32, p], i32),
        "qd_rope_table": ([f32, i32, i32, p], i32),
        "qd_rope": ([p, i32, i32, i64, p, i32, p, i32, i32, p], i32),
        "qd_kv_append": ([p, p, i64, p, p, i32, i32, p, i32, i32, p], i32),
        "qd_gqa_decode_attn_workspace": ([i32, i32, i32, i32], sz),
        "qd_gqa_decode_attn": ([p, i64, p, p, p, i32, i32, i32, p, i32, i32, p, sz, p], i32),
        "qd_gqa_decode_attn_noalloc": ([p, i64, p, p, p, i32, i32, i32, p, i32, i32, p], i32),
        "qd_swiglu": ([p, p, p, i64, i32, p], i32),
        "qd_argmax": ([p, i64, i32, p, p], i32),
        "qd_embed": ([i32, p, i64, i64, p, i32, p, p], i32),
        "qd_model_weight_bytes": ([ctypes.POINTER(Config)], sz),
        "qd_model_state_bytes": ([ctypes.POINTER(Config)], sz),
        "qd_model_create": ([ctypes.POINTER(Config), p, p, sz, p, sz, p, ctypes.POINTER(p)], i32),
        "qd_model_destroy": ([p], None),
        "qd_decode_step": ([p, p, i32, p, p, p], i32),
        "qd_prefill_workspace": ([ctypes.POINTER(Config), i32], sz),
        "qd_prefill": ([p, i32, p, i32, ctypes.c_uint, p, sz, p, p, p], i32),
        "qd_model_reset": ([p, p], i32),
        "qd_model_set_pos": ([p, p, i32, p], i32),
        "qd_model_pos": ([p, p, i32, p], i32),
        "qd_model_kv_cache": ([p, ctypes.POINTER(p), ctypes.POINTER(p)], i32),
        "qd_model_act_q8_buffer": ([p, ctypes.POINTER(p), ctypes.POINTER(sz), ctypes.POINTER(i32)], i32),
        "qd_model_check": ([p, p], i32),
        "qd_model_launches_per_step": ([p], i32),
        "qd_model_set_step_path": ([p, i32], i32),
        "qd_model_step_path": ([p], i32),
        "qd_model_cluster_available": ([p], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# ------------------------------------------------------------------------------ marshalling

def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != 0:
        raise QDError(fn, st)


def status_str(s: int) -> str:
    return load().qd_status_str(s).decode()


def src_bytes(fmt: str, rows: int, cols: int) -> int:
    return int(load().qd_src_bytes(FMT[fmt], rows, cols))


def packed_bytes(fmt: str, rows: int, cols: int) -> int:
    return int(load().qd_packed_bytes(FMT[fmt], rows, cols))


def f16_to_f32(inp, out, n=None, stream=None):
    n = inp.numel() if n is None else n
    _check("qd_f16_to_f32", load().qd_f16_to_f32(_ptr(inp), _ptr(out), n, _stream(stream)))


def bf16_to_f32(inp, out, n=None, stream=None):
    n = inp.numel() if n is None else n
    _check("qd_bf16_to_f32", load().qd_bf16_to_f32(_ptr(inp), _ptr(out), n, _stream(stream)))


def repack(fmt, src, rows, cols, dst, dst_bytes=None, stream=None):
    nbytes = dst.numel() * dst.element_size() if dst_bytes is None else dst_bytes
    _check("qd_repack", load().qd_repack(FMT[fmt], _ptr(src), rows, cols, _ptr(dst), nbytes, _stream(stream)))


def unpack(fmt, packed, rows, cols, dst, dst_bytes=None, stream=None):
    nbytes = dst.numel() * dst.element_size() if dst_bytes is None else dst_bytes
    _check("qd_unpack", load().qd_unpack(FMT[fmt], _ptr(packed), rows, cols, _ptr(dst), nbytes, _stream(stream)))


def dequant(fmt, packed, rows, cols, out, stream=None):
    _check("qd_dequant", load().qd_dequant(FMT[fmt], _ptr(packed), rows, cols, _ptr(out), _stream(stream)))


def quantize_i4_rows(w_bf16, rows, cols, out, out_bytes=None, stream=None):
    nbytes = out.numel() * out.element_size() if out_bytes is None else out_bytes
    _check("qd_quantize_i4_rows", load().qd_quantize_i4_rows(_ptr(w_bf16), rows, cols, _ptr(out), nbytes,
                                                             _stream(stream)))


def quantize_i8_rows(w_bf16, rows, cols, out, out_bytes=None, stream=None):
    """BF16 weights (uint16/int16/bfloat16 tensor [rows][cols]) -> per-row INT8 source layout."""
    nbytes = out.numel() * out.element_size() if out_bytes is None else out_bytes
    _check("qd_quantize_i8_rows",
           load().qd_quantize_i8_rows(_ptr(w_bf16), rows, cols, _ptr(out), nbytes, _stream(stream)))


def q_gemv_workspace(fmt, rows, cols, batch) -> int:
    return int(load().qd_q_gemv_workspace(FMT[fmt], rows, cols, batch))


def q_gemm_workspace(fmt, rows, cols, t) -> int:
    return int(load().qd_q_gemm_workspace(FMT[fmt], rows, cols, t))


def q_gemm(fmt, W, rows, cols, x, y, t, workspace, workspace_bytes=None, stream=None):
    """y[n][r] = sum_c deq(W)[r][c] x[n][c] for n < t on the tensor cores (see qdecode.h)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("qd_q_gemm", load().qd_q_gemm(FMT[fmt], _ptr(W), rows, cols, _ptr(x), _ptr(y), t, _ptr(workspace),
                                         workspace_bytes, _stream(stream)))


def q8_bytes(batch, cols, with_sum=False) -> int:
    return int(load().qd_q8_bytes(batch, cols, 1 if with_sum else 0))


def quantize_q8(x, batch, cols, out, with_sum=False, out_bytes=None, stream=None):
    """ggml-exact Q8_0 (Q8_1 with with_sum) activations of x [batch][cols] into out."""
    nbytes = out.numel() * out.element_size() if out_bytes is None else out_bytes
    _check("qd_quantize_q8", load().qd_quantize_q8(_ptr(x), batch, cols, 1 if with_sum else 0, _ptr(out), nbytes,
                                                   _stream(stream)))


def q_gemv_q8(fmt, W, rows, cols, xq, y, batch, xq_bytes=None, stream=None):
    """y = W x over quantised activations xq (quantize_q8 output) in integers."""
    nbytes = xq.numel() * xq.element_size() if xq_bytes is None else xq_bytes
    _check("qd_q_gemv_q8", load().qd_q_gemv_q8(FMT[fmt], _ptr(W), rows, cols, _ptr(xq), nbytes, _ptr(y), batch,
                                               _stream(stream)))


def q_gemv(fmt, W, rows, cols, x, y, batch, workspace=None, workspace_bytes=0, stream=None):
    _check("qd_q_gemv", load().qd_q_gemv(FMT[fmt], _ptr(W), rows, cols, _ptr(x), _ptr(y), batch, _ptr(workspace),
                                         workspace_bytes, _stream(stream)))


GEMV_OVERLAP = 1


def q_gemv_ex(fmt, W, rows, cols, x, y, batch, flags=0, stream=None):
    _check("qd_q_gemv_ex", load().qd_q_gemv_ex(FMT[fmt], _ptr(W), rows, cols, _ptr(x), _ptr(y), batch, flags,
                                               _stream(stream)))


def read_ceiling(buf, nbytes, ctas_per_sm, threads, flags=0, sink=None, stream=None):
    """Roofline calibration: one plain read of nbytes of buf (see qd_read_ceiling)."""
    _check("qd_read_ceiling", load().qd_read_ceiling(_ptr(buf), nbytes, ctas_per_sm, threads, flags, _ptr(sink),
                                                     _stream(stream)))


def rmsnorm(x, g, out, n, batch, eps, stream=None):
    _check("qd_rmsnorm", load().qd_rmsnorm(_ptr(x), _ptr(g), _ptr(out), n, batch, eps, _stream(stream)))


def rope_table(theta, head_dim, ctx, dst_host_ptr):
    _check("qd_rope_table", load().qd_rope_table(theta, head_dim, ctx, dst_host_ptr))


def rope(v, n_heads, head_dim, batch_stride, pos, pairing, cos_sin, max_ctx, batch, stream=None):
    _check("qd_rope", load().qd_rope(_ptr(v), n_heads, head_dim, batch_stride, _ptr(pos), PAIRING[pairing],
                                     _ptr(cos_sin), max_ctx, batch, _stream(stream)))


def kv_append(k, v, src_batch_stride, k_cache, v_cache, n_kv_heads, head_dim, pos, max_ctx, batch, stream=None):
    _check("qd_kv_append", load().qd_kv_append(_ptr(k), _ptr(v), src_batch_stride, _ptr(k_cache), _ptr(v_cache),
                                               n_kv_heads, head_dim, _ptr(pos), max_ctx, batch, _stream(stream)))


def gqa_decode_attn_workspace(n_heads, head_dim, max_ctx, batch) -> int:
    return int(load().qd_gqa_decode_attn_workspace(n_heads, head_dim, max_ctx, batch))


def gqa_decode_attn(q, q_batch_stride, k_cache, v_cache, out, n_heads, n_kv_heads, head_dim, pos, max_ctx, batch,
                    workspace, workspace_bytes, stream=None):
    _check("qd_gqa_decode_attn",
           load().qd_gqa_decode_attn(_ptr(q), q_batch_stride, _ptr(k_cache), _ptr(v_cache), _ptr(out), n_heads,
                                     n_kv_heads, head_dim, _ptr(pos), max_ctx, batch, _ptr(workspace),
                                     workspace_bytes, _stream(stream)))


def gqa_decode_attn_noalloc(q, q_batch_stride, k_cache, v_cache, out, n_heads, n_kv_heads, head_dim, pos, max_ctx,
                            batch, stream=None):
    """Attention without a caller workspace (the library's fixed device scratch)."""
    _check("qd_gqa_decode_attn_noalloc",
           load().qd_gqa_decode_attn_noalloc(_ptr(q), q_batch_stride, _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                             n_heads, n_kv_heads, head_dim, _ptr(pos), max_ctx, batch,
                                             _stream(stream)))


def swiglu(gate, up, out, n, batch, stream=None):
    _check("qd_swiglu", load().qd_swiglu(_ptr(gate), _ptr(up), _ptr(out), n, batch, _stream(stream)))


def argmax(logits, n, batch, out_idx, stream=None):
    _check("qd_argmax", load().qd_argmax(_ptr(logits), n, batch, _ptr(out_idx), _stream(stream)))


def embed(fmt, E, vocab, dim, tokens, batch, x, stream=None):
    _check("qd_embed", load().qd_embed(FMT[fmt], _ptr(E), vocab, dim, _ptr(tokens), batch, _ptr(x),
                                       _stream(stream)))


def make_config(cfg: dict, max_ctx: int, max_batch: int, tied: bool = True, kv_f16: bool | None = None,
                act_q8: bool | None = None) -> Config:
    """kv_f16: binary16 KV cache (default: cfg.get("kv_f16", False)); act_q8: products over
    Q8_0 activations (default: cfg.get("act_q8", False)).  A config naming any of qkv_fmt,
    wo_fmt, gate_up_fmt or down_fmt is a mixed-format model (the classes it does not name
    take w_fmt)."""
    f16 = cfg.get("kv_f16", False) if kv_f16 is None else kv_f16
    q8 = cfg.get("act_q8", False) if act_q8 is None else act_q8
    classes = ("qkv_fmt", "wo_fmt", "gate_up_fmt", "down_fmt")
    mixed = any(k in cfg for k in classes)
    per = [FMT[cfg.get(k, cfg["w_fmt"])] for k in classes]
    return Config(cfg["layers"], cfg["dim"], cfg["ffn"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                  cfg["vocab"], max_ctx, max_batch, cfg["rope_theta"], cfg["eps"], PAIRING[cfg["pairing"]],
                  FMT[cfg["w_fmt"]], FMT[cfg["emb_fmt"]], 1 if tied else 0, 1 if f16 else 0, 1 if q8 else 0,
                  1 if mixed else 0, *per)


class Model:
    """A decode model over caller-owned device memory (torch uint8 tensors)."""

    def __init__(self, cfg: Config, src_tensors: list, stream=None):
        import torch

        lib = load()
        self.cfg = cfg
        wb = lib.qd_model_weight_bytes(ctypes.byref(cfg))
        sb = lib.qd_model_state_bytes(ctypes.byref(cfg))
        if not wb or not sb:
            raise QDError("qd_model_weight_bytes", 4)
        self.weights = torch.empty(wb, dtype=torch.uint8, device="cuda")
        self.state = torch.empty(sb, dtype=torch.uint8, device="cuda")
        ptrs = (ctypes.c_void_p * len(src_tensors))(*[_ptr(t) for t in src_tensors])
        h = ctypes.c_void_p()
        _check("qd_model_create", lib.qd_model_create(ctypes.byref(cfg), ptrs, self.weights.data_ptr(), wb,
                                                      self.state.data_ptr(), sb, _stream(stream), ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            load().qd_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def decode_step(self, tokens, batch, out_tokens, logits_out=None, stream=None):
        """tokens / out_tokens / logits_out: torch tensors (host or device) or raw pointers."""
        _check("qd_decode_step", load().qd_decode_step(self.handle, _ptr(tokens), batch, _ptr(out_tokens),
                                                       _ptr(logits_out), _stream(stream)))

    def prefill_workspace(self, t):
        """Bytes of the workspace qd_prefill needs for t tokens (0: not available)."""
        return load().qd_prefill_workspace(ctypes.byref(self.cfg), t)

    def prefill(self, seq, tokens, t, out_token, logits_out=None, flags=0, workspace=None, stream=None):
        """Run t prompt tokens of sequence seq in one call (qd_prefill).  tokens, out_token,
        logits_out: torch tensors (host or device) or raw pointers; workspace: a device
        tensor of at least prefill_workspace(t) bytes (allocated here when None)."""
        import torch

        need = self.prefill_workspace(t)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        nbytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else need
        _check("qd_prefill", load().qd_prefill(self.handle, seq, _ptr(tokens), t, flags, _ptr(workspace), nbytes,
                                               _ptr(out_token), _ptr(logits_out), _stream(stream)))

    def reset(self, stream=None):
        _check("qd_model_reset", load().qd_model_reset(self.handle, _stream(stream)))

    def set_pos(self, pos_list, stream=None):
        arr = (ctypes.c_int32 * len(pos_list))(*pos_list)
        _check("qd_model_set_pos", load().qd_model_set_pos(self.handle, arr, len(pos_list), _stream(stream)))

    def pos(self, batch, stream=None):
        arr = (ctypes.c_int32 * batch)()
        _check("qd_model_pos", load().qd_model_pos(self.handle, arr, batch, _stream(stream)))
        return list(arr)

    def kv_cache_ptrs(self):
        k, v = ctypes.c_void_p(), ctypes.c_void_p()
        _check("qd_model_kv_cache", load().qd_model_kv_cache(self.handle, ctypes.byref(k), ctypes.byref(v)))
        return k.value, v.value

    def act_q8_buffer(self):
        """(device pointer, bytes per slot, slots) of the act_q8 quantised inputs of the last
        step ((None, 0, 0) without act_q8)."""
        b, n, k = ctypes.c_void_p(), ctypes.c_size_t(), ctypes.c_int()
        _check("qd_model_act_q8_buffer", load().qd_model_act_q8_buffer(self.handle, ctypes.byref(b), ctypes.byref(n),
                                                                       ctypes.byref(k)))
        return b.value, n.value, k.value

    def check(self, stream=None) -> int:
        return int(load().qd_model_check(self.handle, _stream(stream)))

    def set_step_path(self, path: int):
        """STEP_AUTO, STEP_KERNEL_CHAIN or STEP_CLUSTER (see qd_model_set_step_path)."""
        _check("qd_model_set_step_path", load().qd_model_set_step_path(self.handle, int(path)))

    def step_path(self) -> int:
        return int(load().qd_model_step_path(self.handle))

    def cluster_available(self) -> bool:
        return bool(load().qd_model_cluster_available(self.handle))

    def launches_per_step(self) -> int:
        return int(load().qd_model_launches_per_step(self.handle))
