"""Python face of the CPU oracle (``qd_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline
leg are the only callers.  The oracle shares no code with the CUDA library and imports
nothing from it; it is handed the same seeded input bytes (from ``qdsynth``) and computes
the plain definition of every operation in double precision.

Function-by-function sources are cited in ``qd_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

FMT = {"q4_0": 0, "q8_0": 1, "q4_k": 2, "i8": 3, "q4_1": 4, "q5_0": 5, "q5_k": 6, "q6_k": 7, "f16": 8, "i4": 9}
PAIRING = {"adjacent": 0, "half": 1}


def build(force: bool = False, sanitize: bool = False) -> str:
    """Compile liboracle.so (gcc -O2, OpenMP when available).  ``sanitize`` builds an
    ASan/UBSan variant under another name for the sanitizer test."""
    out = _LIB_PATH if not sanitize else os.path.join(_HERE, "liboracle_san.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    flags = ["-O2", "-std=c99", "-fPIC", "-shared", "-Wall", "-Wno-unknown-pragmas"]
    if sanitize:
        flags = ["-O1", "-g", "-std=c99", "-fPIC", "-shared", "-fsanitize=address,undefined",
                 "-fno-omit-frame-pointer"]
    base = ["gcc"] + flags + [_SRC, "-o", out + ".tmp", "-lm"]
    if sanitize:
        subprocess.run(base, check=True, capture_output=True)
    else:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


class _Config(ctypes.Structure):
    _fields_ = [("layers", ctypes.c_int), ("dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("vocab", ctypes.c_int), ("max_ctx", ctypes.c_int), ("rope_theta", ctypes.c_double),
                ("eps", ctypes.c_double), ("pairing", ctypes.c_int), ("w_fmt", ctypes.c_int),
                ("emb_fmt", ctypes.c_int), ("kv_f16", ctypes.c_int), ("act_q8", ctypes.c_int),
                ("qkv_fmt", ctypes.c_int), ("wo_fmt", ctypes.c_int), ("gate_up_fmt", ctypes.c_int),
                ("down_fmt", ctypes.c_int)]


class _Q8TF(ctypes.Structure):
    _fields_ = [("q_given", ctypes.c_void_p), ("d_given", ctypes.c_void_p), ("x_out", ctypes.c_void_p),
                ("slot_cols", ctypes.c_int64)]


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p, i64, i32, d = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.or_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_f64.restype = d
        lib.or_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.or_bf16_to_f32.restype = ctypes.c_float
        lib.or_bf16_to_f32_array.argtypes = [p, i64, p]
        lib.or_f16_to_f32_array.argtypes = [p, i64, p]
        lib.or_get_scale_min_k4.argtypes = [i32, p, p, p]
        lib.or_dequant.argtypes = [i32, p, i64, i64, i64, i64, p]
        lib.or_dequant.restype = i32
        lib.or_gemv.argtypes = [i32, p, i64, i64, p, i32, i64, i64, p]
        lib.or_gemv.restype = i32
        lib.or_quantize_i4_rows.argtypes = [p, i64, i64, p, p]
        lib.or_quantize_i4_rows.restype = i32
        lib.or_quantize_q8.argtypes = [p, i64, p, p, p]
        lib.or_quantize_q8.restype = i32
        lib.or_gemv_q8act.argtypes = [i32, p, i64, i64, p, p, p, i32, i64, i64, p]
        lib.or_gemv_q8act.restype = i32
        lib.or_rmsnorm.argtypes = [p, p, i32, i32, d, p]
        lib.or_rmsnorm.restype = i32
        lib.or_rope.argtypes = [p, i32, i32, i32, i32, d, p]
        lib.or_rope.restype = i32
        lib.or_rope_table.argtypes = [d, i32, i32, p]
        lib.or_rope_table.restype = i32
        lib.or_attention.argtypes = [p, p, p, i32, i32, i32, i32, i64, p]
        lib.or_attention.restype = i32
        lib.or_swiglu.argtypes = [p, p, i64, p]
        lib.or_swiglu.restype = i32
        lib.or_round_f16.argtypes = [ctypes.c_float]
        lib.or_round_f16.restype = ctypes.c_float
        lib.or_quantize_i8_rows.argtypes = [p, i64, i64, p, p]
        lib.or_quantize_i8_rows.restype = i32
        lib.or_set_threads.argtypes = [i32]
        lib.or_set_threads.restype = i32
        lib.or_argmax_f32.argtypes = [p, i64]
        lib.or_argmax_f32.restype = i64
        lib.or_argmax_f64.argtypes = [p, i64]
        lib.or_argmax_f64.restype = i64
        lib.or_silu.argtypes = [d]
        lib.or_silu.restype = d
        lib.or_decode_step.argtypes = [ctypes.POINTER(_Config), p, p, p, i64, i32, i32, p,
                                       ctypes.POINTER(ctypes.c_int64)]
        lib.or_decode_step.restype = i32
        lib.or_decode_step_tf.argtypes = [ctypes.POINTER(_Config), p, p, p, i64, i32, i32, p,
                                          ctypes.POINTER(ctypes.c_int64), i32, p, p, ctypes.POINTER(_Q8TF)]
        lib.or_decode_step_tf.restype = i32
        lib.or_gemv_xd.argtypes = [i32, p, i64, i64, p, i32, i64, i64, p]
        lib.or_gemv_xd.restype = i32
        lib.or_rmsnorm_d.argtypes = [p, p, i32, d, p]
        lib.or_rmsnorm_d.restype = None
        lib.or_rope_head_d.argtypes = [p, i32, i32, i32, d]
        lib.or_rope_head_d.restype = None
        lib.or_attention_d.argtypes = [p, p, p, i32, i32, i32, i32, i64, p]
        lib.or_attention_d.restype = None
        _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def f16_to_f64(h: int) -> float:
    return float(_L().or_f16_to_f64(int(h) & 0xFFFF))


def bf16_to_f32(b: int) -> float:
    return float(_L().or_bf16_to_f32(int(b) & 0xFFFF))


def bf16_to_f32_array(bits) -> np.ndarray:
    b, bp = _c(bits, np.uint16)
    out = np.empty(b.size, dtype=np.float32)
    _L().or_bf16_to_f32_array(bp, b.size, out.ctypes.data)
    return out


def f16_to_f32_array(bits) -> np.ndarray:
    b, bp = _c(bits, np.uint16)
    out = np.empty(b.size, dtype=np.float32)
    _L().or_f16_to_f32_array(bp, b.size, out.ctypes.data)
    return out


def get_scale_min_k4(j: int, q12) -> tuple[int, int]:
    q, qp = _c(q12, np.uint8)
    assert q.size == 12
    sc, m = ctypes.c_uint8(), ctypes.c_uint8()
    _L().or_get_scale_min_k4(j, qp, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def dequant(fmt: str, w, rows: int, cols: int, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """Dequantised f32 values of rows [row0, row0+nrows) of a model-file-layout tensor."""
    nrows = rows - row0 if nrows is None else nrows
    w, wp = _c(w, np.uint8)
    out = np.empty((nrows, cols), dtype=np.float32)
    rc = _L().or_dequant(FMT[fmt], wp, rows, cols, row0, nrows, out.ctypes.data)
    if rc:
        raise ValueError(f"or_dequant rc={rc}")
    return out


def gemv(fmt: str, w, rows: int, cols: int, x, row0: int = 0, nrows: int | None = None) -> np.ndarray:
    """y[b][r] = sum_c deq(W)[r][c] x[b][c] in double, for rows [row0, row0+nrows)."""
    nrows = rows - row0 if nrows is None else nrows
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    batch = x.shape[0]
    assert x.shape[1] == cols
    w, wp = _c(w, np.uint8)
    y = np.empty((batch, nrows), dtype=np.float64)
    rc = _L().or_gemv(FMT[fmt], wp, rows, cols, x.ctypes.data, batch, row0, nrows, y.ctypes.data)
    if rc:
        raise ValueError(f"or_gemv rc={rc}")
    return y


def gemv_xd(fmt: str, w, rows: int, cols: int, x) -> np.ndarray:
    """The product over double activations x float64 [batch][cols] (the decode step's own
    intermediate vectors are double): y float64 [batch][rows]."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    batch = x.shape[0]
    assert x.shape[1] == cols
    w, wp = _c(w, np.uint8)
    y = np.empty((batch, rows), dtype=np.float64)
    rc = _L().or_gemv_xd(FMT[fmt], wp, rows, cols, x.ctypes.data, batch, 0, rows, y.ctypes.data)
    if rc:
        raise ValueError(f"or_gemv_xd rc={rc}")
    return y


def rmsnorm_d(x, g, eps: float) -> np.ndarray:
    """RMSNorm of one double vector (the step's own form): float64 [n]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    g, gp = _c(g, np.float32)
    assert g.size == x.size
    out = np.empty(x.size, dtype=np.float64)
    _L().or_rmsnorm_d(x.ctypes.data, gp, x.size, eps, out.ctypes.data)
    return out


def rope_d(v, n_heads: int, head_dim: int, pos: int, pairing: str, theta: float) -> np.ndarray:
    """RoPE of n_heads heads of a double vector (the step's own form): a rotated copy."""
    out = np.array(v, dtype=np.float64, copy=True)
    assert out.size == n_heads * head_dim and head_dim % 2 == 0 and pos >= 0
    for h in range(n_heads):
        _L().or_rope_head_d(out.ctypes.data + 8 * h * head_dim, head_dim, pos, PAIRING[pairing], theta)
    return out


def attention_d(q, k_cache, v_cache, n_heads: int, n_kv_heads: int, head_dim: int, n_pos: int,
                max_ctx: int) -> np.ndarray:
    """attention() over a double q (the step's own form)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k_cache, kp = _c(k_cache, np.float32)
    v_cache, vp = _c(v_cache, np.float32)
    assert q.size == n_heads * head_dim and n_heads % n_kv_heads == 0 and 0 < n_pos <= max_ctx
    assert k_cache.size >= n_kv_heads * max_ctx * head_dim and v_cache.size >= n_kv_heads * max_ctx * head_dim
    out = np.empty(n_heads * head_dim, dtype=np.float64)
    _L().or_attention_d(q.ctypes.data, kp, vp, n_heads, n_kv_heads, head_dim, n_pos, max_ctx, out.ctypes.data)
    return out


def rmsnorm(x, g, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    g, gp = _c(g, np.float32)
    out = np.empty(x.shape, dtype=np.float64)
    rc = _L().or_rmsnorm(x.ctypes.data, gp, x.shape[1], x.shape[0], eps, out.ctypes.data)
    if rc:
        raise ValueError(f"or_rmsnorm rc={rc}")
    return out


def rope(v, n_heads: int, head_dim: int, pos: int, pairing: str, theta: float) -> np.ndarray:
    v, vp = _c(v, np.float32)
    assert v.size == n_heads * head_dim
    out = np.empty(v.size, dtype=np.float64)
    rc = _L().or_rope(vp, n_heads, head_dim, pos, PAIRING[pairing], theta, out.ctypes.data)
    if rc:
        raise ValueError(f"or_rope rc={rc}")
    return out


def rope_table(theta: float, head_dim: int, ctx: int) -> np.ndarray:
    out = np.empty((ctx, head_dim // 2, 2), dtype=np.float32)
    rc = _L().or_rope_table(theta, head_dim, ctx, out.ctypes.data)
    if rc:
        raise ValueError(f"or_rope_table rc={rc}")
    return out


def attention(q, k_cache, v_cache, n_heads: int, n_kv_heads: int, head_dim: int, n_pos: int,
              max_ctx: int) -> np.ndarray:
    """q f32[n_heads*hd]; caches f32 [n_kv_heads][max_ctx][hd] for one layer/sequence."""
    q, qp = _c(q, np.float32)
    k_cache, kp = _c(k_cache, np.float32)
    v_cache, vp = _c(v_cache, np.float32)
    assert k_cache.size >= n_kv_heads * max_ctx * head_dim
    out = np.empty(n_heads * head_dim, dtype=np.float64)
    rc = _L().or_attention(qp, kp, vp, n_heads, n_kv_heads, head_dim, n_pos, max_ctx, out.ctypes.data)
    if rc:
        raise ValueError(f"or_attention rc={rc}")
    return out


def swiglu(g, u) -> np.ndarray:
    g, gp = _c(g, np.float32)
    u, up = _c(u, np.float32)
    out = np.empty(g.shape, dtype=np.float64)
    rc = _L().or_swiglu(gp, up, g.size, out.ctypes.data)
    if rc:
        raise ValueError(f"or_swiglu rc={rc}")
    return out


def round_f16(f: float) -> float:
    """f32 rounded through binary16 (what an f16 KV cache stores)."""
    return float(_L().or_round_f16(float(np.float32(f))))


def quantize_i4_rows(w_bf16, rows: int, cols: int) -> tuple[np.ndarray, np.ndarray]:
    """Per-row symmetric INT4 of BF16 weights (bit patterns, uint16 [rows][cols]):
    (codes uint8 [rows][cols/2], two per byte, scales f32 [rows]); see or_quantize_i4_rows."""
    w, wp = _c(np.asarray(w_bf16, np.uint16).reshape(-1), np.uint16)
    assert w.size == rows * cols
    codes = np.empty(rows * (cols // 2), np.uint8)
    scales = np.empty(rows, np.float32)
    rc = _L().or_quantize_i4_rows(wp, rows, cols, codes.ctypes.data, scales.ctypes.data)
    if rc:
        raise ValueError(f"or_quantize_i4_rows rc={rc}")
    return codes.reshape(rows, cols // 2), scales


def quantize_q8(x, with_sum: bool = False):
    """ggml-exact Q8_0 (Q8_1 with with_sum) activations of x f32 [batch][cols] (see
    or_quantize_q8): (codes int8 [batch][cols], d f32 [batch][cols/32], s or None), d and
    s holding their binary16 values."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    batch, cols = x.shape
    q = np.empty((batch, cols), np.int8)
    d = np.empty((batch, cols // 32), np.float32)
    s = np.empty((batch, cols // 32), np.float32) if with_sum else None
    for b in range(batch):
        rc = _L().or_quantize_q8(x[b].ctypes.data, cols, q[b].ctypes.data, d[b].ctypes.data,
                                 s[b].ctypes.data if with_sum else None)
        if rc:
            raise ValueError(f"or_quantize_q8 rc={rc}")
    return q, d, s


def gemv_q8act(fmt: str, w, rows: int, cols: int, xq, xd, xs=None, row0: int = 0, nrows: int | None = None):
    """The product over quantised activations (or_gemv_q8act), double [batch][nrows]."""
    nrows = rows - row0 if nrows is None else nrows
    xq = np.ascontiguousarray(np.atleast_2d(xq), dtype=np.int8)
    xd = np.ascontiguousarray(np.atleast_2d(xd), dtype=np.float32)
    batch = xq.shape[0]
    w, wp = _c(w, np.uint8)
    y = np.empty((batch, nrows), dtype=np.float64)
    xsp = None
    if xs is not None:
        xs = np.ascontiguousarray(np.atleast_2d(xs), dtype=np.float32)
        xsp = xs.ctypes.data
    rc = _L().or_gemv_q8act(FMT[fmt], wp, rows, cols, xq.ctypes.data, xd.ctypes.data, xsp, batch, row0, nrows,
                            y.ctypes.data)
    if rc:
        raise ValueError(f"or_gemv_q8act rc={rc}")
    return y


def quantize_i8_rows(w_bf16, rows: int, cols: int) -> tuple[np.ndarray, np.ndarray]:
    """Per-row symmetric INT8 of BF16 weights (bit patterns, uint16 [rows][cols]):
    (codes int8 [rows][cols], scales f32 [rows]); see or_quantize_i8_rows."""
    w, wp = _c(np.asarray(w_bf16, np.uint16).reshape(-1), np.uint16)
    assert w.size == rows * cols
    codes = np.empty(rows * cols, np.int8)
    scales = np.empty(rows, np.float32)
    rc = _L().or_quantize_i8_rows(wp, rows, cols, codes.ctypes.data, scales.ctypes.data)
    if rc != 0:
        raise ValueError("quantize_i8_rows: bad shape")
    return codes.reshape(rows, cols), scales


def silu(z: float) -> float:
    return float(_L().or_silu(z))


def argmax(v) -> int:
    v = np.ascontiguousarray(v)
    if v.dtype == np.float64:
        return int(_L().or_argmax_f64(v.ctypes.data, v.size))
    v = np.ascontiguousarray(v, dtype=np.float32)
    return int(_L().or_argmax_f32(v.ctypes.data, v.size))


class Model:
    """A llama-style model held as host tensors in model-file layouts (see qd_oracle.c)."""

    def __init__(self, cfg: dict, tensors: list):
        self.cfg = cfg
        self._keep = [np.ascontiguousarray(t) if t is not None else None for t in tensors]
        ptrs = [t.ctypes.data if t is not None else None for t in self._keep]
        self._ptrs = (ctypes.c_void_p * len(ptrs))(*ptrs)
        self._c = _Config(cfg["layers"], cfg["dim"], cfg["ffn"], cfg["n_heads"], cfg["n_kv_heads"],
                          cfg["head_dim"], cfg["vocab"], cfg["max_ctx"], cfg["rope_theta"], cfg["eps"],
                          PAIRING[cfg["pairing"]], FMT[cfg["w_fmt"]], FMT[cfg["emb_fmt"]],
                          1 if cfg.get("kv_f16") else 0, 1 if cfg.get("act_q8") else 0,
                          *[FMT[cfg.get(k, cfg["w_fmt"])] for k in ("qkv_fmt", "wo_fmt", "gate_up_fmt", "down_fmt")])

    def decode_step(self, k_cache: np.ndarray, v_cache: np.ndarray, layer_stride: int, pos: int,
                    token: int, seq_offset: int = 0):
        """One token for one sequence.  The caches are float32 arrays; this sequence's
        element (l, kvh, p, i) sits at seq_offset + l*layer_stride + (kvh*max_ctx+p)*hd + i.
        Writes the new k, v at ``pos``.  Returns (logits f64[vocab], argmax)."""
        assert k_cache.dtype == np.float32 and v_cache.dtype == np.float32
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        logits = np.empty(self.cfg["vocab"], dtype=np.float64)
        nxt = ctypes.c_int64()
        rc = _L().or_decode_step(ctypes.byref(self._c), self._ptrs, k_cache.ctypes.data + 4 * seq_offset,
                                 v_cache.ctypes.data + 4 * seq_offset, layer_stride, pos, token,
                                 logits.ctypes.data, ctypes.byref(nxt))
        if rc:
            raise ValueError(f"or_decode_step rc={rc}")
        return logits, int(nxt.value)


    def q8_slots(self) -> tuple[int, int]:
        """(slots, row length) of the step's quantised inputs in act_q8 mode: per layer the
        QKV input, the attention output, the feed-forward input and the SwiGLU output, then
        the head's input."""
        c = self.cfg
        return 4 * c["layers"] + 1, max(c["dim"], c["ffn"], c["n_heads"] * c["head_dim"])

    def decode_step_tf(self, k_cache: np.ndarray, v_cache: np.ndarray, layer_stride: int, pos: int, token: int,
                       kv_given: bool, seq_offset: int = 0, q8_codes=None, q8_d=None):
        """The step with the teacher-forcing hooks of or_decode_step_tf: with ``kv_given`` the
        caches already hold this step's k and v at ``pos`` (another implementation's values)
        and are not written; with ``q8_codes`` (int8 [slots][cols]) and ``q8_d`` (f32
        [slots][cols/32]) each quantised product (act_q8) multiplies those codes instead of
        its own (slots as in q8_slots()).  Returns (logits f64[vocab], argmax, kv f32
        [layers][2][n_kv*hd] as formed before any binary16 rounding, head input f32 [dim],
        the f32 input of every quantised product [slots][cols] or None without act_q8)."""
        assert k_cache.dtype == np.float32 and v_cache.dtype == np.float32
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        c = self.cfg
        kd = c["n_kv_heads"] * c["head_dim"]
        logits = np.empty(c["vocab"], dtype=np.float64)
        kv = np.empty((c["layers"], 2, kd), dtype=np.float32)
        hx = np.empty(c["dim"], dtype=np.float32)
        nxt = ctypes.c_int64()
        tf, xo = None, None
        if c.get("act_q8"):
            slots, cols = self.q8_slots()
            xo = np.zeros((slots, cols), np.float32)
            tf = _Q8TF(None, None, xo.ctypes.data, cols)
            if q8_codes is not None:
                qg = np.ascontiguousarray(q8_codes, dtype=np.int8).reshape(slots, cols)
                dg = np.ascontiguousarray(q8_d, dtype=np.float32).reshape(slots, cols // 32)
                tf.q_given, tf.d_given = qg.ctypes.data, dg.ctypes.data
        else:
            assert q8_codes is None
        rc = _L().or_decode_step_tf(ctypes.byref(self._c), self._ptrs, k_cache.ctypes.data + 4 * seq_offset,
                                    v_cache.ctypes.data + 4 * seq_offset, layer_stride, pos, token,
                                    logits.ctypes.data, ctypes.byref(nxt), 1 if kv_given else 0, kv.ctypes.data,
                                    hx.ctypes.data, ctypes.byref(tf) if tf is not None else None)
        if rc:
            raise ValueError(f"or_decode_step_tf rc={rc}")
        return logits, int(nxt.value), kv, hx, xo


def set_threads(n: int) -> int:
    """OpenMP threads for the oracle's loops (results do not depend on it); returns the count in use."""
    return int(_L().or_set_threads(int(n)))
