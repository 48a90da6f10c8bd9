"""qdsynth — seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle's tests.

This module produces bytes and numbers only: GGUF-style block bytes filled with seeded
random fields, f32 activations, token ids and KV-cache contents.  It performs none of
the method's arithmetic (no dequantisation, no dot products); both the oracle and the
CUDA library consume exactly the bytes it writes.

Random streams are SplitMix64 (Steele, Lea & Flood 2014), counter-based, one stream per
named tensor (see ``qdsynth.c``).  f16 fields are drawn as doubles and rounded to binary16
with numpy's round-to-nearest-even conversion.

Block byte layouts written here (the model-file block layouts the pages load):
  * Q4_0 (18 B / 32 weights): f16 ``d`` at bytes 0-1, then 16 bytes of packed 4-bit codes.
    Every code uniform on 0..15 is the same as every code byte uniform on 0..255.
  * Q8_0 (34 B / 32 weights): f16 ``d`` at bytes 0-1, then 32 int8 codes uniform on -127..127.
  * Q4_K (144 B / 256 weights): f16 ``d``, f16 ``dmin``, 12 bytes of packed 6-bit
    scales/mins, 128 bytes of 4-bit codes; every byte of the last two fields uniform.
  * per-row INT8: int8 codes ``[rows][cols]`` uniform on -127..127, one f32 scale per row.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qdsynth.c")
_LIB_PATH = os.path.join(_HERE, "libqdsynth.so")
_lib = None

BLOCK_BYTES = {"q4_0": 18, "q8_0": 34, "q4_k": 144, "q4_1": 20, "q5_0": 22, "q5_k": 176, "q6_k": 210, "f16": 2}
BLOCK_WEIGHTS = {"q4_0": 32, "q8_0": 32, "q4_k": 256, "q4_1": 32, "q5_0": 32, "q5_k": 256, "q6_k": 256, "f16": 1}


def build(force: bool = False) -> str:
    """Compile libqdsynth.so next to its source (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        u64, i64, d = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
        p = ctypes.c_void_p
        lib.qs_stream.argtypes = [u64, ctypes.c_char_p]
        lib.qs_stream.restype = u64
        lib.qs_fill_u64.argtypes = [u64, u64, i64, p]
        lib.qs_fill_uniform_f64.argtypes = [u64, u64, i64, d, d, p]
        lib.qs_fill_uniform_f32.argtypes = [u64, u64, i64, d, d, p]
        lib.qs_fill_int_i32.argtypes = [u64, u64, i64, i64, i64, p]
        lib.qs_fill_int_u8.argtypes = [u64, u64, i64, i64, i64, p]
        lib.qs_fill_normal_f32.argtypes = [u64, u64, i64, p]
        _lib = lib
    return _lib


def stream(seed: int, name: str) -> int:
    return int(_L().qs_stream(seed & 0xFFFFFFFFFFFFFFFF, name.encode()))


def raw_u64(seed: int, name: str, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _L().qs_fill_u64(stream(seed, name), offset, n, out.ctypes.data)
    return out


def uniform_f64(seed, name, n, lo, hi, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    _L().qs_fill_uniform_f64(stream(seed, name), offset, n, lo, hi, out.ctypes.data)
    return out


def uniform_f32(seed, name, n, lo, hi, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _L().qs_fill_uniform_f32(stream(seed, name), offset, n, lo, hi, out.ctypes.data)
    return out


def normal_f32(seed, name, n, offset=0, out=None) -> np.ndarray:
    """Standard normals; ``out`` may be a preallocated float32 array (e.g. pinned memory)."""
    if out is None:
        out = np.empty(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    _L().qs_fill_normal_f32(stream(seed, name), offset, n, out.ctypes.data)
    return out


def ints_i32(seed, name, n, lo, hi, offset=0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _L().qs_fill_int_i32(stream(seed, name), offset, n, lo, hi, out.ctypes.data)
    return out


def ints_u8(seed, name, n, lo, hi, offset=0, out=None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.uint8)
    assert out.itemsize == 1 and out.flags.c_contiguous and out.size == n
    _L().qs_fill_int_u8(stream(seed, name), offset, n, lo, hi, out.ctypes.data)
    return out


def f16_bits_uniform(seed, name, n, lo, hi, offset=0) -> np.ndarray:
    """Uniform doubles on [lo, hi) rounded to binary16 (RNE); returned as uint16 bit patterns."""
    return uniform_f64(seed, name, n, lo, hi, offset).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------------------------------
# Block tensors (model-file layout).  ``row0``/``nrows`` select a slice of rows of the
# full tensor: the bytes of a slice equal the same rows of the full tensor.
# ---------------------------------------------------------------------------------------

D_RANGE = (0.002, 0.02)


def q4_0_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q4_0 tensor as uint8 ``[nrows][cols/32][18]``."""
    assert cols % 32 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 32
    out = np.empty((nrows, nb, 18), dtype=np.uint8)
    d = f16_bits_uniform(seed, name + ".d", nrows * nb, *D_RANGE, offset=row0 * nb)
    out[:, :, 0:2] = d.reshape(nrows, nb, 1).view(np.uint8).reshape(nrows, nb, 2)
    q = ints_u8(seed, name + ".qs", nrows * nb * 16, 0, 255, offset=row0 * nb * 16)
    out[:, :, 2:] = q.reshape(nrows, nb, 16)
    return out


def q8_0_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q8_0 tensor as uint8 ``[nrows][cols/32][34]`` (codes are int8 bytes)."""
    assert cols % 32 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 32
    out = np.empty((nrows, nb, 34), dtype=np.uint8)
    d = f16_bits_uniform(seed, name + ".d", nrows * nb, *D_RANGE, offset=row0 * nb)
    out[:, :, 0:2] = d.reshape(nrows, nb, 1).view(np.uint8).reshape(nrows, nb, 2)
    q = ints_u8(seed, name + ".qs", nrows * nb * 32, -127, 127, offset=row0 * nb * 32)
    out[:, :, 2:] = q.reshape(nrows, nb, 32)
    return out


def q4_k_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q4_K tensor as uint8 ``[nrows][cols/256][144]``."""
    assert cols % 256 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 256
    out = np.empty((nrows, nb, 144), dtype=np.uint8)
    d = f16_bits_uniform(seed, name + ".d", nrows * nb, *D_RANGE, offset=row0 * nb)
    dm = f16_bits_uniform(seed, name + ".dmin", nrows * nb, *D_RANGE, offset=row0 * nb)
    out[:, :, 0:2] = d.reshape(nrows, nb, 1).view(np.uint8).reshape(nrows, nb, 2)
    out[:, :, 2:4] = dm.reshape(nrows, nb, 1).view(np.uint8).reshape(nrows, nb, 2)
    sc = ints_u8(seed, name + ".scales", nrows * nb * 12, 0, 255, offset=row0 * nb * 12)
    out[:, :, 4:16] = sc.reshape(nrows, nb, 12)
    q = ints_u8(seed, name + ".qs", nrows * nb * 128, 0, 255, offset=row0 * nb * 128)
    out[:, :, 16:] = q.reshape(nrows, nb, 128)
    return out


def _f16_field(out, lo_byte, seed, name, nrows, nb, rng, row0):
    v = f16_bits_uniform(seed, name, nrows * nb, *rng, offset=row0 * nb)
    out[:, :, lo_byte:lo_byte + 2] = v.reshape(nrows, nb, 1).view(np.uint8).reshape(nrows, nb, 2)


def _byte_field(out, lo, hi, seed, name, nrows, nb, row0, vlo=0, vhi=255):
    n = hi - lo
    q = ints_u8(seed, name, nrows * nb * n, vlo, vhi, offset=row0 * nb * n)
    out[:, :, lo:hi] = q.reshape(nrows, nb, n)


M_RANGE = (-0.16, 0.0)  # Q4_1 block minimum (about -8 d, so values straddle 0)


def q4_1_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q4_1 tensor as uint8 ``[nrows][cols/32][20]``: d, m, 16 code bytes."""
    assert cols % 32 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 32
    out = np.empty((nrows, nb, 20), dtype=np.uint8)
    _f16_field(out, 0, seed, name + ".d", nrows, nb, D_RANGE, row0)
    _f16_field(out, 2, seed, name + ".m", nrows, nb, M_RANGE, row0)
    _byte_field(out, 4, 20, seed, name + ".qs", nrows, nb, row0)
    return out


def q5_0_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q5_0 tensor as uint8 ``[nrows][cols/32][22]``: d, 4 bytes of fifth bits, 16 code bytes."""
    assert cols % 32 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 32
    out = np.empty((nrows, nb, 22), dtype=np.uint8)
    _f16_field(out, 0, seed, name + ".d", nrows, nb, D_RANGE, row0)
    _byte_field(out, 2, 6, seed, name + ".qh", nrows, nb, row0)
    _byte_field(out, 6, 22, seed, name + ".qs", nrows, nb, row0)
    return out


def q5_k_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q5_K tensor as uint8 ``[nrows][cols/256][176]``: d, dmin, 12 scale bytes, 32 bytes
    of fifth bits, 128 code bytes."""
    assert cols % 256 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 256
    out = np.empty((nrows, nb, 176), dtype=np.uint8)
    _f16_field(out, 0, seed, name + ".d", nrows, nb, D_RANGE, row0)
    _f16_field(out, 2, seed, name + ".dmin", nrows, nb, D_RANGE, row0)
    _byte_field(out, 4, 16, seed, name + ".scales", nrows, nb, row0)
    _byte_field(out, 16, 48, seed, name + ".qh", nrows, nb, row0)
    _byte_field(out, 48, 176, seed, name + ".qs", nrows, nb, row0)
    return out


Q6K_D_RANGE = (0.0002, 0.002)  # d of a Q6_K super-block (scales are whole int8)


def q6_k_blocks(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """Q6_K tensor as uint8 ``[nrows][cols/256][210]``: 128 low-nibble bytes, 64 high-part
    bytes, 16 int8 scales, d."""
    assert cols % 256 == 0
    nrows = rows - row0 if nrows is None else nrows
    nb = cols // 256
    out = np.empty((nrows, nb, 210), dtype=np.uint8)
    _byte_field(out, 0, 192, seed, name + ".q", nrows, nb, row0)
    _byte_field(out, 192, 208, seed, name + ".scales", nrows, nb, row0, -127, 127)
    _f16_field(out, 208, seed, name + ".d", nrows, nb, Q6K_D_RANGE, row0)
    return out


def f16_weights(seed, name, rows, cols, row0=0, nrows=None) -> np.ndarray:
    """F16 tensor as uint8 ``[nrows][cols][2]``: values ~U[-1, 1) rounded to binary16."""
    nrows = rows - row0 if nrows is None else nrows
    v = f16_bits_uniform(seed, name, nrows * cols, -1.0, 1.0, offset=row0 * cols)
    return v.view(np.uint8).reshape(nrows, cols, 2)


I8_SCALE_RANGE = (1e-4, 1e-2)


def i8_row(seed, name, rows, cols, row0=0, nrows=None):
    """Per-row symmetric INT8: (codes int8 ``[nrows][cols]``, scales f32 ``[nrows]``)."""
    nrows = rows - row0 if nrows is None else nrows
    q = ints_u8(seed, name + ".q", nrows * cols, -127, 127, offset=row0 * cols).view(np.int8)
    s = uniform_f32(seed, name + ".s", nrows, *I8_SCALE_RANGE, offset=row0)
    return q.reshape(nrows, cols), s


def i8_row_src(seed, name, rows, cols) -> np.ndarray:
    """INT8 tensor as one byte buffer: codes ``[rows][cols]`` then f32 scales ``[rows]``."""
    q, s = i8_row(seed, name, rows, cols)
    return np.concatenate([q.reshape(-1).view(np.uint8), s.view(np.uint8)])


I4_SCALE_RANGE = (1e-3, 1e-1)


def i4_row_src(seed, name, rows, cols) -> np.ndarray:
    """Per-row INT4 tensor as one byte buffer: codes ``[rows][cols/2]`` (two nibbles per byte,
    values -7..7 in two's complement) then f32 scales ``[rows]``."""
    q = ints_u8(seed, name + ".q", rows * cols, -7, 7).reshape(rows, cols // 2, 2) & 0x0F
    packed = (q[:, :, 0] | (q[:, :, 1] << 4)).astype(np.uint8)
    s = uniform_f32(seed, name + ".s", rows, *I4_SCALE_RANGE)
    return np.concatenate([packed.reshape(-1), s.view(np.uint8)])


def weight_src(fmt: str, seed: int, name: str, rows: int, cols: int) -> np.ndarray:
    """Any format's tensor as the flat byte buffer both sides read."""
    if fmt == "q4_0":
        return q4_0_blocks(seed, name, rows, cols).reshape(-1)
    if fmt == "q8_0":
        return q8_0_blocks(seed, name, rows, cols).reshape(-1)
    if fmt == "q4_k":
        return q4_k_blocks(seed, name, rows, cols).reshape(-1)
    if fmt == "i8":
        return i8_row_src(seed, name, rows, cols)
    if fmt == "i4":
        return i4_row_src(seed, name, rows, cols)
    gen = {"q4_1": q4_1_blocks, "q5_0": q5_0_blocks, "q5_k": q5_k_blocks, "q6_k": q6_k_blocks,
           "f16": f16_weights}.get(fmt)
    if gen is None:
        raise ValueError(fmt)
    return gen(seed, name, rows, cols).reshape(-1)


def src_bytes(fmt: str, rows: int, cols: int) -> int:
    if fmt == "i8":
        return rows * cols + 4 * rows
    if fmt == "i4":
        return rows * cols // 2 + 4 * rows
    return rows * (cols // BLOCK_WEIGHTS[fmt]) * BLOCK_BYTES[fmt]


def activations(seed, name, batch, n) -> np.ndarray:
    """x ~ N(0,1), float32 ``[batch][n]``."""
    return normal_f32(seed, name, batch * n).reshape(batch, n)


def tokens(seed, name, n, vocab) -> np.ndarray:
    return ints_i32(seed, name, n, 0, vocab - 1)


def norm_gains(seed, name, n) -> np.ndarray:
    """RMSNorm gains ~U[0.9, 1.1] (float32)."""
    return uniform_f32(seed, name, n, 0.9, 1.1)


# ---------------------------------------------------------------------------------------
# Synthetic llama-style models.  Tensor order (shared interface of the oracle and the
# library's model loader): [0] token embedding (emb_fmt, vocab x dim), [1] output norm
# gains f32[dim], [2] output head or None when tied, then per layer l at 3 + 9l:
# attn_norm, wq, wk, wv, wo, ffn_norm, wg, wu, wd.
# ---------------------------------------------------------------------------------------

SMOL_135M = dict(layers=30, dim=576, ffn=1536, n_heads=9, n_kv_heads=3, head_dim=64, vocab=49152,
                 rope_theta=1e5, eps=1e-5, pairing="half", w_fmt="q4_0", emb_fmt="q8_0")
SMOL_1_7B = dict(layers=24, dim=2048, ffn=8192, n_heads=32, n_kv_heads=32, head_dim=64, vocab=49152,
                 rope_theta=1e5, eps=1e-5, pairing="half", w_fmt="i8", emb_fmt="i8")


def layer_shapes(cfg: dict):
    """(name suffix, rows, cols) of the seven matrices of one layer."""
    D, F = cfg["dim"], cfg["ffn"]
    QD, KD = cfg["n_heads"] * cfg["head_dim"], cfg["n_kv_heads"] * cfg["head_dim"]
    return [("wq", QD, D), ("wk", KD, D), ("wv", KD, D), ("wo", D, QD),
            ("wg", F, D), ("wu", F, D), ("wd", D, F)]


# The class of each layer matrix and the config key of its format (a mixed model names
# them; otherwise every matrix takes w_fmt).
MATRIX_CLASS = {"wq": "qkv_fmt", "wk": "qkv_fmt", "wv": "qkv_fmt", "wo": "wo_fmt", "wg": "gate_up_fmt",
                "wu": "gate_up_fmt", "wd": "down_fmt"}


def matrix_fmt(cfg: dict, name: str) -> str:
    """The format of layer matrix `name` (wq .. wd) in a model config."""
    return cfg.get(MATRIX_CLASS[name], cfg["w_fmt"])


def model_tensors(cfg: dict, seed: int, tied: bool = True) -> list:
    """All tensors of a synthetic model as flat numpy arrays, in the order above."""
    D = cfg["dim"]
    t = [weight_src(cfg["emb_fmt"], seed, "tok_emb", cfg["vocab"], D),
         norm_gains(seed, "out_norm", D),
         None if tied else weight_src(cfg["emb_fmt"], seed, "head", cfg["vocab"], D)]
    shapes = dict((n, (r, c)) for n, r, c in layer_shapes(cfg))
    for l in range(cfg["layers"]):
        p = f"blk{l}."
        for name in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd"):
            if name.endswith("norm"):
                t.append(norm_gains(seed, p + name, D))
            else:
                r, c = shapes[name]
                t.append(weight_src(matrix_fmt(cfg, name), seed, p + name, r, c))
    return t


def model_weight_src_bytes(cfg: dict, tied: bool = True) -> int:
    """Bytes of all model-file-layout weight tensors (norm gains included)."""
    D = cfg["dim"]
    n = src_bytes(cfg["emb_fmt"], cfg["vocab"], D) * (1 if tied else 2) + 4 * D
    per = sum(src_bytes(matrix_fmt(cfg, n), r, c) for n, r, c in layer_shapes(cfg)) + 8 * D
    return n + cfg["layers"] * per
