"""Pins of the oracle's dequantisers for the formats a Q4_K_M-class file mixes in (Q4_1,
Q5_0, Q5_K, Q6_K, F16; go-llm package overview, llamini "Quants", llmoxide 10).  The pages
name the formats; the byte layouts are the GGUF ones stated in qdecode.h.  Pinned by
hand-worked blocks (values worked out from the layout, written out literally below), by
identities with the already-pinned Q4_0 / Q4_K decoders, and by numpy's binary16 cast."""
import numpy as np

import oracle
import qdsynth


def _blk(*parts) -> np.ndarray:
    return np.frombuffer(b"".join(parts), dtype=np.uint8).copy()


def _f16(v: float) -> bytes:
    return np.array([v], np.float16).tobytes()


def _check(fmt, blk, cols, want, total):
    deq = oracle.dequant(fmt, blk, 1, cols)[0].astype(np.float64)
    assert np.array_equal(deq, np.asarray(want, np.float64)), (fmt, deq)
    y = oracle.gemv(fmt, blk, 1, cols, np.ones((1, cols), np.float32))
    assert y[0, 0] == total


def test_q4_1_hand_block():
    # d = 0.5, m = -1, code byte j = j | (15 - j) << 4: element j = 0.5 j - 1,
    # element j + 16 = 0.5 (15 - j) - 1
    blk = _blk(_f16(0.5), _f16(-1.0), bytes(j | ((15 - j) << 4) for j in range(16)))
    want = [-1.0, -0.5, 0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 3.0, 3.5, 4.0, 4.5, 5.0, 5.5, 6.0, 6.5,
            6.5, 6.0, 5.5, 5.0, 4.5, 4.0, 3.5, 3.0, 2.5, 2.0, 1.5, 1.0, 0.5, 0.0, -0.5, -1.0]
    _check("q4_1", blk, 32, want, 88.0)


def test_q5_0_hand_blocks():
    # d = 0.25; fifth bits of elements 0-15 set; low nibbles 0, high nibbles 3:
    # elements 0-15: q = 16 -> 0; elements 16-31: q = 3 -> -3.25
    blk = _blk(_f16(0.25), bytes([0xFF, 0xFF, 0x00, 0x00]), bytes([0x30] * 16))
    _check("q5_0", blk, 32, [0.0] * 16 + [-3.25] * 16, -52.0)
    # only bit 31 set; low nibbles 0, high nibbles 15: elements 0-15: q = 0 -> -4;
    # elements 16-30: q = 15 -> -0.25; element 31: q = 31 -> 3.75
    blk = _blk(_f16(0.25), bytes([0x00, 0x00, 0x00, 0x80]), bytes([0xF0] * 16))
    _check("q5_0", blk, 32, [-4.0] * 16 + [-0.25] * 15 + [3.75], -64.0)


def test_q5_k_hand_block():
    # d = 1, dmin = 0.5; scale bytes 0 and 4 = 1 and 2 (sub-block 0: sc 1, m 2), all other
    # sub-blocks sc = m = 0; every fifth-bit byte 0x01 (bit 0: sub-block 0); code bytes 0x73.
    # Sub-block 0 (elements 0-31): q = 3 + 16 = 19 -> 19 - 1 = 18; everything else 0.
    scales = bytes([1, 0, 0, 0, 2, 0, 0, 0, 0, 0, 0, 0])
    blk = _blk(_f16(1.0), _f16(0.5), scales, bytes([0x01] * 32), bytes([0x73] * 128))
    _check("q5_k", blk, 256, [18.0] * 32 + [0.0] * 224, 576.0)


def test_q6_k_hand_block():
    # d = 1, scales 1 except scale 9 = 3 and scale 15 = -2; code bytes 0 except
    # ql[0] = 0x21, ql[64] = 0x0F, qh[0] = 0b11100100.  Every element with q = 0 is -32 x
    # its scale; the exceptions:
    #   element 0   (half 0, quarter 0, l 0): low nibble of ql[0] = 1, qh bits 0-1 = 0 -> -31
    #   element 32  (quarter 1): low nibble of ql[32] = 0, qh bits 2-3 = 1 -> 16 - 32 = -16
    #   element 64  (quarter 2): high nibble of ql[0] = 2, qh bits 4-5 = 2 -> 34 - 32 = 2
    #   element 96  (quarter 3): high nibble of ql[32] = 0, qh bits 6-7 = 3 -> 48 - 32 = 16
    #   element 128 (half 1, quarter 0, l 0): low nibble of ql[64] = 15 -> -17
    #   elements 144-159 use scale 9 (= 3): -96; elements 240-255 scale 15 (= -2): 64
    ql = bytearray(128)
    ql[0], ql[64] = 0x21, 0x0F
    qh = bytearray(64)
    qh[0] = 0b11100100
    sc = [1] * 16
    sc[9], sc[15] = 3, -2
    blk = _blk(bytes(ql), bytes(qh), np.array(sc, np.int8).tobytes(), _f16(1.0))
    want = [-32.0] * 256
    want[0], want[32], want[64], want[96], want[128] = -31.0, -16.0, 2.0, 16.0, -17.0
    want[144:160] = [-96.0] * 16
    want[240:256] = [64.0] * 16
    _check("q6_k", blk, 256, want, -7566.0)


def test_f16_weights_match_numpy_cast():
    w = qdsynth.f16_weights(5, "f16w", 3, 40)
    want = w.reshape(3, 40, 2).view(np.float16)[..., 0].astype(np.float32)
    assert np.array_equal(oracle.dequant("f16", w.reshape(-1), 3, 40), want)


def _d(blocks, off):
    return blocks[:, :, off:off + 2].copy().view(np.float16)[..., 0].astype(np.float64)


def test_q5_0_all_fifth_bits_is_q4_0_plus_8d():
    rows, cols = 5, 256
    w5 = qdsynth.q5_0_blocks(6, "w5", rows, cols)
    w5[:, :, 2:6] = 0xFF
    w4 = np.concatenate([w5[:, :, 0:2], w5[:, :, 6:22]], axis=2)
    d = np.repeat(_d(w5, 0), 32, axis=1)
    got = oracle.dequant("q5_0", w5.reshape(-1), rows, cols).astype(np.float64)
    base = oracle.dequant("q4_0", w4.reshape(-1), rows, cols).astype(np.float64)
    assert np.array_equal(got, base + 8 * d)


def test_q5_k_without_fifth_bits_is_q4_k():
    rows, cols = 4, 512
    w5 = qdsynth.q5_k_blocks(7, "w5k", rows, cols)
    w5[:, :, 16:48] = 0
    w4 = np.concatenate([w5[:, :, 0:16], w5[:, :, 48:176]], axis=2)
    assert np.array_equal(oracle.dequant("q5_k", w5.reshape(-1), rows, cols),
                          oracle.dequant("q4_k", w4.reshape(-1), rows, cols))


def test_q4_1_with_m_minus_8d_is_q4_0():
    rows, cols = 6, 128
    w1 = qdsynth.q4_1_blocks(8, "w41", rows, cols)
    d = w1[:, :, 0:2].copy().view(np.float16)
    w1[:, :, 2:4] = (-8 * d).astype(np.float16).view(np.uint8)  # -8 d is exact in binary16
    w0 = np.concatenate([w1[:, :, 0:2], w1[:, :, 4:20]], axis=2)
    assert np.array_equal(oracle.dequant("q4_1", w1.reshape(-1), rows, cols),
                          oracle.dequant("q4_0", w0.reshape(-1), rows, cols))


def test_new_formats_row_slices():
    for fmt, cols in (("q4_1", 64), ("q5_0", 96), ("q5_k", 256), ("q6_k", 512), ("f16", 48)):
        rows = 9
        w = qdsynth.weight_src(fmt, 9, "sl" + fmt, rows, cols)
        full = oracle.dequant(fmt, w, rows, cols)
        assert np.array_equal(oracle.dequant(fmt, w, rows, cols, 3, 4), full[3:7])
        assert w.size == qdsynth.src_bytes(fmt, rows, cols)
