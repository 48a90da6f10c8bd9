"""Helpers for the GPU parity tests: device copies of seeded inputs, packing through the
C ABI, and the tolerance checks."""
import numpy as np
import torch

import qdsynth

# Tolerance for floating-point outputs: per output vector, max |gpu - oracle| <= TOL *
# max |oracle| (the bound the pages' Go oracle uses for logits, "Oracle tolerances").
TOL = 1e-3


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def packed(qd, fmt: str, src: np.ndarray, rows: int, cols: int) -> torch.Tensor:
    """Source-layout bytes -> packed device tensor through qd_repack."""
    s = dev(src.reshape(-1).view(np.uint8))
    out = torch.empty(qd.packed_bytes(fmt, rows, cols), dtype=torch.uint8, device="cuda")
    qd.repack(fmt, s, rows, cols, out)
    return out


def weights(qd, fmt, seed, name, rows, cols):
    src = qdsynth.weight_src(fmt, seed, name, rows, cols)
    return src, packed(qd, fmt, src, rows, cols)


def rel_err_rows(gpu: np.ndarray, ora: np.ndarray) -> np.ndarray:
    """Per leading-axis row: max |gpu - ora| / max |ora|."""
    g = np.atleast_2d(np.asarray(gpu, np.float64))
    o = np.atleast_2d(np.asarray(ora, np.float64))
    den = np.abs(o).max(axis=1)
    den[den == 0] = 1.0
    return np.abs(g - o).max(axis=1) / den


def assert_close(gpu, ora, tol=TOL, what=""):
    e = rel_err_rows(gpu, ora)
    assert np.all(np.isfinite(np.asarray(gpu, np.float64))), f"{what}: non-finite output"
    assert e.max() <= tol, f"{what}: max relative error {e.max():.3e} > {tol}"
    return float(e.max())
