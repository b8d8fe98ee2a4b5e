"""Shared pieces of the GPU parity tests: seeded cases on the device, the
oracle on the host, row sampling for the largest shapes, the tolerance check.

Tolerance: for every token t, max_r |gpu[t][r] - oracle[t][r]| must be at most
1e-4 of the L2 norm of the oracle's output row oracle[t][:].  The GPU sums the
same exact integer dots in fp32 (in a different order) while the oracle sums
in f64, so only rounding separates them; 1e-4 of the row norm leaves a wide
margin (observed errors are ~1e-7 of the norm).
"""
from __future__ import annotations

import numpy as np

import oracle

REL_TOL = 1e-4
_ORA = None


def ora():
    global _ORA
    if _ORA is None:
        _ORA = oracle.Oracle()
    return _ORA


def threads():
    return oracle.default_threads()


def dev(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def row_sample(od: int, max_rows: int = 2048) -> np.ndarray:
    """All rows when od is small; else the first and last 128 rows (the
    ragged tail included) and an evenly spread subset."""
    if od <= max_rows:
        return np.arange(od)
    step = max(1, (od - 256) // (max_rows - 256))
    mid = np.arange(128, od - 128, step)
    return np.unique(np.concatenate([np.arange(128), mid, np.arange(od - 128, od)]))


def oracle_rows(qtype, W, x, rows):
    """Oracle output restricted to the given weight rows: [nt][len(rows)]."""
    Wsub = np.ascontiguousarray(W[rows])
    return ora().matmul(qtype, Wsub, x, len(rows), nthreads=threads())


def assert_close_rows(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), what
    norm = np.linalg.norm(ref.astype(np.float64), axis=1)
    err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64)).max(axis=1)
    rel = err / np.maximum(norm, 1e-30)
    if not (rel <= REL_TOL).all():
        full = np.abs(gpu.astype(np.float64) - ref.astype(np.float64)) / np.maximum(norm, 1e-30)[:, None]
        bt, br = np.nonzero(full > REL_TOL)
        raise AssertionError(
            f"{what}: worst row error {rel.max():.3e} of the row norm; {len(bt)} outputs off, "
            f"tokens {np.unique(bt)[:12].tolist()} ({len(np.unique(bt))}), columns {np.unique(br)[:12].tolist()} "
            f"({len(np.unique(br))}), column tiles of 128: {np.unique(br // 128)[:12].tolist()}")
    return float(rel.max())
