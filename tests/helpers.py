"""Shared test utilities: device inputs, the oracle's expected values and the GEMM tolerance.

The tolerance is the one stated for this layer: per element
    |y - y_ref| <= 1e-3 * ||x_m||_2 * ||w_n||_2 + 1e-3,
with y_ref the fp64 oracle product (never rounded) and w_n the oracle's fp64
dequantized weight row.
"""
from __future__ import annotations

import numpy as np

import oracle


def row_norms_dequant(qw, s, zw, N, K, g, chunk=2048) -> np.ndarray:
    """||w_n||_2 of the oracle's dequantized rows, in row chunks to bound memory."""
    out = np.empty(N)
    for a in range(0, N, chunk):
        b = min(N, a + chunk)
        w = oracle.dequant(qw[a:b], s[a:b], zw[a:b], b - a, K, g)
        out[a:b] = np.linalg.norm(w, axis=1)
    return out


def gemm_tolerance(x_rows: np.ndarray, wnorm: np.ndarray) -> np.ndarray:
    xn = np.linalg.norm(x_rows.astype(np.float64), axis=1)
    return 1e-3 * xn[:, None] * wnorm[None, :] + 1e-3


def assert_within_tolerance(y_gpu_rows: np.ndarray, y_ref: np.ndarray, tol: np.ndarray, what: str = ""):
    yg = y_gpu_rows.astype(np.float64)
    assert np.isfinite(yg).all(), f"{what}: non-finite GEMM output"
    err = np.abs(yg - y_ref)
    bad = err > tol
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; first at (row {i}, n {j}): "
                             f"gpu {yg[i, j]!r} ref {y_ref[i, j]!r} tol {tol[i, j]!r}; "
                             f"max err/tol {float((err / tol).max()):.3g}")
    return float((err / tol).max())
