"""Shared test utilities: device inputs, the oracle's expected values and the GEMM tolerance.

The tolerance is the one stated for this layer: per element
    |y - y_ref| <= 1e-3 * ||x_m||_2 * ||w_n||_2 + 1e-3,
with y_ref the fp64 oracle product (never rounded) and w_n the oracle's fp64
dequantized weight row. For bf16 the same derivation -- one rounding of each
weight to the type, fp32 accumulation, one rounding of y, Cauchy-Schwarz --
with bf16's unit roundoff 2^-8 in place of fp16's 2^-11 gives
2 * 2^-8 = 7.8e-3 plus the fp32 summation term K * 2^-24 <= 2.0e-3 for
K <= 32768, so its coefficient is 1e-2.
"""
from __future__ import annotations

import numpy as np

import oracle


TOL_COEF = {"f16": 1e-3, "bf16": 1e-2}


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bits -> fp64 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def values_f64(a: np.ndarray, dtype: str = "f16") -> np.ndarray:
    """fp16 values, or uint16 bits of dtype, as fp64."""
    return bf16_bits_to_f64(a) if dtype == "bf16" else np.asarray(a).astype(np.float64)


def row_norms_dequant(qw, s, zw, N, K, g, chunk=2048, dtype: str = "f16") -> np.ndarray:
    """||w_n||_2 of the oracle's dequantized rows, in row chunks to bound memory."""
    out = np.empty(N)
    for a in range(0, N, chunk):
        b = min(N, a + chunk)
        w = oracle.dequant(qw[a:b], s[a:b], zw[a:b], b - a, K, g, dtype)
        out[a:b] = np.linalg.norm(w, axis=1)
    return out


def gemm_tolerance(x_rows: np.ndarray, wnorm: np.ndarray, dtype: str = "f16") -> np.ndarray:
    xn = np.linalg.norm(values_f64(x_rows, dtype), axis=1)
    return TOL_COEF[dtype] * xn[:, None] * wnorm[None, :] + 1e-3


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


def silu_mul_tolerance(y_ref: np.ndarray, tol_y: np.ndarray, dtype: str = "f16") -> np.ndarray:
    """Per-element bound for h = silu(gate) * up from the gate and up sums' bounds tol_y (columns 2j, 2j + 1).
    With |gate - gate_ref| <= eg and |up - up_ref| <= eu:
        |h - h_ref| <= L eg (|up_ref| + eu) + |silu(gate_ref)| eu + u |h_ref|,
    L = max |silu'| < 1.1 (mean value theorem), u the output's rounding (2^-11 fp16, 2^-8 bf16, doubled
    here for the fp32 evaluation of silu)."""
    g, up = y_ref[:, 0::2], y_ref[:, 1::2]
    eg, eu = tol_y[:, 0::2], tol_y[:, 1::2]
    h = oracle.silu(g) * up
    u = 2.0 ** -10 if dtype == "f16" else 2.0 ** -7
    return 1.1 * eg * (np.abs(up) + eu) + np.abs(oracle.silu(g)) * eu + u * np.abs(h) + 1e-6
