"""bf16 activations, scales and outputs, and symmetric (z = 8) weights, on the GPU against the oracle.

Same structure as the fp16 GEMM tests: the oracle packs the seeded bf16 weights, the GPU repacks the
canonical buffers, and every checked element must satisfy the per-element bound
    |y - y_ref| <= 1e-2 * ||x_m|| * ||w_n|| + 1e-3        (bf16; helpers.TOL_COEF)
against the oracle's fp64 product of the bf16 inputs. One-hot rows must return bf16(w) bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_group_quantized_gb300 as w4
import workloads
from helpers import assert_within_tolerance, bf16_bits_to_f64, gemm_tolerance, row_norms_dequant

pytestmark = pytest.mark.gpu

_cache = {}


def layer_bf16(N, K, g, symmetric=False, seed=0):
    key = (N, K, g, symmetric, seed)
    if key not in _cache:
        W = workloads.weights_bf16(N, K, seed=seed)
        qw, s, zw = oracle.pack(W, g, "bf16", symmetric)
        packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(),
                              torch.from_numpy(s.view(np.int16)).cuda().view(torch.bfloat16),
                              torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
        wn = row_norms_dequant(qw, s, zw, N, K, g, dtype="bf16")
        if len(_cache) > 6:
            _cache.clear()
        _cache[key] = (qw, s, zw, packed, wn)
    return _cache[key]


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def from_dev_bf16(t: torch.Tensor) -> np.ndarray:
    assert t.dtype == torch.bfloat16
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_bf16(M, N, K, g, rows=None, outliers=False, symmetric=False, seed_x=1, **opts):
    qw, s, zw, packed, wn = layer_bf16(N, K, g, symmetric)
    x = workloads.activations_bf16(M, K, seed=seed_x, outliers=outliers)
    ws = w4.Workspace()
    if opts:
        y = w4.w4a16_gemm_opts(to_dev_bf16(x), packed, N, K, g, workspace=ws, **opts)
    else:
        y = w4.w4a16_gemm(to_dev_bf16(x), packed, N, K, g, workspace=ws)
    torch.cuda.synchronize()
    assert y.dtype == torch.bfloat16
    assert w4.w4_last_device_error(ws) == 0
    if rows is None:
        rows = np.arange(M)
    yref = oracle.gemm(x, qw, s, zw, N, K, g, rows=rows, dtype="bf16")
    yg = bf16_bits_to_f64(from_dev_bf16(y)[rows])
    tol = gemm_tolerance(x[rows], wn, "bf16")
    return assert_within_tolerance(yg, yref, tol, f"bf16 M={M} N={N} K={K} g={g} sym={symmetric} {opts}")


def _sample_rows(M, k, seed=0):
    if M <= k:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, k - 2, replace=False)]))


def test_tiny_config_bf16():
    check_bf16(4, 256, 512, 128)


@pytest.mark.parametrize("M", [1, 8, 64])
@pytest.mark.parametrize("L", workloads.PARTIAL_LAYERS, ids=lambda L: L.name)
def test_partial_last_group_bf16(M, L):
    check_bf16(M, L.n, L.k, L.g)


@pytest.mark.parametrize("L", workloads.DECODE_LAYERS, ids=lambda L: L.name)
def test_decode_sweep_bf16(L):
    for M in workloads.DECODE_MS:
        check_bf16(M, L.n, L.k, L.g, rows=_sample_rows(M, 16))


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16, 17, 33, 64, 100, 128, 257])
def test_tile_edges_bf16(M):
    check_bf16(M, 1000, 1000 // 8 * 8, 128)


@pytest.mark.parametrize("g", [8, 24, 64, 128, 192, 256, 1024])
@pytest.mark.parametrize("kernel,M", [(1, 4), (1, 16), (2, 16), (2, 128)], ids=["dec8", "dec16", "tmem16", "tmem128"])
def test_group_modes_both_kernels_bf16(g, kernel, M):
    # every dequant mode (integer path for g % 64 == 0 on the decode kernel, rounded per 8 codes
    # otherwise and on the tensor-memory kernel) in bf16
    opts = dict(kernel=kernel)
    if kernel == 1:
        opts["block_n"] = 8 if M <= 8 else 16
    check_bf16(M, 700, 960, g, **opts)


@pytest.mark.parametrize("M,N,K", [(512, 8192, 8192), (1024, 10240, 8192)])
def test_prefill_sampled_bf16(M, N, K):
    check_bf16(M, N, K, 128, rows=_sample_rows(M, 8), outliers=True)


@pytest.mark.parametrize("opts", [dict(kernel=1, block_n=8), dict(kernel=1, block_n=16),
                                  dict(kernel=2, block_n=16), dict(kernel=2, block_n=128)],
                         ids=["dec8", "dec16", "tmem16", "tmem128"])
@pytest.mark.parametrize("g", [128, 40])
def test_one_hot_rows_return_bf16_weights_exactly(opts, g):
    # x row m is the unit vector e_{k_m}: y[m, n] = bf16_RN(w[n, k_m]) exactly (the product by one and
    # the fp32 sum are exact, and (q - z) * s is rounded once either way)
    N, K = 300, 320
    qw, s, zw, packed, _ = layer_bf16(N, K, g)
    M = 8 if opts["block_n"] <= 8 else 16
    ks = np.array([0, 1, 63, 64, 127, 200, 319, 255, 5, 77, 128, 129, 256, 300, 318, 31])[:M]
    x = np.zeros((M, K), np.uint16)
    x[np.arange(M), ks] = 0x3F80  # bf16 1.0
    y = w4.w4a16_gemm_opts(to_dev_bf16(x), packed, N, K, g, **opts)
    torch.cuda.synchronize()
    w = oracle.dequant(qw, s, zw, N, K, g, "bf16")
    want = np.array([[oracle.double_to_bf16(v) for v in w[:, k]] for k in ks], dtype=np.uint16)
    assert (from_dev_bf16(y) == want).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("M", [1, 8, 16, 64, 128])
def test_symmetric_weights(dtype, M):
    # symmetric packing: z = 8 in every group; the GEMM reads the zeros like any other
    N, K, g = 4096, 4000, 128
    if dtype == "bf16":
        check_bf16(M, N, K, g, rows=_sample_rows(M, 16), symmetric=True)
        return
    W = workloads.weights_f16(N, K)
    qw, s, zw = oracle.pack(W, g, "f16", True)
    packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                          torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
    x = workloads.activations_f16(M, K)
    y = w4.w4a16_gemm(torch.from_numpy(x).cuda(), packed, N, K, g).cpu().numpy()
    rows = _sample_rows(M, 16)
    yref = oracle.gemm(x, qw, s, zw, N, K, g, rows=rows)
    tol = gemm_tolerance(x[rows], row_norms_dequant(qw, s, zw, N, K, g))
    assert_within_tolerance(y[rows], yref, tol, f"symmetric f16 M={M}")


@pytest.mark.parametrize("symmetric", [False, True])
def test_end_to_end_from_bf16_weights(symmetric):
    # GPU pack -> GPU repack -> GEMM, against the oracle's pack of the same bf16 weights
    N, K, g, M = 2048, 4096, 128, 8
    W = workloads.weights_bf16(N, K, seed=5)
    qw, s, zw = w4.w4_pack(to_dev_bf16(W), g, symmetric=symmetric)
    packed = w4.w4_repack(qw, s, zw, N, K, g)
    x = workloads.activations_bf16(M, K)
    y = w4.w4a16_gemm(to_dev_bf16(x), packed, N, K, g)
    torch.cuda.synchronize()
    oq, os_, oz = oracle.pack(W, g, "bf16", symmetric)
    yref = oracle.gemm(x, oq, os_, oz, N, K, g, dtype="bf16")
    tol = gemm_tolerance(x, row_norms_dequant(oq, os_, oz, N, K, g, dtype="bf16"), "bf16")
    assert_within_tolerance(bf16_bits_to_f64(from_dev_bf16(y)), yref, tol, f"end to end bf16 sym={symmetric}")


def test_dtype_mismatch_rejected_on_host():
    N, K, g = 256, 512, 128
    _, _, _, packed, _ = layer_bf16(N, K, g)
    x = torch.zeros((4, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        w4.w4a16_gemm(x, packed, N, K, g, y=torch.empty((4, N), dtype=torch.float16, device="cuda"))
