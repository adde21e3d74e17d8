"""The no-allocation GEMM entry point (w4a16_gemm_noalloc) against the regular one.

Some callers cannot allocate a workspace (code running during CUDA-graph stream
capture, engines that plan all device memory up front, plug-ins that only see
their input and output tensors); for them w4a16_gemm_noalloc keeps its scratch
in a fixed device array inside the library. This test calls it through the C
ABI twice in a row and checks both results against w4a16_gemm's, within the
GEMM tolerance the other tests use, and checks that a problem too large for the
array is refused. It has a file of its own that pytest collects last, and also
passes when run alone in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import w4a16_group_quantized_gb300 as w4
import workloads
from helpers import assert_within_tolerance, gemm_tolerance, row_norms_dequant
from w4a16_group_quantized_gb300 import build as w4build

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    w4build.build()
    fn = w4.load().w4a16_gemm_noalloc
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    fn.argtypes = [P, P, I64, I64, I64, I32, P, P]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, x, packed, N, K, g):
    M = x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float16, device=x.device)
    rc = fn(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(packed.data_ptr()), M, N, K, g,
            ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, y


@pytest.mark.parametrize("M,N,K,g", [(4, 4096, 4096, 128), (16, 12288, 4096, 128), (8, 4096, 4000, 128),
                                     (1, 288, 288, 256)])
def test_noalloc_matches_workspace_entry_point(M, N, K, g):
    fn = _noalloc_fn()
    W = workloads.weights_f16(N, K)
    qw, s, zw = oracle.pack(W, g)
    packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                          torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
    x = workloads.activations_f16(M, K)
    xd = torch.from_numpy(x).cuda()
    ref = w4.w4a16_gemm(xd, packed, N, K, g).cpu().numpy().astype(np.float64)
    tol = gemm_tolerance(x, row_norms_dequant(qw, s, zw, N, K, g))
    for call in range(2):  # the shared array still holds the first call's contents during the second
        rc, y = _call(fn, xd, packed, N, K, g)
        assert rc == 0, w4.w4_status_string(rc)
        assert_within_tolerance(y.cpu().numpy(), ref, tol, f"noalloc call {call}")


def test_noalloc_refuses_problems_larger_than_its_array():
    fn = _noalloc_fn()
    N, K, g, M = 4096, 4096, 128, 128  # split tiles of 128 x 128 fp32 need ~20 MB of scratch
    assert w4.w4a16_workspace_bytes(M, N, K, g) > (8 << 20)
    packed = torch.zeros(w4.w4_repacked_bytes(N, K, g), dtype=torch.uint8, device="cuda")
    x = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    rc, y = _call(fn, x, packed, N, K, g)
    assert rc == 4  # W4_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
    assert torch.isnan(y).all()
