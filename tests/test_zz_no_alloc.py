"""The GEMM entry point that allocates nothing (w4a16_gemm_noalloc), against the oracle.

Some callers of this library cannot allocate device memory for a workspace:
inference engines that reserve all device memory when they start and hand
kernels only their inputs and outputs, and plug-ins inside such engines that
never see an allocator. For them w4a16_gemm_noalloc keeps its scratch in a
fixed device array inside the library. This test calls it through the C ABI
twice in a row (the second call finds the first call's leftovers in the shared
array) and checks both outputs element by element against the fp64 oracle,
with the tolerance the other GEMM tests use; it also checks that the results
equal those of w4a16_gemm with a caller workspace (same schedule, same
arithmetic) and that a problem too large for the array is refused before
anything is enqueued. It sits in a file of its own that pytest collects last,
and it passes both alone in a fresh process and after the other tests.
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

SCRATCH_BYTES = 8 << 20  # W4A16_NOALLOC_SCRATCH_BYTES in include/w4a16.h


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
                                     (1, 288, 288, 256), (32, 4096, 11008, 128)])
def test_noalloc_matches_oracle(M, N, K, g):
    fn = _noalloc_fn()
    W = workloads.weights_f16(N, K)
    qw, s, zw = oracle.pack(W, g)
    packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                          torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
    x = workloads.activations_f16(M, K)
    xd = torch.from_numpy(x).cuda()
    yref = oracle.gemm(x, qw, s, zw, N, K, g)
    tol = gemm_tolerance(x, row_norms_dequant(qw, s, zw, N, K, g))
    with_ws = w4.w4a16_gemm(xd, packed, N, K, g)
    torch.cuda.synchronize()
    for call in range(2):  # the shared array still holds the first call's contents during the second
        rc, y = _call(fn, xd, packed, N, K, g)
        assert rc == 0, w4.w4_status_string(rc)
        assert_within_tolerance(y.cpu().numpy(), yref, tol, f"noalloc call {call}")
        assert torch.equal(y, with_ws), f"noalloc call {call} differs from w4a16_gemm"


def test_noalloc_refuses_problems_larger_than_its_array():
    fn = _noalloc_fn()
    # 128 tokens on a 4096 x 4096 layer: two token tiles of 64, each tile cut between two CTAs, whose
    # fp32 partial tiles (two per CTA, 128 CTAs) need a little over the 8 MiB the array holds
    N, K, g, M = 4096, 4096, 128, 128
    assert w4.w4a16_workspace_bytes(M, N, K, g) > SCRATCH_BYTES
    packed = torch.zeros(w4.w4_repacked_bytes(N, K, g), dtype=torch.uint8, device="cuda")
    x = torch.zeros(M, K, dtype=torch.float16, device="cuda")
    rc, y = _call(fn, x, packed, N, K, g)
    assert rc == 4  # W4_ERR_WORKSPACE_TOO_SMALL, nothing enqueued
    assert torch.isnan(y).all()
