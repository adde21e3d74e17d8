"""The bounded waits' timeout path, on the GPU, without a fault.

Every pipeline wait in the kernels gives up after a limit, raises the CTA's
abort flag and the workspace error word, drains its own copies and returns.
W4_FLAG_TEST_TIMEOUT makes one wait expect more than will ever come (the decode
kernel's reducer a few bytes more, the tensor-memory kernel's owner of a cut
tile one piece more); with a short limit the kernel must return early, leave
the device usable and report W4_ERR_TIMEOUT through w4_last_device_error; the
next call on the zeroed workspace must match the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_group_quantized_gb300 as w4
import workloads
from helpers import assert_within_tolerance, gemm_tolerance, row_norms_dequant

pytestmark = pytest.mark.gpu

W4_ERR_TIMEOUT = 6
SHORT_LIMIT = 2_000_000  # clock cycles: about a millisecond


@pytest.mark.parametrize("opts", [
    dict(kernel=1, block_n=8, cluster=4),          # decode kernel, K split across a cluster of 4
    dict(kernel=1, block_n=8, cluster=1),          # decode kernel, whole tiles
    dict(kernel=1, block_n=16, cluster=2, ctas=3),  # 16-token tiles, several tiles per cluster
    dict(kernel=2, block_n=16, ctas=5, schedule=1),  # tensor-memory kernel, stream-K with cut tiles
], ids=["dec_c4", "dec_c1", "dec16_c2", "tmem_streamk"])
def test_wait_runs_out_then_next_call_is_correct(opts):
    N, K, g = 1000, 2048, 128
    M = 4 if opts["block_n"] == 8 else 12
    W = workloads.weights_f16(N, K)
    qw, s, zw = oracle.pack(W, g)
    packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                          torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
    x = workloads.activations_f16(M, K)
    xd = torch.from_numpy(x).cuda()
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")

    w4.w4a16_gemm_opts(xd, packed, N, K, g, flags=w4.FLAG_TEST_TIMEOUT, wait_limit_cycles=SHORT_LIMIT,
                       workspace=ws, **opts)
    torch.cuda.synchronize()  # the kernel came back: no hang, no fault
    assert w4.w4_last_device_error(ws) == W4_ERR_TIMEOUT

    ws.zero_()  # a timeout leaves the tile counters undefined
    y = w4.w4a16_gemm_opts(xd, packed, N, K, g, workspace=ws, **opts)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0
    yref = oracle.gemm(x, qw, s, zw, N, K, g)
    assert_within_tolerance(y.cpu().numpy(), yref, gemm_tolerance(x, row_norms_dequant(qw, s, zw, N, K, g)),
                            f"after timeout {opts}")


def test_grouped_wait_runs_out_then_next_call_is_correct():
    # two problems with different x: the decode kernel reloads x between them (the consumers' x_free wait)
    g, M = 128, 4
    specs = [(1000, 2048, 0), (700, 1024, 1)]
    data = []
    for N, K, seed in specs:
        W = workloads.weights_f16(N, K, seed=seed)
        qw, s, zw = oracle.pack(W, g)
        packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                              torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
        x = workloads.activations_f16(M, K, seed=seed + 5)
        data.append((N, K, qw, s, zw, packed, x, torch.from_numpy(x).cuda()))
    problems = [dict(x=xd, packed=packed, N=N, K=K) for N, K, _, _, _, packed, _, xd in data]
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    w4.w4a16_gemm_grouped(problems, g, kernel=1, block_n=8, flags=w4.FLAG_TEST_TIMEOUT,
                          wait_limit_cycles=SHORT_LIMIT, workspace=ws)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == W4_ERR_TIMEOUT
    ws.zero_()
    outs = w4.w4a16_gemm_grouped(problems, g, kernel=1, block_n=8, workspace=ws)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0
    for (N, K, qw, s, zw, _, x, _), y in zip(data, outs):
        yref = oracle.gemm(x, qw, s, zw, N, K, g)
        assert_within_tolerance(y.cpu().numpy(), yref, gemm_tolerance(x, row_norms_dequant(qw, s, zw, N, K, g)),
                                "grouped, after timeout")
