"""Output epilogues (silu(gate) * up, the q/k/v split by head group) and grouped GEMMs on the GPU,
against the oracle: the oracle's fp64 GEMM output put through its plain restatement of the epilogue
(oracle.silu_mul, oracle.qkv_split), within the per-element GEMM bound carried through the epilogue
(helpers.silu_mul_tolerance; the split only moves elements)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_group_quantized_gb300 as w4
import workloads
from helpers import (assert_within_tolerance, gemm_tolerance, row_norms_dequant, silu_mul_tolerance,
                     values_f64)

pytestmark = pytest.mark.gpu

_cache = {}


def layer(N, K, g, seed=0, dtype="f16"):
    """Seeded weights [N, K] through the oracle's pack, the GPU's repack of those buffers."""
    key = (N, K, g, seed, dtype)
    if key not in _cache:
        W = workloads.weights_bf16(N, K, seed=seed) if dtype == "bf16" else workloads.weights_f16(N, K, seed=seed)
        qw, s, zw = oracle.pack(W, g, dtype)
        st = torch.from_numpy(s.view(np.int16)).cuda()
        st = st.view(torch.bfloat16 if dtype == "bf16" else torch.float16)
        packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), st,
                              torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
        wn = row_norms_dequant(qw, s, zw, N, K, g, dtype=dtype)
        if len(_cache) > 8:
            _cache.clear()
        _cache[key] = (qw, s, zw, packed, wn)
    return _cache[key]


def acts(M, K, seed=1, dtype="f16", outliers=False):
    if dtype == "bf16":
        x = workloads.activations_bf16(M, K, seed=seed, outliers=outliers)
        return x, torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    x = workloads.activations_f16(M, K, seed=seed, outliers=outliers)
    return x, torch.from_numpy(x).cuda()


def host(t: torch.Tensor, dtype="f16") -> np.ndarray:
    if dtype == "bf16":
        return values_f64(t.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    return t.cpu().numpy().astype(np.float64)


def oracle_y(x, N, K, g, seed=0, rows=None, dtype="f16"):
    qw, s, zw, _, wn = layer(N, K, g, seed, dtype)
    rows = np.arange(x.shape[0]) if rows is None else rows
    return oracle.gemm(x, qw, s, zw, N, K, g, rows=rows, dtype=dtype), gemm_tolerance(x[rows], wn, dtype), rows


def check_silu(M, N, K, g, dtype="f16", **opts):
    _, _, _, packed, _ = layer(N, K, g, dtype=dtype)
    x, xd = acts(M, K, dtype=dtype)
    h = w4.w4a16_gemm_silu_mul(xd, packed, N, K, g, **opts)
    torch.cuda.synchronize()
    assert tuple(h.shape) == (M, N // 2)
    y_ref, tol, _ = oracle_y(x, N, K, g, dtype=dtype)
    assert_within_tolerance(host(h, dtype), oracle.silu_mul(y_ref), silu_mul_tolerance(y_ref, tol, dtype),
                            f"silu*up M={M} N={N} {dtype} {opts}")


def check_qkv(M, N, K, g, d, r, dtype="f16", rows=None, **opts):
    _, _, _, packed, _ = layer(N, K, g, dtype=dtype)
    x, xd = acts(M, K, dtype=dtype)
    q, k, v = w4.w4a16_gemm_qkv(xd, packed, N, K, g, d, r, **opts)
    torch.cuda.synchronize()
    y_ref, tol, rows = oracle_y(x, N, K, g, rows=rows, dtype=dtype)
    for got, want, t, name in zip((q, k, v), oracle.qkv_split(y_ref, d, r), oracle.qkv_split(tol, d, r), "qkv"):
        assert_within_tolerance(host(got, dtype)[rows], want, t, f"{name} M={M} N={N} d={d} r={r} {opts}")


# ------------------------------------------------------------------- silu(gate) * up

@pytest.mark.parametrize("M", [1, 3, 8, 16, 64, 130])
def test_silu_mul_gate_up_7b(M):
    # the fused 22016 x 4096 gate/up projection (rows interleaved): the decode kernel at M <= 8, the
    # tensor-memory kernel above (stream-K with cut tiles at 16 and 64, two token tiles at 130)
    check_silu(M, 22016, 4096, 128)


@pytest.mark.parametrize("opts", [dict(kernel=1, block_n=8, cluster=1), dict(kernel=1, block_n=8, cluster=4),
                                  dict(kernel=1, block_n=16, cluster=2), dict(kernel=2, block_n=16, ctas=7, schedule=1),
                                  dict(kernel=2, block_n=32, schedule=2), dict(kernel=2, block_n=128, ctas=5)],
                         ids=["dec_c1", "dec_c4", "dec16_c2", "tmem16_cut", "tmem32_whole", "tmem128_cut"])
@pytest.mark.parametrize("N,K,g", [(1000, 1024, 128), (258, 1032, 40)])
def test_silu_mul_schedules(opts, N, K, g):
    # every output path: the decode reducer, the tensor-memory epilogue of whole tiles and the owner's
    # fixup of cut tiles (N = 258: a last tile of two rows; g = 40: the rounded dequant)
    M = 8 if opts.get("block_n") == 8 else 16 if opts.get("kernel") == 1 else 19
    check_silu(M, N, K, g, **opts)


@pytest.mark.parametrize("M", [1, 8, 64])
def test_silu_mul_bf16(M):
    check_silu(M, 2048, 4096, 128, dtype="bf16")


# ------------------------------------------------------------------- q / k / v split

@pytest.mark.parametrize("M", [1, 8, 16, 64])
def test_qkv_split_7b_mha(M):
    # the fused 12288 x 4096 projection of 32 heads of 128: groups of (q, k, v) heads
    check_qkv(M, 12288, 4096, 128, 128, 1)


@pytest.mark.parametrize("M", [4, 512])
def test_qkv_split_70b_gqa(M):
    # 64 query heads over 8 key/value heads of 128: N = 8 * (8 + 2) * 128 = 10240
    rows = None if M <= 16 else np.unique(np.r_[0, M - 1, np.random.default_rng(0).choice(M, 6, replace=False)])
    check_qkv(M, 10240, 8192, 128, 128, 8, rows=rows)


@pytest.mark.parametrize("opts", [dict(kernel=1, block_n=8, cluster=2), dict(kernel=1, block_n=16),
                                  dict(kernel=2, block_n=16, ctas=9, schedule=1), dict(kernel=2, block_n=64)],
                         ids=["dec_c2", "dec16", "tmem16_cut", "tmem64"])
@pytest.mark.parametrize("d,r", [(4, 1), (12, 3), (64, 2)])
def test_qkv_split_head_shapes(opts, d, r):
    # heads that do not align with the 128-row tiles
    N = (r + 2) * d * max(1, 600 // ((r + 2) * d))
    M = 5 if opts.get("block_n") == 8 else 13
    check_qkv(M, N, 512, 64, d, r, **opts)


def test_qkv_split_bf16():
    check_qkv(8, 12288, 4096, 128, 128, 1, dtype="bf16")


# ------------------------------------------------------------------- grouped GEMMs

def run_group(M, specs, g=128, dtype="f16", **opts):
    """specs: (N, K, seed, x_key, kind) per problem; problems with the same x_key share x."""
    xs = {}
    problems = []
    for N, K, seed, xk, kind in specs:
        if (xk, K) not in xs:
            xs[(xk, K)] = acts(M, K, seed=10 + xk, dtype=dtype)
        _, _, _, packed, _ = layer(N, K, g, seed, dtype)
        pr = dict(x=xs[(xk, K)][1], packed=packed, N=N, K=K)
        if kind == "silu":
            pr["silu_mul"] = True
        elif kind == "qkv":
            pr["qkv"] = (128, 1)
        problems.append(pr)
    ws = w4.Workspace()
    outs = w4.w4a16_gemm_grouped(problems, g, workspace=ws, **opts)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0
    for (N, K, seed, xk, kind), out in zip(specs, outs):
        x = xs[(xk, K)][0]
        y_ref, tol, _ = oracle_y(x, N, K, g, seed, dtype=dtype)
        what = f"group M={M} N={N} K={K} {kind} {opts}"
        if kind == "silu":
            assert_within_tolerance(host(out, dtype), oracle.silu_mul(y_ref), silu_mul_tolerance(y_ref, tol, dtype),
                                    what)
        elif kind == "qkv":
            for got, want, t in zip(out, oracle.qkv_split(y_ref, 128, 1), oracle.qkv_split(tol, 128, 1)):
                assert_within_tolerance(host(got, dtype), want, t, what)
        else:
            assert_within_tolerance(host(out, dtype), y_ref, tol, what)


# one decoder layer's linears at M <= 8 in dependency order, as they would be grouped
LAYER_7B = [(4096, 4096, 1, 0, "y"), (4096, 4096, 2, 0, "y"), (4096, 4096, 3, 0, "y"),  # q, k, v: one x
            (4096, 4096, 4, 1, "y"),                                                       # o
            (11008, 4096, 5, 2, "y"), (11008, 4096, 6, 2, "y"),                            # gate, up: one x
            (4096, 11008, 7, 3, "y")]                                                      # down


@pytest.mark.parametrize("M", [1, 4, 8])
def test_group_of_a_decoder_layer(M):
    # every linear of a 7B decoder layer in one group: x shared by q, k, v and by gate, up; a change of
    # x and of K (down) between problems
    run_group(M, LAYER_7B)


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_group_cluster_sizes(cluster):
    run_group(4, [(4096, 4096, 1, 0, "y"), (1000, 4096, 2, 1, "y"), (300, 2048, 3, 2, "y"),
                  (4096, 11008, 4, 3, "y")], kernel=1, block_n=8, cluster=cluster)


def test_group_with_epilogues():
    run_group(4, [(12288, 4096, 1, 0, "qkv"), (4096, 4096, 2, 1, "y"), (22016, 4096, 3, 2, "silu"),
                  (4096, 11008, 4, 3, "y")])


def test_group_longer_than_one_launch():
    # 20 problems: two launches of the decode kernel (16 + 4 problems), each problem its own x
    run_group(2, [(256 + 128 * (i % 3), 512, 20 + i, i, "y") for i in range(20)])


def test_group_of_16_token_tiles_and_bf16():
    run_group(16, LAYER_7B[:4], dtype="bf16", kernel=1, block_n=16)


def test_group_above_decode_m_runs_one_launch_each():
    # M = 32: the tensor-memory kernel, one launch per problem, the same workspace reused in order
    run_group(32, LAYER_7B[:3] + [(22016, 4096, 5, 2, "silu")])


@pytest.mark.parametrize("M", [32, 64, 128, 200])
def test_group_sharing_x_runs_one_tensor_memory_launch(M):
    # q, k, v of one x above the decode kernel's range: one tensor-memory launch over their weight tiles
    run_group(M, LAYER_7B[:3])


@pytest.mark.parametrize("M", [24, 64])
def test_tensor_memory_group_with_epilogues(M):
    # a q/k/v split, a silu * up problem and a plain one on one x, each through its own epilogue
    run_group(M, [(12288, 4096, 1, 0, "qkv"), (22016, 4096, 3, 0, "silu"), (4096, 4096, 2, 0, "y")])


@pytest.mark.parametrize("opts", [dict(kernel=2, block_n=32, ctas=7, schedule=1),
                                  dict(kernel=2, block_n=64, ctas=5, schedule=1),
                                  dict(kernel=2, block_n=16, ctas=3, schedule=2),
                                  dict(kernel=2, block_n=128, ctas=0, schedule=0)],
                         ids=["bn32-streamk7", "bn64-streamk5", "bn16-whole3", "bn128-auto"])
@pytest.mark.parametrize("K,g", [(1024, 128), (1032, 40)])
def test_tensor_memory_group_ragged(opts, K, g):
    # ragged problems (partial last weight tiles) whose tiles follow one another; stream-K ranges that
    # cut tiles and cross from one problem into the next; g = 40 looks groups up per 8 codes, K = 1032
    # has a short last stage
    run_group(40, [(1000, K, 1, 0, "y"), (300, K, 2, 0, "y"), (130, K, 3, 0, "y"), (258, K, 4, 0, "silu")],
              g=g, **opts)


@pytest.mark.parametrize("count", [8, 9])
def test_tensor_memory_group_size_limit(count):
    # eight problems of one x fill the launch's problem table; a ninth sends the group back to one
    # launch per problem
    run_group(48, [(128 * (1 + i % 3) + 8 * i, 512, 30 + i, 0, "y") for i in range(count)])


def test_tensor_memory_group_bf16():
    run_group(64, LAYER_7B[:3] + [(11008, 4096, 5, 0, "y")], dtype="bf16")


def test_group_rejects_bad_epilogues_on_host():
    _, _, _, packed, _ = layer(1000, 1024, 128)
    x = torch.zeros((2, 1024), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):  # N not a multiple of (r + 2) d
        w4.w4a16_gemm_qkv(x, packed, 1000, 1024, 128, 128, 1)
    _, _, _, packed_odd, _ = layer(999, 1024, 128)
    with pytest.raises(w4.W4Error):  # silu * up needs N even
        w4.w4a16_gemm_silu_mul(x, packed_odd, 999, 1024, 128)
