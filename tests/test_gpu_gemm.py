"""w4a16_gemm on the GPU against the fp64 CPU oracle.

Tolerance per element: |y - y_ref| <= 1e-3 * ||x_m|| * ||w_n|| + 1e-3 (y_ref
and w_n from the oracle). Small cases compare every element; the full-size
layers compare every row the oracle can afford plus sampled rows, in the same
launch configuration the bench times (automatic tiling)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_group_quantized_gb300 as w4
import workloads
from helpers import assert_within_tolerance, gemm_tolerance, row_norms_dequant

pytestmark = pytest.mark.gpu

_cache = {}


def layer(N, K, g, seed=0):
    """Oracle canonical form of a seeded layer and its GPU tile layout (via the oracle's canonical buffers)."""
    key = (N, K, g, seed)
    if key not in _cache:
        W = workloads.weights_f16(N, K, seed=seed)
        qw, s, zw = oracle.pack(W, g)
        packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                              torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
        wn = row_norms_dequant(qw, s, zw, N, K, g)
        if len(_cache) > 6:
            _cache.clear()
        _cache[key] = (qw, s, zw, packed, wn)
    return _cache[key]


def run_gemm(x, packed, N, K, g, block_n=0, ctas=0, schedule=0, ws=None):
    xd = torch.from_numpy(x).cuda()
    if block_n or ctas or schedule:
        y = w4.w4a16_gemm_ex(xd, packed, N, K, g, block_n, ctas, schedule, workspace=ws)
    else:
        y = w4.w4a16_gemm(xd, packed, N, K, g, workspace=ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(M, N, K, g, block_n=0, ctas=0, schedule=0, rows=None, outliers=False, seed_x=1):
    qw, s, zw, packed, wn = layer(N, K, g)
    x = workloads.activations_f16(M, K, seed=seed_x, outliers=outliers)
    ws = w4.Workspace()
    y = run_gemm(x, packed, N, K, g, block_n, ctas, schedule, ws)
    assert w4.w4_last_device_error(ws) == 0
    if rows is None:
        rows = np.arange(M)
    yref = oracle.gemm(x, qw, s, zw, N, K, g, rows=rows)
    tol = gemm_tolerance(x[rows], wn)
    return assert_within_tolerance(y[rows], yref, tol,
                                   f"M={M} N={N} K={K} g={g} bn={block_n} ctas={ctas} schedule={schedule}")


def _dec_clusters(K, M):
    """Cluster sizes the decode kernel takes for this K and M: at most the number of 256-wide K stages,
    and enough CTAs that each one's K range of x (M rows of 512 bytes per stage, at most 48 stages)
    fits its 96 KB of shared memory."""
    stages = -(-K // 256)
    per_cta_max = min(48, 96 * 1024 // (512 * M))
    return [c for c in (1, 2, 4, 8) if c <= stages and -(-stages // c) <= per_cta_max]


def check_opts(M, N, K, g, rows=None, outliers=False, seed_x=1, **opts):
    """As check, through w4a16_gemm_opts with the given options."""
    qw, s, zw, packed, wn = layer(N, K, g)
    x = workloads.activations_f16(M, K, seed=seed_x, outliers=outliers)
    ws = w4.Workspace()
    y = w4.w4a16_gemm_opts(torch.from_numpy(x).cuda(), packed, N, K, g, workspace=ws, **opts)
    torch.cuda.synchronize()
    assert w4.w4_last_device_error(ws) == 0
    if rows is None:
        rows = np.arange(M)
    yref = oracle.gemm(x, qw, s, zw, N, K, g, rows=rows)
    tol = gemm_tolerance(x[rows], wn)
    return assert_within_tolerance(y.cpu().numpy()[rows], yref, tol, f"M={M} N={N} K={K} g={g} {opts}")


# ------------------------------------------------------------ small, every element


def test_tiny_config():
    L = workloads.TINY
    check(workloads.TINY_M, L.n, L.k, L.g)


@pytest.mark.parametrize("M", [1, 8, 64])
@pytest.mark.parametrize("L", workloads.PARTIAL_LAYERS, ids=lambda L: L.name)
def test_partial_last_group_configs(M, L):
    check(M, L.n, L.k, L.g)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 7, 15, 16, 17, 31, 33, 63, 65, 127, 129, 255, 257, 300])
def test_tile_edges(M):
    # N = 300: a partial n-tile; K = 520: a 64-block tail of 8 and a last group 8 wide
    check(M, 300, 520, 128)


@pytest.mark.parametrize("block_n", [8, 16, 32, 64, 128])
@pytest.mark.parametrize("ctas,schedule", [(1, 1), (2, 1), (3, 1), (7, 1), (13, 1), (64, 1), (1, 2), (5, 2)])
def test_forced_schedules(block_n, ctas, schedule):
    # 3 n-tiles x 8 K stages (x m-tiles): stream-K cuts tiles at many places, incl. one CTA holding
    # the tail of one tile and the head of the next, and CTAs whose whole range sits inside one tile.
    # block_n 8 is the decode kernel (at most 8 tokens): ctas counts its clusters, schedule 2 runs
    # whole tiles, schedule 1 splits tiles along K between the CTAs of a cluster.
    check(20 if block_n > 8 else 8, 260, 2048, 128, block_n=block_n, ctas=ctas, schedule=schedule)


@pytest.mark.parametrize("M,N,K,g,ctas,schedule", [
    (256, 260, 2048, 128, 0, 0),   # odd number of weight tiles: the last pair's second tile is past N
    (300, 260, 960, 64, 5, 1),     # 15 K blocks: the last 128-wide stage holds one block
    (256, 384, 1000, 40, 3, 1),    # g not a multiple of 64: groups looked up per 8 codes
    (257, 130, 1088, 128, 7, 1),   # a 1-row last token tile, a 2-row last weight tile
    (512, 260, 960, 128, 0, 2),    # whole tile pairs
    (256, 1000, 4000, 128, 0, 0),  # the partial-group shape
])
def test_two_tile_units(M, N, K, g, ctas, schedule):
    # block_n 128 from M = 256 up schedules units of two weight tiles on one x tile (128-wide stages)
    check(M, N, K, g, block_n=128, ctas=ctas, schedule=schedule)


@pytest.mark.parametrize("M,N,K,g,block_n,ctas", [
    (64, 256, 4096, 128, 64, 10),    # one-tile units, 5 pieces per tile: copied into the owner's ring at once
    (64, 256, 4096, 128, 64, 14),    # 7 pieces: the ring's capacity for 32 KB pieces
    (64, 256, 4096, 128, 64, 16),    # 8 pieces: more than the ring holds, the shared fixup
    (200, 256, 4096, 128, 128, 8),   # block_n 128 (64 KB pieces), 2 pieces: ring
    (200, 256, 4096, 128, 128, 12),  # 3 pieces: ring at capacity
    (200, 256, 4096, 128, 128, 20),  # 5 pieces: shared fixup
    (256, 512, 4096, 128, 128, 8),   # two-tile units (128 KB pieces), 2 pieces: ring
    (256, 512, 4096, 128, 128, 12),  # 3 pieces: one weight tile's part of every piece at a time
    (256, 512, 4096, 128, 128, 16),  # 4 pieces: one weight tile at a time, at capacity
    (256, 512, 4096, 128, 128, 20),  # 5 pieces: shared fixup
    (256, 512, 4000, 40, 128, 8),    # g = 40 (two-stage ring), 2 pieces: one weight tile at a time
    (256, 512, 4000, 40, 128, 12),   # 3 pieces: read from L2 in the epilogue's loop
])
def test_cut_tile_fixups(M, N, K, g, block_n, ctas):
    # stream-K forced over few CTAs, so that every tile is cut into the stated number of pieces and the
    # owner takes each way of adding them; the sums must match the oracle like any other schedule
    check(M, N, K, g, block_n=block_n, ctas=ctas, schedule=1, rows=_sample_rows(M, 16))


@pytest.mark.parametrize("M,N,K,g,block_n,ctas", [
    (300, 1000, 1024, 128, 64, 7),  # 5 token tiles x 8 weight tiles over 7 CTAs: uneven tile counts
    (512, 700, 960, 128, 128, 5),   # two-tile units, a ragged pair, a one-block last stage
    (100, 300, 520, 40, 32, 3),     # per-word group lookup
    (40, 260, 256, 128, 16, 9),     # one K stage per tile: consecutive units are different tiles
])
def test_interleaved_whole_tiles(M, N, K, g, block_n, ctas):
    # whole tiles of several token tiles go round-robin: CTA c takes tiles c, c + P, c + 2P, ...
    check(M, N, K, g, block_n=block_n, ctas=ctas, schedule=2)


@pytest.mark.parametrize("g", [8, 16, 24, 32, 40, 64, 96, 128, 192, 256, 384, 512, 1024])
def test_group_sizes(g):
    # g % 64 == 0 puts one group in each 64-wide K block: the decode kernel (block_n 8) then scales
    # the block's fp32 partial sums, the tensor-memory kernel (16..128) scales in the dequant; any
    # other g looks the group up per 8 codes in both.
    # K = 1000 leaves a partial last group and a last stage of 4 blocks whose last block is ragged.
    check(9, 200, 1000, g)
    check(5, 200, 1000, g, block_n=8, ctas=3, schedule=1)
    check(9, 200, 1000, g, block_n=16, ctas=3, schedule=1)
    check(30, 200, 1000, g, block_n=32, ctas=5, schedule=1)
    check(70, 200, 1000, g, block_n=64, ctas=4, schedule=1)
    check(100, 200, 1000, g, block_n=128, ctas=3, schedule=1)


@pytest.mark.parametrize("block_n", [8, 16])
@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
def test_decode_kernel_clusters(block_n, cluster):
    # The decode kernel splits each weight tile's K stages between the CTAs of a cluster and sums the
    # partials in distributed shared memory. N = 300: three weight tiles, the last one 44 rows;
    # K = 2048: eight 256-wide stages, split 1, 2, 4 or 8 ways. ctas = 1: one cluster takes all three
    # tiles in turn (three reductions through the same slots); ctas = 2: rounds of unequal count.
    for M in sorted({1, 5, block_n}):
        for ctas in (0, 1, 2):
            check_opts(M, 300, 2048, 128, kernel=1, block_n=block_n, cluster=cluster, ctas=ctas)


@pytest.mark.parametrize("g", [8, 24, 40, 64, 128, 192, 256, 512, 1024])
@pytest.mark.parametrize("cluster", [1, 4])
def test_decode_kernel_group_modes(g, cluster):
    # g % 256 == 0: a stage lies in one group; g == 128: two groups per stage; other multiples of 64:
    # one group per 64-wide block; any other g: (q - z) * s per 8 codes. K = 1000: a partial last group,
    # a last stage of 4 blocks whose last block is ragged (K % 64 != 0: x comes in per-block copies).
    check_opts(7, 200, 1000, g, kernel=1, block_n=8, cluster=cluster)
    check_opts(13, 200, 1000, g, kernel=1, block_n=16, cluster=cluster)


@pytest.mark.parametrize("M,N,K,g,block_n", [(1, 4096, 4096, 128, 8), (8, 12288, 4096, 128, 8),
                                             (16, 4096, 11008, 128, 16), (3, 700, 960, 64, 8),
                                             (11, 288, 288, 256, 16)])
def test_decode_kernel_weights_static(M, N, K, g, block_n):
    # W4_FLAG_WEIGHTS_STATIC: the first stages' weight copies start before the previous grid is
    # waited for; results must not change, launch after launch
    rows = _sample_rows(M, 16)
    for cluster in [0] + _dec_clusters(K, M):
        check_opts(M, N, K, g, rows=rows, kernel=1, block_n=block_n, cluster=cluster, flags=w4.FLAG_WEIGHTS_STATIC)
    qw, s, zw, packed, wn = layer(N, K, g)
    x = torch.from_numpy(workloads.activations_f16(M, K)).cuda()
    ws = w4.Workspace()
    first = w4.w4a16_gemm_opts(x, packed, N, K, g, kernel=1, block_n=block_n, workspace=ws)
    for _ in range(20):
        y = w4.w4a16_gemm_opts(x, packed, N, K, g, kernel=1, block_n=block_n, flags=w4.FLAG_WEIGHTS_STATIC,
                               workspace=ws)
        assert torch.equal(y, first)
    assert w4.w4_last_device_error(ws) == 0


@pytest.mark.parametrize("K,g", [(288, 256), (320, 64), (320, 128), (448, 128), (576, 192), (4000, 128), (200, 8)])
@pytest.mark.parametrize("block_n", [8, 16, 32, 64, 128])
def test_short_last_stage(K, g, block_n):
    # A stage is four 64-wide K blocks; these K leave a last stage of 1..3 blocks (K % 64 != 0 also
    # switches x to one tensor copy per block). Forced small grids start CTA ranges on that stage.
    M = {8: 7, 16: 13, 32: 29, 64: 50, 128: 90}[block_n]
    check(M, 264, K, g, block_n=block_n)
    for ctas in (2, 3, 5):
        check(M, 264, K, g, block_n=block_n, ctas=ctas, schedule=1)


def test_one_hot_rows_return_rounded_weights_exactly():
    N, K, g = 384, 640, 128
    qw, s, zw, packed, wn = layer(N, K, g)
    ks = [0, 1, 63, 64, 127, 128, 300, 511, 600, 639]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    wd = oracle.dequant(qw, s, zw, N, K, g)
    expect = wd[:, ks].T.astype(np.float16)  # (q - z) * s is exact in fp64; one rounding to fp16
    for bn, ctas, sch in [(0, 0, 0), (16, 1, 2), (16, 4, 1), (128, 1, 1), (64, 5, 1), (16, 11, 1), (32, 3, 1)]:
        y = run_gemm(x, packed, N, K, g, bn, ctas, sch)
        assert (y.view(np.uint16) == expect.view(np.uint16)).all(), (bn, ctas, sch)
    for bn, cluster in [(8, 1), (8, 2), (16, 1), (16, 2)]:  # the decode kernel, K split 1 or 2 ways
        xs = torch.from_numpy(x[: min(bn, len(ks))]).cuda()
        y = w4.w4a16_gemm_opts(xs, packed, N, K, g, kernel=1, block_n=bn, cluster=cluster).cpu().numpy()
        assert (y.view(np.uint16) == expect[: xs.shape[0]].view(np.uint16)).all(), (bn, cluster)


def test_q_equal_z_gives_exact_zero():
    N, K, g = 256, 512, 64
    G = K // g
    rng = np.random.default_rng(4)
    z = rng.integers(0, 16, (N, G)).astype(np.uint8)
    q = z[:, np.arange(K) // g]
    s = (np.abs(rng.standard_normal((N, G))) + 0.01).astype(np.float16)
    qw, zw = oracle.pack_nibbles(q), oracle.pack_nibbles(z)
    packed = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                          torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
    x = workloads.activations_f16(17, K)
    y = run_gemm(x, packed, N, K, g)
    assert (y == 0).all()
    for bn, m in ((8, 7), (16, 16)):  # the decode kernel, K split 2 ways
        y = w4.w4a16_gemm_opts(torch.from_numpy(x[:m]).cuda(), packed, N, K, g, kernel=1, block_n=bn, cluster=2)
        assert (y == 0).all()


def test_deterministic_and_workspace_reuse():
    N, K, g, M = 1000, 2048, 128, 12
    qw, s, zw, packed, wn = layer(N, K, g)
    x = torch.from_numpy(workloads.activations_f16(M, K)).cuda()
    ws = w4.Workspace()
    outs = [w4.w4a16_gemm_ex(x, packed, N, K, g, 16, 5, 1, workspace=ws).clone() for _ in range(3)]
    outs += [w4.w4a16_gemm(x, packed, N, K, g, workspace=ws).clone() for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert torch.equal(outs[3], outs[4])
    # counters were left at zero: a fresh workspace gives the same bits
    y2 = w4.w4a16_gemm_ex(x, packed, N, K, g, 16, 5, 1, workspace=w4.Workspace())
    assert torch.equal(outs[0], y2)
    assert w4.w4_last_device_error(ws) == 0


def test_end_to_end_from_fp16_weights():
    # GPU pack -> GPU repack -> GEMM, against the oracle run from the same fp16 weights
    N, K, g, M = 512, 768, 128, 6
    W = workloads.weights_f16(N, K, seed=21)
    qw, s, zw = w4.w4_pack(torch.from_numpy(W).cuda(), g)
    packed = w4.w4_repack(qw, s, zw, N, K, g)
    x = workloads.activations_f16(M, K, seed=22)
    y = w4.w4a16_gemm(torch.from_numpy(x).cuda(), packed, N, K, g).cpu().numpy()
    oq, os_, oz = oracle.pack(W, g)
    yref = oracle.gemm(x, oq, os_, oz, N, K, g)
    assert_within_tolerance(y, yref, gemm_tolerance(x, row_norms_dequant(oq, os_, oz, N, K, g)), "e2e")


def test_host_errors_on_device_tensors():
    N, K, g = 256, 512, 128
    qw, s, zw, packed, wn = layer(N, K, g)
    flat = torch.zeros(3 * K + 8, dtype=torch.float16, device="cuda")
    x_mis = flat[1:1 + 3 * K].view(3, K)  # contiguous but 2 bytes off a 16-byte boundary
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemm(x_mis, packed, N, K, g)
    assert e.value.status == 3
    x12 = torch.zeros(3, 12, dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemm(x12, packed, N, 12, 8)
    assert e.value.status == 2
    x = torch.zeros(16, K, dtype=torch.float16, device="cuda")
    with pytest.raises(w4.W4Error) as e:
        w4.w4a16_gemm_ex(x, packed, N, K, g, 16, 4, 1,
                         workspace=torch.zeros(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4


# ------------------------------------------------------- full-size layers, sampled


def _sample_rows(M, k=24, seed=5):
    if M <= k:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, M - 1], rng.choice(M, k - 2, replace=False)]))


@pytest.mark.parametrize("L", workloads.DECODE_LAYERS, ids=lambda L: L.name)
def test_decode_sweep_layers(L):
    for M in workloads.DECODE_MS:
        check(M, L.n, L.k, L.g, rows=_sample_rows(M, 16))


@pytest.mark.parametrize("L", workloads.PREFILL_LAYERS, ids=lambda L: L.name)
def test_prefill_layers_sampled(L):
    # every prefill batch size: M = 512 and 1024 run stream-K over two-tile units and interleaved
    # whole tiles, the schedules the prefill measurements come from
    for M in workloads.PREFILL_MS:
        check(M, L.n, L.k, L.g, rows=_sample_rows(M, 8), outliers=True)


@pytest.mark.parametrize("M,N,K,g", [(80, 22016, 4096, 128), (128, 22016, 4096, 128), (200, 10240, 8192, 128),
                                     (255, 8192, 2048, 128), (100, 19584, 1000, 40), (200, 10240, 1000, 40)])
def test_two_tile_units_below_256_tokens(M, N, K, g):
    # block_n 128 below 256 tokens takes units of two weight tiles where the tile pairs are many (at
    # least 0.4 per SM): one token tile (80 and 100 rows ragged, 128 full) or two with a ragged second
    # (72 and 127 rows), stream-K with cut pairs; g = 40 looks its groups up per 8 codes, and 153
    # weight tiles (19584 rows) leave the last pair's second tile past N
    check(M, N, K, g, rows=_sample_rows(M, 8), outliers=True)


@pytest.mark.parametrize("M,N,K", [(160, 8192, 8192), (255, 4096, 4096), (129, 11008, 4096)])
def test_block_n_64_above_128_tokens(M, N, K):
    # three or four token tiles of 64 on layers with fewer weight tiles than SMs, the last one ragged
    check(M, N, K, 128, rows=_sample_rows(M, 8), outliers=True)


@pytest.mark.parametrize("L", [workloads.STACK_LAYER[4], workloads.STACK_HEAD], ids=lambda L: L.name)
def test_stack_only_layers(L):
    # the decode stack's shapes that the decode sweep does not have: the unfused 11008 x 4096 gate/up
    # projection and the 32000 x 4096 lm_head (250 weight tiles: more than one per SM); every row at
    # M <= 16, sampled rows at M = 128
    for M in workloads.STACK_MS:
        check(M, L.n, L.k, L.g, rows=None if M <= 16 else _sample_rows(M, 16))


@pytest.mark.parametrize("N,K,M,block_n,ctas,schedule", [
    (10240, 8192, 256, 128, 80, 2), (10240, 8192, 256, 128, 0, 1), (10240, 8192, 256, 64, 0, 1),
    (10240, 8192, 256, 32, 0, 1), (10240, 8192, 256, 16, 0, 1),
    # 172 tiles over 152 CTAs: many CTAs hold a short head or tail segment that some dequant groups skip
    (22016, 4096, 64, 64, 0, 1), (22016, 4096, 128, 128, 0, 1), (22016, 4096, 16, 16, 0, 1),
    (22016, 4096, 8, 8, 0, 1), (4096, 4096, 3, 8, 0, 1)])
def test_repeated_launches_bit_identical(N, K, M, block_n, ctas, schedule):
    # The schedule is deterministic, so back-to-back launches must agree bit for bit; a pipeline
    # hazard (a stage, slot or accumulator used before it was ready) shows up as a differing launch.
    qw, s, zw, packed, wn = layer(N, K, 128)
    x = torch.from_numpy(workloads.activations_f16(M, K, outliers=True)).cuda()
    ws = w4.Workspace()
    first = w4.w4a16_gemm_ex(x, packed, N, K, 128, block_n, ctas, schedule, workspace=ws)
    ndiff = 0
    for _ in range(30):
        y = w4.w4a16_gemm_ex(x, packed, N, K, 128, block_n, ctas, schedule, workspace=ws)
        ndiff += int(not torch.equal(y, first))
    assert ndiff == 0
    rows = np.unique(np.array([0, min(17, M - 1), M // 2, M - 1]))
    yref = oracle.gemm(x.cpu().numpy()[rows], qw, s, zw, N, K, 128)
    assert_within_tolerance(first.cpu().numpy()[rows], yref, gemm_tolerance(x.cpu().numpy()[rows], wn), "repeat")
    assert w4.w4_last_device_error(ws) == 0
