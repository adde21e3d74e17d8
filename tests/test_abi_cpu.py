"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/w4a16.h declares, sizes its buffers by the documented formulas and
rejects bad arguments on the host before any CUDA call."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import w4a16_group_quantized_gb300 as w4
from w4a16_group_quantized_gb300 import build as w4build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def lib():
    w4build.build()
    return w4.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"W4_API\s+[\w\s\*]*?\b(w4\w*)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for required in ("w4_pack", "w4_repack", "w4a16_gemm"):
        assert required in names
    assert len(names) >= 10


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in w4.STATUS.items():
        assert w4.w4_status_string(code).startswith(name)
    assert "unknown" in w4.w4_status_string(99)


def test_repacked_bytes_formula(lib):
    for (N, K, g) in [(256, 512, 128), (288, 288, 256), (4096, 4000, 128), (12288, 4096, 128), (1, 8, 8),
                      (57344, 8192, 128), (130, 72, 8)]:
        NT, KB, G = -(-N // 128), -(-K // 64), -(-K // g)
        assert w4.w4_repacked_bytes(N, K, g) == NT * KB * 4096 + NT * G * 320
    assert w4.w4_repacked_bytes(0, 8, 8) == 0
    assert w4.w4_repacked_bytes(8, 8, 12) == 0  # g not a multiple of 8


def test_workspace_sizes(lib):
    # whole tiles: error word block + per-tile counters only; block_n 128 with M >= 256 schedules
    # units of two 128-row weight tiles, so 512 x 8192 has 4 x 32 output tiles
    b = w4.w4a16_workspace_bytes_ex(512, 8192, 8192, 128, 128, 0, 2)
    assert b == 256 + 512  # 4 x 32 tile counters of 4 bytes
    b = w4.w4a16_workspace_bytes_ex(512, 8192, 8192, 128, 64, 0, 2)
    assert b == 256 + 2048  # 8 x 64 tile counters
    # stream-K with P CTAs: plus two fp32 partial tiles (128 x block_n, two of them for block_n 128)
    M, N, K, P = 16, 300, 1024, 4
    b = w4.w4a16_workspace_bytes_ex(M, N, K, 128, 16, P, 1)
    assert b == 256 + 256 + P * 2 * 128 * 16 * 4
    b = w4.w4a16_workspace_bytes_ex(M, N, K, 128, 128, P, 1)  # M < 256, two tile pairs: units of one weight tile
    assert b == 256 + 256 + P * 2 * 128 * 128 * 4
    b = w4.w4a16_workspace_bytes_ex(256, N, K, 128, 128, P, 1)  # M >= 256: units of two weight tiles
    assert b == 256 + 256 + P * 2 * 2 * 128 * 128 * 4
    assert w4.w4a16_workspace_bytes(0, 1, 8, 8) == 0
    assert w4.w4a16_workspace_bytes_ex(1, 1, 8, 8, 24, 0, 0) == 0  # block_n must be 8..128, a power of two
    assert w4.w4a16_workspace_bytes_ex(1, 1, 8, 8, 8, 0, 0) > 0
    assert w4.w4a16_workspace_bytes_ex(1, 1, 8, 8, 256, 0, 0) == 0
    assert w4.w4a16_workspace_bytes_ex(1, 1, 8, 8, 16, 0, 3) == 0  # no schedule 3


def _grouped_bytes(lib, M, specs, g=128):
    """w4a16_grouped_workspace_bytes for problems (x address, N, K); the host only compares and checks
    the addresses, it never reads through them."""
    arr = (w4.Problem * len(specs))()
    for i, (x, N, K) in enumerate(specs):
        arr[i].x_dev = x
        arr[i].packed_dev = 0x1000000 * (i + 1)
        arr[i].y_dev = 0x40000000 + 0x1000000 * i
        arr[i].N = N
        arr[i].K = K
    return int(lib.w4a16_grouped_workspace_bytes(arr, len(specs), M, g, ctypes.byref(w4.Options())))


def test_grouped_workspace_follows_the_group_plan(lib):
    X, X2 = 0x100000, 0x200000
    ws = w4.w4a16_workspace_bytes
    # q, k, v of one x above the decode kernel's range: one tensor-memory launch, planned as one GEMM
    # of their weight tiles laid end to end
    assert _grouped_bytes(lib, 64, [(X, 4096, 4096)] * 3) == ws(64, 3 * 4096, 4096, 128)
    # ragged problems count whole weight tiles (8 + 3 here)
    assert _grouped_bytes(lib, 40, [(X, 1000, 1024), (X, 300, 1024)]) == ws(40, 128 * 11, 1024, 128)
    # different x, or different K: one launch each, so the largest single workspace
    assert _grouped_bytes(lib, 64, [(X, 4096, 4096), (X2, 11008, 4096)]) == max(ws(64, 4096, 4096, 128),
                                                                               ws(64, 11008, 4096, 128))
    assert _grouped_bytes(lib, 64, [(X, 4096, 4096), (X, 4096, 11008)]) == max(ws(64, 4096, 4096, 128),
                                                                              ws(64, 4096, 11008, 128))
    # the 7B gate/up pair at M = 128: alone, 172 weight tiles would take two-tile units (86 pairs); the
    # group keeps one launch of one-tile units (stream-K over every SM, one counter per tile, two
    # partial tiles of 128 x 128 per CTA)
    sms = 148  # no GPU here: the planner's default SM count
    one_tile = 256 + 768 + sms * 2 * 128 * 128 * 4
    assert _grouped_bytes(lib, 128, [(X, 11008, 4096)] * 2) == one_tile
    assert ws(128, 22016, 4096, 128) != one_tile
    # two-tile units (M >= 256) are not grouped
    assert _grouped_bytes(lib, 512, [(X, 8192, 8192)] * 2) == ws(512, 8192, 8192, 128)
    # more than eight problems: one launch each
    assert _grouped_bytes(lib, 64, [(X, 256, 1024)] * 9) == ws(64, 256, 1024, 128)
    # the decode range: the decode kernel's 256-byte error block, grouped or not
    assert _grouped_bytes(lib, 4, [(X, 4096, 4096)] * 3) == 256


def test_automatic_block_n(lib):
    # 65..128 tokens: block_n 64 (two token tiles) on layers with fewer 128-row weight tiles than
    # SMs, else 128; the workspace size shows the choice (stream-K, 100 CTAs: two fp32 partial
    # tiles of 128 x block_n per CTA, one counter per output tile)
    P = 100
    b = w4.w4a16_workspace_bytes_ex(128, 4096, 4096, 128, 0, P, 1)  # 32 weight tiles
    assert b == 256 + 256 + P * 2 * 128 * 64 * 4
    b = w4.w4a16_workspace_bytes_ex(96, 12288, 4096, 128, 0, P, 1)  # 96 weight tiles
    assert b == 256 + 768 + P * 2 * 128 * 64 * 4  # 2 x 96 counters
    # 172 weight tiles: block_n 128, in units of two weight tiles (86 pairs, at least 0.4 per SM):
    # 86 counters, partial tiles of 2 x 128 x 128
    b = w4.w4a16_workspace_bytes_ex(128, 22016, 4096, 128, 0, P, 1)
    assert b == 256 + 512 + P * 2 * 2 * 128 * 128 * 4
    # 129..192 tokens, and up to 255 on layers of at most 32 weight tiles (K <= 16384): block_n 64 too
    b = w4.w4a16_workspace_bytes_ex(200, 4096, 4096, 128, 0, P, 1)  # 4 token tiles x 32 weight tiles
    assert b == 256 + 512 + P * 2 * 128 * 64 * 4
    b = w4.w4a16_workspace_bytes_ex(160, 8192, 8192, 128, 0, P, 1)  # 3 x 64 output tiles
    assert b == 256 + 768 + P * 2 * 128 * 64 * 4
    # ... but K = 28672 keeps block_n 128, in two-tile units (2 token tiles x 32 pairs)
    b = w4.w4a16_workspace_bytes_ex(160, 8192, 28672, 128, 0, P, 1)
    assert b == 256 + 256 + P * 2 * 2 * 128 * 128 * 4
    # 200 tokens on 80 weight tiles: 2 token tiles x 40 pairs = 80 pairs, two-tile units
    b = w4.w4a16_workspace_bytes_ex(200, 10240, 4096, 128, 0, P, 1)
    assert b == 256 + 512 + P * 2 * 2 * 128 * 128 * 4
    # the decode kernel (8-token tiles) reduces its split along K in distributed shared memory: its
    # workspace is the error word alone
    assert w4.w4a16_workspace_bytes_ex(8, 4096, 4096, 128, 0, P, 1) == 256
    assert w4.w4a16_workspace_bytes(1, 22016, 4096, 128) == 256


def test_grid_shrinks_to_the_piece_bound(lib):
    # one weight tile of 16 K stages: stream-K over more than 8 CTAs would cut it into more than 8
    # pieces, so the planner shrinks the grid to 8 CTAs (8 x two 128 x 8 fp32 partial tiles)
    for schedule in (0, 1):
        assert w4.w4a16_workspace_bytes_ex(16, 128, 4096, 128, 16, 0, schedule) == 256 + 256 + 8 * 2 * 128 * 16 * 4
    # two-tile units (M >= 256, block_n 128): 4 token tiles x 4 tile pairs = 16 output tiles over
    # 10 CTAs, not a multiple: stream-K with partial tiles of 2 x 128 x 128 fp32
    b = w4.w4a16_workspace_bytes_ex(512, 1024, 1024, 128, 128, 10, 0)
    assert b == 256 + 256 + 10 * 2 * 2 * 128 * 128 * 4


def test_options_validation(lib):
    O = w4.Options
    # the decode kernel: up to 16 tokens (block_n 8 or 16, M <= block_n); clusters of 1, 2, 4 or 8 CTAs,
    # at most the number of 256-wide K stages of a tile
    assert w4.w4a16_workspace_bytes_opts(16, 4096, 4096, 128, O(1, 16, 0, 0, 4, 0, 0)) == 256
    assert w4.w4a16_workspace_bytes_opts(9, 4096, 4096, 128, O(1, 8, 0, 0, 0, 0, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(17, 4096, 4096, 128, O(1, 0, 0, 0, 0, 0, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(1, 32, 0, 0, 0, 0, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(1, 8, 0, 0, 3, 0, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 1024, 128, O(1, 8, 0, 0, 8, 0, 0)) == 0  # 4 K stages
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 1024, 128, O(1, 8, 0, 0, 4, 0, 0)) == 256
    # the tensor-memory kernel takes no 8-token tiles; unknown flags and kernels are refused
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(2, 8, 0, 0, 0, 0, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(2, 16, 4, 1, 0, 0, 0)) == 256 + 256 + 4 * 2 * 128 * 16 * 4
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(0, 0, 0, 0, 0, 4, 0)) == 0  # no flag 4
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(3, 0, 0, 0, 0, 0, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(0, 0, 0, 0, 0, 1, 0)) == 256
    # value types: fp16 (0) or bf16 (1), the reserved field zero
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(0, 0, 0, 0, 0, 0, 0, 1, 0)) == 256
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(0, 0, 0, 0, 0, 0, 0, 2, 0)) == 0
    assert w4.w4a16_workspace_bytes_opts(4, 4096, 4096, 128, O(0, 0, 0, 0, 0, 0, 0, 0, 1)) == 0


def _vp(v):
    return ctypes.c_void_p(v)


def test_host_side_argument_checks(lib):
    fake = _vp(0x10000)  # never dereferenced: every case below fails its host-side check first
    ws = _vp(0x20000)
    S = w4
    # null pointers / bad sizes / bad group
    assert lib.w4a16_gemm(None, fake, 1, 1, 8, 8, fake, ws, 4096, None) == 1
    assert lib.w4a16_gemm(fake, fake, 0, 1, 8, 8, fake, ws, 4096, None) == 1
    assert lib.w4a16_gemm(fake, fake, 1, 1, 8, 12, fake, ws, 4096, None) == 1
    assert lib.w4a16_gemm(fake, fake, 1, 1, 8, 0, fake, ws, 4096, None) == 1
    # K not a multiple of 8
    assert lib.w4a16_gemm(fake, fake, 1, 1, 12, 8, fake, ws, 4096, None) == 2
    # misaligned x / packed / workspace
    assert lib.w4a16_gemm(_vp(0x10008), fake, 1, 1, 8, 8, fake, ws, 4096, None) == 3
    assert lib.w4a16_gemm(fake, _vp(0x10004), 1, 1, 8, 8, fake, ws, 4096, None) == 3
    assert lib.w4a16_gemm(fake, fake, 1, 1, 8, 8, fake, _vp(0x20010), 4096, None) == 3
    # workspace too small
    assert lib.w4a16_gemm(fake, fake, 1, 1, 8, 8, fake, ws, 16, None) == 4
    assert lib.w4a16_gemm_ex(fake, fake, 16, 300, 1024, 128, fake, ws, 1024, 16, 4, 1, None) == 4
    # forced schedule out of range
    assert lib.w4a16_gemm_ex(fake, fake, 16, 300, 1024, 128, fake, ws, 1 << 30, 48, 1, 0, None) == 1
    assert lib.w4a16_gemm_ex(fake, fake, 16, 300, 1024, 128, fake, ws, 1 << 30, 16, -1, 0, None) == 1
    assert lib.w4a16_gemm_ex(fake, fake, 16, 300, 1024, 128, fake, ws, 1 << 30, 16, 1, 7, None) == 1
    # pack / repack
    assert lib.w4_pack(None, 4, 8, 8, fake, fake, fake, None) == 1
    assert lib.w4_pack(fake, 4, 8, 7, fake, fake, fake, None) == 1
    assert lib.w4_pack(_vp(0x10001), 4, 8, 8, fake, fake, fake, None) == 3
    # w4_pack_ex: dtype 0 or 1, symmetric 0 or 1
    assert lib.w4_pack_ex(fake, 4, 8, 8, 2, 0, fake, fake, fake, None) == 1
    assert lib.w4_pack_ex(fake, 4, 8, 8, 0, 2, fake, fake, fake, None) == 1
    assert lib.w4_pack_ex(fake, 4, 8, 8, -1, 0, fake, fake, fake, None) == 1
    assert lib.w4_pack_ex(_vp(0x10001), 4, 8, 8, 1, 1, fake, fake, fake, None) == 3
    assert lib.w4_repack(fake, fake, fake, 4, 8, 8, _vp(0x10008), None) == 3
    assert lib.w4_repack(fake, fake, fake, -1, 8, 8, fake, None) == 1
    assert lib.w4_last_device_error(None, None) == 1
    del S


def test_binding_has_no_cpu_path():
    import torch

    x = torch.zeros(4, 8, dtype=torch.float16)
    with pytest.raises(ValueError):
        w4.w4a16_gemm(x, torch.zeros(16, dtype=torch.uint8), 8, 8, 8)
    with pytest.raises(ValueError):
        w4.w4_pack(torch.zeros(4, 8, dtype=torch.float16), 8)
