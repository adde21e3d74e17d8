"""w4_pack and w4_repack on the GPU, bit-exact against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import w4a16_group_quantized_gb300 as w4
import workloads

pytestmark = pytest.mark.gpu

PACK_CASES = [
    (256, 512, 128),      # tiny layer
    (288, 288, 256),      # torchchat's 288 x 288 with group size 256: last group 32 wide
    (4096, 4000, 128),    # last group 32 wide
    (100, 1001, 8),       # K not a multiple of 8, last group 1 wide, G = 126 (not a multiple of 8)
    (130, 200, 24),       # g not dividing 64
    (64, 520, 32),
    (33, 136, 64),
    (4096, 4096, 128),    # o_proj
    (4096, 11008, 128),   # down_proj
]


def _pack_gpu(W, g):
    qw, s, zw = w4.w4_pack(torch.from_numpy(W).cuda(), g)
    torch.cuda.synchronize()
    return qw.cpu().numpy().view(np.uint32), s.cpu().numpy(), zw.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("N,K,g", PACK_CASES)
def test_pack_bit_exact(N, K, g):
    W = workloads.weights_f16(N, K, seed=N + K)
    W[0, :] = 0  # degenerate all-zero groups
    W[min(1, N - 1), :] = np.abs(W[min(1, N - 1), :])
    qw, s, zw = _pack_gpu(W, g)
    oq, os_, oz = oracle.pack(W, g)
    assert (qw == oq).all()
    assert (s.view(np.uint16) == os_.view(np.uint16)).all()
    assert (zw == oz).all()


def test_pack_bit_exact_gate_up_shape():
    N, K, g = 22016, 4096, 128
    W = workloads.weights_f16(N, K)
    qw, s, zw = _pack_gpu(W, g)
    oq, os_, oz = oracle.pack(W, g)
    assert (qw == oq).all() and (s.view(np.uint16) == os_.view(np.uint16)).all() and (zw == oz).all()


def test_pack_wide_dynamic_range():
    # values spanning fp16's range, including subnormal-sized groups and large magnitudes
    rng = np.random.default_rng(9)
    N, K, g = 64, 256, 32
    mag = np.exp2(rng.uniform(-24, 15, (N, 1)))
    W = (rng.standard_normal((N, K)) * mag).clip(-60000, 60000).astype(np.float16)
    qw, s, zw = _pack_gpu(W, g)
    oq, os_, oz = oracle.pack(W, g)
    assert (qw == oq).all() and (s.view(np.uint16) == os_.view(np.uint16)).all() and (zw == oz).all()


def _pack_gpu_ex(Wbits, g, dtype, symmetric):
    t = torch.from_numpy(Wbits.view(np.int16)).cuda().view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    qw, s, zw = w4.w4_pack(t, g, symmetric=symmetric)
    torch.cuda.synchronize()
    assert s.dtype == t.dtype
    return (qw.cpu().numpy().view(np.uint32), s.view(torch.int16).cpu().numpy().view(np.uint16),
            zw.cpu().numpy().view(np.uint32))


VARIANT_CASES = [(256, 512, 128), (288, 288, 256), (100, 1001, 8), (130, 200, 24), (4096, 4096, 128)]


@pytest.mark.parametrize("dtype,symmetric", [("f16", True), ("bf16", False), ("bf16", True)])
@pytest.mark.parametrize("N,K,g", VARIANT_CASES)
def test_pack_variants_bit_exact(N, K, g, dtype, symmetric):
    if dtype == "bf16":
        W = workloads.weights_bf16(N, K, seed=N + K)
    else:
        W = workloads.weights_f16(N, K, seed=N + K).view(np.uint16)
    W = W.copy()
    W[0, :] = 0                                # all-zero groups: s = 1, every code = z
    W[min(1, N - 1), :] &= np.uint16(0x7FFF)   # a non-negative row
    W[min(2, N - 1), : K // 2] |= np.uint16(0x8000)  # a non-positive half row
    qw, s, zw = _pack_gpu_ex(W, g, dtype, symmetric)
    oq, os_, oz = oracle.pack(W if dtype == "bf16" else W.view(np.float16), g, dtype, symmetric)
    assert (qw == oq).all()
    assert (s == os_.view(np.uint16)).all()
    assert (zw == oz).all()
    if symmetric:
        G = oracle.ngroups(K, g)
        assert (oracle.unpack_nibbles(zw, G) == 8).all()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pack_variants_wide_range(dtype):
    # magnitudes across the type's range, subnormal-sized groups included
    rng = np.random.default_rng(10)
    N, K, g = 64, 256, 32
    if dtype == "bf16":
        mag = np.exp2(rng.uniform(-130, 120, (N, 1)))
        W = workloads.f32_to_bf16_bits((rng.standard_normal((N, K)) * mag).astype(np.float32))
    else:
        mag = np.exp2(rng.uniform(-24, 15, (N, 1)))
        W = (rng.standard_normal((N, K)) * mag).clip(-60000, 60000).astype(np.float16).view(np.uint16)
    for symmetric in (False, True):
        qw, s, zw = _pack_gpu_ex(W, g, dtype, symmetric)
        oq, os_, oz = oracle.pack(W if dtype == "bf16" else W.view(np.float16), g, dtype, symmetric)
        assert (qw == oq).all() and (s == os_.view(np.uint16)).all() and (zw == oz).all(), symmetric


@pytest.mark.parametrize("N,K,g", PACK_CASES + [(1, 8, 8), (129, 72, 8)])
def test_repack_bit_exact(N, K, g):
    # canonical input from the oracle, so repack is checked on its own
    rng = np.random.default_rng(N * 7 + K)
    G = oracle.ngroups(K, g)
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    z = rng.integers(0, 16, (N, G)).astype(np.uint8)
    s = rng.standard_normal((N, G)).astype(np.float16)
    qw, zw = oracle.pack_nibbles(q), oracle.pack_nibbles(z)
    if K % 8:
        qw[:, -1] |= np.uint32(0xF0000000)  # garbage in the padding nibbles must not leak into the tiles
    got = w4.w4_repack(torch.from_numpy(qw.view(np.int32)).cuda(), torch.from_numpy(s).cuda(),
                       torch.from_numpy(zw.view(np.int32)).cuda(), N, K, g)
    torch.cuda.synchronize()
    qw_clean = oracle.pack_nibbles(q)
    ref = oracle.repack(qw_clean, s, zw, N, K, g)
    assert got.numel() == ref.size
    assert (got.cpu().numpy() == ref).all()
