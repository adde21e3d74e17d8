"""Pins for the CPU oracle, checked against things other than the oracle itself.

Each test ties an oracle function to an independent fact: numpy's IEEE
binary16 and binary32 conversions (bfloat16 is the top half of a binary32),
exact rational arithmetic (``fractions.Fraction``), a closed form, an invariant
proved from the definition, a library matmul, or a value derived by hand in
``tests/golden/``. None of them calls the CUDA path.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f16(vals) -> np.ndarray:
    a = np.asarray(vals, dtype=np.float64).astype(np.float16)
    assert (a.astype(np.float64) == np.asarray(vals, dtype=np.float64)).all(), "fixture value not exact fp16"
    return a


def _fr(h) -> Fraction:
    return Fraction(float(np.float16(h)))


def _val_bits(b: int) -> Fraction:
    return Fraction(float(np.uint16(b).view(np.float16)))


# --------------------------------------------------------------------------- fp16


def test_half_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    # signed zeros keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_half_encode_matches_numpy_rne():
    rng = np.random.default_rng(123)
    vals = [0.0, -0.0, 65504.0, 65519.999, 65520.0, -65520.0, 1e6, 2.0**-24, 2.0**-25,
            3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11]
    mags = np.exp2(rng.uniform(-30, 17, 4000)) * rng.choice([-1.0, 1.0], 4000)
    vals += list(mags)
    # exact midpoints between neighbouring fp16 values (ties), and points next to them
    h = rng.integers(0, 0x7BFF, 3000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2  # exact in fp64
    vals += list(mid) + list(np.nextafter(mid, 0)) + list(np.nextafter(mid, np.inf)) + list(-mid)
    vals = np.array(vals, dtype=np.float64)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(v) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(vals[i], hex(got[i]), hex(ref[i])) for i in bad[:5]]


# ----------------------------------------------------------------------- quantize


def _smallest_f16_at_least(r: Fraction) -> int:
    """Exact: the least positive fp16 (bits) whose value is >= r."""
    b = int(np.float16(float(r)).view(np.uint16)) & 0x7FFF
    while _val_bits(b) < r:
        b += 1
    while b > 0 and _val_bits(b - 1) >= r:
        b -= 1
    return b


def _quantize_exact(w: list[Fraction], K: int, g: int):
    """The quantization definition in exact rational arithmetic (an independent formulation:
    s is 'r/15 rounded up to fp16', Python's round() is round-half-even on Fractions)."""
    G = -(-K // g)
    q, s, z = [0] * K, [0] * G, [0] * G
    for j in range(G):
        grp = w[j * g:min((j + 1) * g, K)]
        lo, hi = min([Fraction(0)] + grp), max([Fraction(0)] + grp)
        r = hi - lo
        if r == 0:
            s[j], z[j] = 0x3C00, 0
            continue
        sb = _smallest_f16_at_least(r / 15)
        sv = _val_bits(sb)
        zj = min(15, max(0, round(-lo / sv)))
        s[j], z[j] = sb, zj
        for i, wk in enumerate(grp):
            q[j * g + i] = min(15, max(0, round(wk / sv) + zj))
    return q, s, z


@pytest.mark.parametrize("K,g,seed", [(8, 8, 0), (40, 16, 1), (24, 8, 2), (100, 32, 3), (288, 256, 4),
                                     (129, 64, 5), (7, 8, 6)])
def test_quantize_equals_exact_rational_definition(K, g, seed):
    rng = np.random.default_rng(seed)
    N = 6
    W = (rng.standard_normal((N, K)) * rng.choice([0.02, 1.0, 300.0], (N, 1))).astype(np.float16)
    W[0, : min(K, g)] = 0  # a degenerate all-zero group
    W[1] = np.abs(W[1])  # all positive: zero is the low end
    W[2] = -np.abs(W[2])  # all negative: zero is the high end
    q, s, z = oracle.quantize(W, g)
    for n in range(N):
        qe, se, ze = _quantize_exact([_fr(v) for v in W[n]], K, g)
        assert list(q[n]) == qe
        assert list(s[n].view(np.uint16)) == se
        assert list(z[n]) == ze


def test_quantize_invariants_on_config_shapes():
    # the tiny config and the torchchat-style partial group, plus a third shape with a 104-wide tail
    for (N, K, g) in [(256, 512, 128), (288, 288, 256), (64, 1000, 128)]:
        W = workloads.weights_f16(N, K, seed=7)
        q, s, z = oracle.quantize(W, g)
        G = oracle.ngroups(K, g)
        assert q.max() <= 15 and z.max() <= 15
        w = W.astype(np.float64)
        sv = s.astype(np.float64)
        idx = np.arange(K) // g
        what = (q.astype(np.float64) - z[:, idx]) * sv[:, idx]
        # round-trip error bound |w - (q - z) s| <= s/2 (plus fp64 division slack)
        assert (np.abs(w - what) <= sv[:, idx] / 2 * (1 + 2.0**-40)).all()
        # s is the least fp16 with 15 s >= r (range including zero)
        for j in range(G):
            blk = w[:, j * g:min((j + 1) * g, K)]
            r = np.maximum(blk.max(1), 0) - np.minimum(blk.min(1), 0)
            nz = r > 0
            assert (15 * sv[nz, j] >= r[nz]).all()
            prev = (s[nz, j].view(np.uint16) - 1).view(np.float16).astype(np.float64)
            assert (15 * prev < r[nz]).all()
            assert (s[~nz, j].view(np.uint16) == 0x3C00).all()


def test_quantize_rejects_non_finite():
    W = np.zeros((2, 16), np.float16)
    W[1, 3] = np.inf
    with pytest.raises(ValueError):
        oracle.quantize(W, 8)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([c.strip() for c in line.split("|")])
    return rows


def test_quantize_hand_derived_groups():
    for name, ws, sbits, zz, codes in _read_golden("quantize_groups.txt"):
        W = _f16([float(v) for v in ws.split()])[None, :]
        q, s, z = oracle.quantize(W, 8)
        assert int(s[0, 0].view(np.uint16)) == int(sbits, 16), name
        assert int(z[0, 0]) == int(zz), name
        assert list(q[0]) == [int(c) for c in codes.split()], name


def test_partial_last_group_hand_derived():
    (head, ws, sbits, zz, codes), = _read_golden("partial_group.txt")
    K, g = (int(v) for v in head.split())
    W = _f16([float(v) for v in ws.split()])[None, :]
    q, s, z = oracle.quantize(W, g)
    assert list(s[0].view(np.uint16)) == [int(b, 16) for b in sbits.split()]
    assert list(z[0]) == [int(v) for v in zz.split()]
    assert list(q[0]) == [int(c) for c in codes.split()]
    # and the GEMM over it: x = ones gives the sum of the dequantized row, by hand:
    # group 0: (-5-2+0+1+4+5+7+10) * 1639/16384, group 1: (7-7+4+0) * 1093/16384
    qw, zw = oracle.pack_nibbles(q), oracle.pack_nibbles(z)
    y = oracle.gemm(np.ones((1, K), np.float16), qw, s, zw, 1, K, g)
    assert y[0, 0] == 20 * 1639 / 16384 + 4 * 1093 / 16384


# ------------------------------------------------------------------------- pack


def test_pack_golden_words():
    for kind, codes, word in _read_golden("layout_words.txt"):
        c = [int(v) for v in codes.split()]
        if kind == "canonical":
            got = oracle.pack_nibbles(np.array([c], np.uint8))
            assert got.shape == (1, 1) and int(got[0, 0]) == int(word, 16)


def test_pack_roundtrip_and_padding():
    rng = np.random.default_rng(5)
    for cols in (1, 7, 8, 9, 63, 500):
        v = rng.integers(0, 16, (5, cols)).astype(np.uint8)
        p = oracle.pack_nibbles(v)
        assert p.shape == (5, -(-cols // 8))
        assert (oracle.unpack_nibbles(p, cols) == v).all()
        if cols % 8:
            assert (p[:, -1] >> np.uint32(4 * (cols % 8)) == 0).all()  # padding nibbles are 0


# ----------------------------------------------------------------------- repack


def test_repack_golden_tile_words():
    for kind, codes, word in _read_golden("layout_words.txt"):
        if kind != "tiled":
            continue
        c = np.array([[int(v) for v in codes.split()]], np.uint8)
        qw = oracle.pack_nibbles(c)
        s = np.ones((1, 1), np.float16)
        zw = np.zeros((1, 1), np.uint32)
        buf = oracle.repack(qw, s, zw, 1, 8, 8)
        assert buf.size == 4096 + 320
        assert int(buf[:4].view(np.uint32)[0]) == int(word, 16)
        assert (buf[4:4096] == 0).all()
        assert int(buf[4096:4098].view(np.uint16)[0]) == 0x3C00


def test_repack_golden_positions():
    # one non-zero code, scale or zero at a time in a 300 x 200, g = 24 layer: the repacked buffer
    # must hold it at the hand-derived byte (and nibble half) and be zero everywhere else; the cases
    # cover rows r > 0, the second K half h = 1, words i > 0, K blocks b > 0, weight tiles t > 0 and
    # odd rows' zero nibbles
    N, K, g = 300, 200, 24
    G = oracle.ngroups(K, g)
    for kind, n, kj, byte, half in _read_golden("tile_positions.txt"):
        n, kj, byte = int(n), int(kj), int(byte)
        q = np.zeros((N, K), np.uint8)
        z = np.zeros((N, G), np.uint8)
        s = np.zeros((N, G), np.float16)
        if kind == "code":
            q[n, kj] = 0xB
        elif kind == "zero":
            z[n, kj] = 0xB
        else:
            s[n, kj] = np.uint16(0x1234).view(np.float16)
        buf = oracle.repack(oracle.pack_nibbles(q), s, oracle.pack_nibbles(z), N, K, g)
        assert buf.size == 57792
        nz = np.flatnonzero(buf)
        if kind == "scale":
            assert list(nz) == [byte, byte + 1] and buf[byte] == 0x34 and buf[byte + 1] == 0x12, (kind, n, kj)
        else:
            assert list(nz) == [byte], (kind, n, kj, nz[:4])
            assert buf[byte] == (0x0B if half == "low" else 0xB0), (kind, n, kj, hex(buf[byte]))


@pytest.mark.parametrize("N,K,g", [(1, 8, 8), (130, 72, 8), (288, 288, 256), (256, 512, 128), (200, 4000 // 10, 128),
                                   (129, 136, 24)])
def test_repack_is_a_zero_padded_permutation(N, K, g):
    rng = np.random.default_rng(N + K)
    G = oracle.ngroups(K, g)
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    z = rng.integers(0, 16, (N, G)).astype(np.uint8)
    s = rng.standard_normal((N, G)).astype(np.float16)
    qw, zw = oracle.pack_nibbles(q), oracle.pack_nibbles(z)
    buf = oracle.repack(qw, s, zw, N, K, g)
    NT, KB = -(-N // 128), -(-K // 64)
    assert buf.size == NT * KB * 4096 + NT * G * 320
    # inverse map gives the canonical form back
    qw2, s2, zw2 = oracle.unrepack(buf, N, K, g)
    assert (qw2 == qw).all() and (s2.view(np.uint16) == s.view(np.uint16)).all() and (zw2 == zw).all()
    # the code region holds exactly the codes plus zero padding (a permutation)
    codes = buf[: NT * KB * 4096]
    nibs = np.concatenate([codes & 0xF, codes >> 4])
    hist = np.bincount(nibs, minlength=16)
    ref = np.bincount(q.ravel(), minlength=16)
    ref[0] += NT * 128 * KB * 64 - N * K
    assert (hist == ref).all()
    # each record's zero nibbles hold that n-tile's zeros of one group (multiset per (tile, group))
    meta = buf[NT * KB * 4096:].reshape(NT, G, 320)
    for t in range(NT):
        rows = slice(128 * t, min(N, 128 * t + 128))
        nrow = rows.stop - rows.start
        for j in range(0, G, max(1, G // 3)):
            zb = meta[t, j, 256:]
            zn = np.stack([zb & 0xF, zb >> 4], 1).ravel()[:128]
            assert sorted(zn[:nrow]) == sorted(z[rows, j]) and (zn[nrow:] == 0).all()
            sc = meta[t, j, :256].view(np.uint16)
            assert sorted(sc[:nrow]) == sorted(s[rows, j].view(np.uint16)) and (sc[nrow:] == 0).all()


# ----------------------------------------------------------------- dequant/gemm


def test_q_equal_z_decodes_to_exact_zero():
    N, K, g = 9, 40, 16
    G = oracle.ngroups(K, g)
    rng = np.random.default_rng(11)
    z = rng.integers(0, 16, (N, G)).astype(np.uint8)
    q = z[:, np.arange(K) // g]
    s = (rng.standard_normal((N, G)) * 100).astype(np.float16)
    w = oracle.dequant(oracle.pack_nibbles(q), s, oracle.pack_nibbles(z), N, K, g)
    assert (w == 0).all()


def test_dequant_hand_derived_values():
    rows = _read_golden("quantize_groups.txt")
    name, ws, sbits, zz, codes = rows[0]
    q = np.array([[int(c) for c in codes.split()]], np.uint8)
    s = np.array([[int(sbits, 16)]], np.uint16).view(np.float16)
    z = np.array([[int(zz)]], np.uint8)
    w = oracle.dequant(oracle.pack_nibbles(q), s, oracle.pack_nibbles(z), 1, 8, 8)
    assert list(w[0]) == [v * 1639 / 16384 for v in (-5, -2, 0, 1, 4, 5, 7, 10)]


def _canonical(N, K, g, seed=0):
    W = workloads.weights_f16(N, K, seed=seed)
    return oracle.pack(W, g)


def test_gemm_one_hot_rows_return_weight_columns():
    N, K, g = 37, 136, 32  # partial last group of 8
    qw, s, zw = _canonical(N, K, g)
    w = oracle.dequant(qw, s, zw, N, K, g)
    ks = [0, 1, 31, 32, 100, 128, 135]
    x = np.zeros((len(ks), K), np.float16)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y = oracle.gemm(x, qw, s, zw, N, K, g)
    for i, k in enumerate(ks):
        assert (y[i] == w[:, k]).all()


def test_gemm_equals_library_matmul():
    N, K, g, M = 96, 520, 128, 5
    qw, s, zw = _canonical(N, K, g)
    x = workloads.activations_f16(M, K)
    y = oracle.gemm(x, qw, s, zw, N, K, g)
    w = oracle.dequant(qw, s, zw, N, K, g)
    ref = x.astype(np.float64) @ w.T
    mag = np.abs(x.astype(np.float64)) @ np.abs(w).T
    assert (np.abs(y - ref) <= 1e-13 * mag).all()
    # sampled rows are the same numbers as the full product
    rows = np.array([4, 0, 2])
    assert (oracle.gemm(x, qw, s, zw, N, K, g, rows=rows) == y[rows]).all()
    # one thread and many threads agree exactly (same summation order)
    assert (oracle.gemm(x, qw, s, zw, N, K, g, nthreads=1) == y).all()


@pytest.mark.parametrize("M,N,K,g", [(1, 2, 8, 8), (2, 3, 40, 16), (3, 5, 24, 8), (2, 4, 72, 64)])
def test_gemm_exact_rational_brute_force(M, N, K, g):
    rng = np.random.default_rng(M * 100 + K)
    W = (rng.standard_normal((N, K)) * 0.5).astype(np.float16)
    x = rng.standard_normal((M, K)).astype(np.float16)
    q, s, z = oracle.quantize(W, g)
    y = oracle.gemm(x, oracle.pack_nibbles(q), s, oracle.pack_nibbles(z), N, K, g)
    for m in range(M):
        for n in range(N):
            terms = [_fr(x[m, k]) * (int(q[n, k]) - int(z[n, k // g])) * _fr(s[n, k // g]) for k in range(K)]
            exact = sum(terms, Fraction(0))
            bound = sum(abs(t) for t in terms) * Fraction(K, 2**52)
            assert abs(Fraction(y[m, n]) - exact) <= bound


def test_gemm_is_linear_in_x():
    N, K, g = 20, 264, 64
    qw, s, zw = _canonical(N, K, g)
    x1 = workloads.activations_f16(1, K, seed=3)
    x2 = workloads.activations_f16(1, K, seed=4)
    x12 = (x1.astype(np.float64) + x2.astype(np.float64))
    assert (x12.astype(np.float16).astype(np.float64) == x12).mean() > 0.3
    exact = x12.astype(np.float16).astype(np.float64) == x12
    x1[~exact] = 0
    x2[~exact] = 0
    x12 = (x1.astype(np.float64) + x2.astype(np.float64)).astype(np.float16)
    ya = oracle.gemm(x1, qw, s, zw, N, K, g) + oracle.gemm(x2, qw, s, zw, N, K, g)
    yb = oracle.gemm(x12, qw, s, zw, N, K, g)
    w = oracle.dequant(qw, s, zw, N, K, g)
    mag = (np.abs(x1.astype(np.float64)) + np.abs(x2.astype(np.float64))) @ np.abs(w).T
    assert (np.abs(ya - yb) <= 1e-13 * mag).all()


# ------------------------------------------------------------------ bf16, symmetric


def _bf16_val(b: int) -> float:
    """bf16 bits -> value through numpy's IEEE float32 (bf16 is the top half of a float32)."""
    return float(np.array([int(b) << 16], np.uint32).view(np.float32)[0])


def _bf16_rne_exact(v: float) -> int:
    """Exact round-to-nearest-even of a finite fp64 value to bfloat16 bits, by search over the grid
    in rational arithmetic (an independent formulation)."""
    if v == 0:
        return 0x8000 if np.signbit(v) else 0
    sign = 0x8000 if v < 0 else 0
    a = Fraction(abs(v))
    if a >= Fraction(2) ** 128 - Fraction(2) ** 119:  # the midpoint above the largest finite value
        return sign | 0x7F80
    # largest bf16 (bits, positive) whose value is <= a, by bisection over the ordered bit patterns
    lo, hi = 0, 0x7F7F
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if Fraction(_bf16_val(mid)) <= a:
            lo = mid
        else:
            hi = mid - 1
    below = lo
    if Fraction(_bf16_val(below)) == a:
        return sign | below
    above = below + 1
    d_lo = a - Fraction(_bf16_val(below))
    d_hi = (Fraction(2) ** 128 if above == 0x7F80 else Fraction(_bf16_val(above))) - a
    pick = below if d_lo < d_hi else above if d_hi < d_lo else (below if below % 2 == 0 else above)
    return sign | pick


def test_bf16_decode_matches_float32_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        ref = (bits << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_bf16_encode_rounds_to_nearest_even():
    rng = np.random.default_rng(321)
    # values that are exact float32: the bf16 rounding of the float32 bit pattern (ties to even on
    # the low 16 bits) is an independent statement of the same rounding
    f32 = (np.exp2(rng.uniform(-140, 127, 3000)) * rng.choice([-1.0, 1.0], 3000)).astype(np.float32)
    u = f32.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in f32], dtype=np.uint16)
    fin = np.isfinite(f32) & (np.abs(f32) < 3.3e38)
    assert (got[fin] == ref[fin]).all()
    # fp64 values between bf16 neighbours, exact ties, subnormals, overflow: exact rational rounding
    vals = [1.0, 1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, -(1.0 + 2.0**-8 + 2.0**-40), 2.0**-133, 2.0**-134,
            3 * 2.0**-135, 2.0**-126 - 2.0**-134, 3.3895313892515355e38, 3.39e38, -1e39, 0.333333333333]
    vals += list(rng.standard_normal(500) * np.exp2(rng.uniform(-130, 120, 500)))
    b = rng.integers(1, 0x7F7F, 300)
    mids = [(_bf16_val(v) + _bf16_val(v + 1)) / 2 for v in b]  # exact in fp64
    vals += mids + [np.nextafter(m, 0) for m in mids]
    for v in vals:
        assert oracle.double_to_bf16(v) == _bf16_rne_exact(v), v
    # hand values: ties go to the even neighbour
    assert oracle.double_to_bf16(1.0 + 2.0**-8) == 0x3F80
    assert oracle.double_to_bf16(1.0 + 3 * 2.0**-8) == 0x3F82
    assert oracle.double_to_bf16(2.0**-133) == 0x0001
    assert oracle.double_to_bf16(3.4e38) == 0x7F80


def _dtype_val(b: int, dtype: str) -> Fraction:
    return Fraction(_bf16_val(b)) if dtype == "bf16" else _val_bits(b)


def _smallest_at_least(r: Fraction, dtype: str) -> int:
    """Exact: the least positive value of the type (bits) that is >= r."""
    b = _bf16_rne_exact(float(r)) if dtype == "bf16" else int(np.float16(float(r)).view(np.uint16))
    b &= 0x7FFF
    while _dtype_val(b, dtype) < r:
        b += 1
    while b > 0 and _dtype_val(b - 1, dtype) >= r:
        b -= 1
    return b


def _quantize_exact_ex(w, K: int, g: int, dtype: str, symmetric: bool):
    """The definition in exact rational arithmetic for either type and either form."""
    one = 0x3F80 if dtype == "bf16" else 0x3C00
    G = -(-K // g)
    q, s, z = [0] * K, [0] * G, [0] * G
    for j in range(G):
        grp = w[j * g:min((j + 1) * g, K)]
        lo, hi = min([Fraction(0)] + grp), max([Fraction(0)] + grp)
        if symmetric:
            amax = max(hi, -lo)
            lo, hi = -amax, amax
        r = hi - lo
        zj = 8 if symmetric else 0
        if r == 0:
            s[j], z[j] = one, zj
            for i in range(len(grp)):
                q[j * g + i] = zj
            continue
        sb = _smallest_at_least(r / 15, dtype)
        sv = _dtype_val(sb, dtype)
        if not symmetric:
            zj = min(15, max(0, round(-lo / sv)))
        s[j], z[j] = sb, zj
        for i, wk in enumerate(grp):
            q[j * g + i] = min(15, max(0, round(wk / sv) + zj))
    return q, s, z


@pytest.mark.parametrize("dtype,symmetric", [("f16", True), ("bf16", False), ("bf16", True)])
@pytest.mark.parametrize("K,g,seed", [(40, 16, 1), (24, 8, 2), (100, 32, 3), (288, 256, 4), (7, 8, 6)])
def test_quantize_variants_equal_exact_rational_definition(dtype, symmetric, K, g, seed):
    rng = np.random.default_rng(seed + 100)
    N = 5
    Wf = (rng.standard_normal((N, K)) * rng.choice([0.02, 1.0, 300.0], (N, 1))).astype(np.float32)
    Wf[0, : min(K, g)] = 0
    Wf[1] = np.abs(Wf[1])
    Wf[2] = -np.abs(Wf[2])
    if dtype == "bf16":
        W = workloads.f32_to_bf16_bits(Wf)
        vals = [[Fraction(_bf16_val(b)) for b in row] for row in W]
    else:
        W = Wf.astype(np.float16)
        vals = [[_fr(v) for v in row] for row in W]
    q, s, z = oracle.quantize(W, g, dtype=dtype, symmetric=symmetric)
    sbits = s.view(np.uint16) if dtype == "f16" else s
    for n in range(N):
        qe, se, ze = _quantize_exact_ex(vals[n], K, g, dtype, symmetric)
        assert list(q[n]) == qe
        assert list(sbits[n]) == se
        assert list(z[n]) == ze


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_symmetric_invariants(dtype):
    N, K, g = 64, 1000, 128
    W = workloads.weights_bf16(N, K, seed=8) if dtype == "bf16" else workloads.weights_f16(N, K, seed=8)
    q, s, z = oracle.quantize(W, g, dtype=dtype, symmetric=True)
    assert (z == 8).all() and q.max() <= 15
    sbits = s.view(np.uint16) if dtype == "f16" else s
    dec = (lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)) if dtype == "bf16" else \
        (lambda b: b.view(np.float16).astype(np.float64))
    w = dec(W if dtype == "bf16" else W.view(np.uint16))
    sv = dec(sbits)
    idx = np.arange(K) // g
    what = (q.astype(np.float64) - 8) * sv[:, idx]
    assert (np.abs(w - what) <= sv[:, idx] / 2 * (1 + 2.0**-40)).all()
    for j in range(oracle.ngroups(K, g)):
        amax = np.abs(w[:, j * g:min((j + 1) * g, K)]).max(1)
        assert (15 * sv[:, j] >= 2 * amax).all()
        prev = dec((sbits[:, j] - 1).astype(np.uint16))
        assert (15 * prev < 2 * amax).all()


def test_quantize_variants_hand_derived():
    for name, dtype, sym, ws, sbits, zz, codes in _read_golden("quantize_variants.txt"):
        vals = np.array([float(v) for v in ws.split()], np.float32)
        W = workloads.f32_to_bf16_bits(vals)[None, :] if dtype == "bf16" else vals.astype(np.float16)[None, :]
        q, s, z = oracle.quantize(W, 8, dtype=dtype, symmetric=bool(int(sym)))
        sb = s.view(np.uint16) if dtype == "f16" else s
        assert int(sb[0, 0]) == int(sbits, 16), name
        assert int(z[0, 0]) == int(zz), name
        assert list(q[0]) == [int(c) for c in codes.split()], name


@pytest.mark.parametrize("dtype,symmetric", [("bf16", False), ("bf16", True), ("f16", True)])
def test_gemm_variants_one_hot_and_matmul(dtype, symmetric):
    N, K, g, M = 70, 200, 64, 5
    W = workloads.weights_bf16(N, K, seed=9) if dtype == "bf16" else workloads.weights_f16(N, K, seed=9)
    qw, s, zw = oracle.pack(W, g, dtype=dtype, symmetric=symmetric)
    wd = oracle.dequant(qw, s, zw, N, K, g, dtype=dtype)
    # the dequantized weights are the exact products (q - z) s of the type's scale values
    q = oracle.unpack_nibbles(qw, K).astype(np.float64)
    z = oracle.unpack_nibbles(zw, oracle.ngroups(K, g)).astype(np.float64)
    sv = ((s.astype(np.uint32) << 16).view(np.float32) if dtype == "bf16" else s).astype(np.float64)
    idx = np.arange(K) // g
    assert (wd == (q - z[:, idx]) * sv[:, idx]).all()
    # one-hot activation rows return weight columns exactly
    ks = [0, 63, 64, 199]
    one = 0x3F80 if dtype == "bf16" else 0x3C00
    x = np.zeros((len(ks), K), np.uint16)
    for i, k in enumerate(ks):
        x[i, k] = one
    y = oracle.gemm(x if dtype == "bf16" else x.view(np.float16), qw, s, zw, N, K, g, dtype=dtype)
    assert (y == wd[:, ks].T).all()
    # random activations against numpy's fp64 matmul
    xb = workloads.activations_bf16(M, K) if dtype == "bf16" else workloads.activations_f16(M, K)
    xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64) if dtype == "bf16" else \
        xb.astype(np.float64)
    y = oracle.gemm(xb, qw, s, zw, N, K, g, dtype=dtype)
    assert np.allclose(y, xv @ wd.T, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ epilogues

def test_silu_closed_forms():
    # sigmoid(ln 3) = 3/4, so silu(ln 3) = (3/4) ln 3; silu(0) = 0; silu(v) - silu(-v) = v for every v
    # (v sigmoid(v) + v sigmoid(-v) = v); and the tanh form silu(v) = v/2 (1 + tanh(v/2))
    assert oracle.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert oracle.silu(0.0) == 0.0
    v = np.linspace(-40, 40, 1001)
    assert np.allclose(oracle.silu(v) - oracle.silu(-v), v, rtol=1e-14, atol=1e-14)
    # (the tanh form cancels for v << 0: an absolute bound of a few ulp of |v|)
    assert np.allclose(oracle.silu(v), 0.5 * v * (1 + np.tanh(0.5 * v)), rtol=1e-13, atol=1e-13)
    assert oracle.silu(-800.0) == 0.0 and oracle.silu(800.0) == 800.0  # saturates without overflow


def test_silu_mul_hand_example():
    # columns alternate gate, up: (ln 3, 2) -> (3/4) ln 3 * 2; (0, 5) -> 0; (-ln 3, 4) -> -(1/4) ln 3 * 4
    y = np.array([[math.log(3.0), 2.0, 0.0, 5.0, -math.log(3.0), 4.0]])
    h = oracle.silu_mul(y)
    assert h.shape == (1, 3)
    assert h[0] == pytest.approx([1.5 * math.log(3.0), 0.0, -math.log(3.0)], rel=1e-15)


def test_qkv_split_hand_example():
    # head_dim 2, two query heads per group, two groups: N = 2 * (2 + 2) * 2 = 16 columns
    y = np.arange(16, dtype=np.float64)[None, :]
    q, k, v = oracle.qkv_split(y, 2, 2)
    assert q.tolist() == [[0, 1, 2, 3, 8, 9, 10, 11]]
    assert k.tolist() == [[4, 5, 12, 13]]
    assert v.tolist() == [[6, 7, 14, 15]]
    # multi-head attention (one query head per group): q, k, v heads interleave per group
    q, k, v = oracle.qkv_split(np.arange(12)[None, :], 2, 1)
    assert q.tolist() == [[0, 1, 6, 7]] and k.tolist() == [[2, 3, 8, 9]] and v.tolist() == [[4, 5, 10, 11]]


def test_weight_row_orders_match_the_epilogues():
    # the binding's offline row orders, read back by the oracle's epilogue maps
    import torch

    import w4a16_group_quantized_gb300 as w4

    d, r, groups, K = 4, 3, 2, 1
    wq = torch.arange(groups * r * d, dtype=torch.float64)[:, None]
    wk = 1000 + torch.arange(groups * d, dtype=torch.float64)[:, None]
    wv = 2000 + torch.arange(groups * d, dtype=torch.float64)[:, None]
    fused = w4.qkv_head_group_rows(wq, wk, wv, d)
    q, k, v = oracle.qkv_split(fused.numpy().T, d, r)  # one token with x = 1: y = the weight column
    assert (q[0] == wq[:, 0].numpy()).all() and (k[0] == wk[:, 0].numpy()).all() and (v[0] == wv[:, 0].numpy()).all()
    gate = torch.arange(5, dtype=torch.float64)[:, None]
    up = 100 + torch.arange(5, dtype=torch.float64)[:, None]
    il = w4.interleave_gate_up(gate, up).numpy().T
    assert (il[0, 0::2] == gate[:, 0].numpy()).all() and (il[0, 1::2] == up[:, 0].numpy()).all()
