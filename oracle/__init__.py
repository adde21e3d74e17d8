"""CPU oracle for the W4A16 group-quantized linear layer.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg may import this package. The product library never
does, and this package imports nothing from it: the two share no code.

The arithmetic lives in ``w4a16_oracle.c`` (plain C, fp64, compiled with
``-ffp-contract=off``); this module compiles it with gcc on first use and
wraps it with numpy arrays. fp16 values cross the boundary as their uint16
bit patterns.

Parity pins for every function here are in ``tests/test_oracle.py``; none is
left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc_w4a16.so")
_lock = threading.Lock()
_lib = None

TN, TK, TILE_BYTES, REC_BYTES = 128, 64, 4096, 320


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liborc_w4a16.so`` (gcc, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int32
        lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_half_to_double.restype = ctypes.c_double
        lib.orc_double_to_half.argtypes = [ctypes.c_double]
        lib.orc_double_to_half.restype = ctypes.c_uint16
        lib.orc_quantize.argtypes = [P, I64, I64, I32, P, P, P]
        lib.orc_quantize.restype = ctypes.c_int
        lib.orc_quantize_ex.argtypes = [P, I64, I64, I32, I32, I32, P, P, P]
        lib.orc_quantize_ex.restype = ctypes.c_int
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_double_to_bf16.argtypes = [ctypes.c_double]
        lib.orc_double_to_bf16.restype = ctypes.c_uint16
        lib.orc_dequant_ex.argtypes = [P, P, P, I64, I64, I32, I32, P]
        lib.orc_dequant_ex.restype = None
        lib.orc_gemm_rows_ex.argtypes = [P, I64, P, I64, P, P, P, I64, I64, I32, I32, P, ctypes.c_int]
        lib.orc_gemm_rows_ex.restype = ctypes.c_int
        lib.orc_pack_nibbles.argtypes = [P, I64, I64, P]
        lib.orc_pack_nibbles.restype = None
        lib.orc_unpack_nibbles.argtypes = [P, I64, I64, P]
        lib.orc_unpack_nibbles.restype = None
        lib.orc_repacked_bytes.argtypes = [I64, I64, I32]
        lib.orc_repacked_bytes.restype = I64
        lib.orc_repack.argtypes = [P, P, P, I64, I64, I32, P]
        lib.orc_repack.restype = None
        lib.orc_unrepack.argtypes = [P, I64, I64, I32, P, P, P]
        lib.orc_unrepack.restype = None
        lib.orc_dequant.argtypes = [P, P, P, I64, I64, I32, P]
        lib.orc_dequant.restype = None
        lib.orc_gemm_rows.argtypes = [P, I64, P, I64, P, P, P, I64, I64, I32, P, ctypes.c_int]
        lib.orc_gemm_rows.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


DTYPES = {"f16": 0, "bf16": 1}


def _bits(a) -> np.ndarray:
    """fp16 array (or uint16 bits of fp16 or bf16 values) -> contiguous uint16 bits."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


def _dt(dtype: str) -> int:
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}")
    return DTYPES[dtype]


def _scales_out(s: np.ndarray, dtype: str) -> np.ndarray:
    return s.view(np.float16) if dtype == "f16" else s


def ngroups(k: int, g: int) -> int:
    return -(-k // g)


# ----------------------------------------------------------------- fp16

def half_to_double(bits: int) -> float:
    return _load().orc_half_to_double(int(bits) & 0xFFFF)


def double_to_half(v: float) -> int:
    return int(_load().orc_double_to_half(float(v)))


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits) & 0xFFFF)


def double_to_bf16(v: float) -> int:
    return int(_load().orc_double_to_bf16(float(v)))


# ------------------------------------------------------------ quantize

def quantize(W, g: int, dtype: str = "f16", symmetric: bool = False):
    """W [N,K] (fp16, or uint16 bits of dtype) -> (q uint8 [N,K], s [N,G], z uint8 [N,G]).
    s is fp16 for dtype 'f16' and uint16 bf16 bits for 'bf16'. symmetric: z = 8, range +-max|w|."""
    Wb = _bits(W)
    N, K = Wb.shape
    G = ngroups(K, g)
    q = np.zeros((N, K), np.uint8)
    s = np.zeros((N, G), np.uint16)
    z = np.zeros((N, G), np.uint8)
    rc = _load().orc_quantize_ex(_ptr(Wb), N, K, g, _dt(dtype), int(bool(symmetric)), _ptr(q), _ptr(s), _ptr(z))
    if rc != 0:
        raise ValueError(f"orc_quantize failed ({rc}): {'non-finite weight' if rc == -2 else 'bad arguments'}")
    return q, _scales_out(s, dtype), z


def pack_nibbles(v: np.ndarray) -> np.ndarray:
    """[rows, cols] values 0..15 -> [rows, ceil(cols/8)] uint32 (element i of a word at bits 4i..)."""
    v = np.ascontiguousarray(v, dtype=np.uint8)
    rows, cols = v.shape
    out = np.zeros((rows, -(-cols // 8)), np.uint32)
    _load().orc_pack_nibbles(_ptr(v), rows, cols, _ptr(out))
    return out


def unpack_nibbles(words: np.ndarray, cols: int) -> np.ndarray:
    words = np.ascontiguousarray(words, dtype=np.uint32)
    rows = words.shape[0]
    out = np.zeros((rows, cols), np.uint8)
    _load().orc_unpack_nibbles(_ptr(words), rows, cols, _ptr(out))
    return out


def pack(W, g: int, dtype: str = "f16", symmetric: bool = False):
    """The canonical packed form: (qw uint32 [N,ceil(K/8)], scales [N,G], zeros uint32 [N,ceil(G/8)])."""
    q, s, z = quantize(W, g, dtype, symmetric)
    return pack_nibbles(q), s, pack_nibbles(z)


# -------------------------------------------------------------- repack

def repacked_bytes(N: int, K: int, g: int) -> int:
    return int(_load().orc_repacked_bytes(N, K, g))


def repack(qw, scales, zeros, N: int, K: int, g: int) -> np.ndarray:
    qw = np.ascontiguousarray(qw, dtype=np.uint32)
    sb = _bits(scales)
    zw = np.ascontiguousarray(zeros, dtype=np.uint32)
    out = np.zeros(repacked_bytes(N, K, g), np.uint8)
    _load().orc_repack(_ptr(qw), _ptr(sb), _ptr(zw), N, K, g, _ptr(out))
    return out


def unrepack(buf, N: int, K: int, g: int):
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    assert buf.size == repacked_bytes(N, K, g)
    G = ngroups(K, g)
    qw = np.zeros((N, -(-K // 8)), np.uint32)
    s = np.zeros((N, G), np.uint16)
    zw = np.zeros((N, -(-G // 8)), np.uint32)
    _load().orc_unrepack(_ptr(buf), N, K, g, _ptr(qw), _ptr(s), _ptr(zw))
    return qw, s.view(np.float16), zw


# ------------------------------------------------------ dequant / gemm

def dequant(qw, scales, zeros, N: int, K: int, g: int, dtype: str = "f16") -> np.ndarray:
    """w [N,K] fp64 = (q - z) * s, exact (s fp16, or bf16 bits for dtype 'bf16')."""
    qw = np.ascontiguousarray(qw, dtype=np.uint32)
    sb = _bits(scales)
    zw = np.ascontiguousarray(zeros, dtype=np.uint32)
    w = np.zeros((N, K), np.float64)
    _load().orc_dequant_ex(_ptr(qw), _ptr(sb), _ptr(zw), N, K, g, _dt(dtype), _ptr(w))
    return w


def gemm(x, qw, scales, zeros, N: int, K: int, g: int, rows=None, nthreads: int | None = None,
         dtype: str = "f16") -> np.ndarray:
    """y [R,N] fp64 = x[rows] . dequant(W)^T by the naive triple loop (rows=None: all M rows).
    x and the scales are fp16, or uint16 bf16 bits for dtype 'bf16'."""
    xb = _bits(x)
    M, Kx = xb.shape
    assert Kx == K
    qw = np.ascontiguousarray(qw, dtype=np.uint32)
    sb = _bits(scales)
    zw = np.ascontiguousarray(zeros, dtype=np.uint32)
    if rows is None:
        R, rows_p, rows_arr = M, None, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        assert rows_arr.ndim == 1 and (rows_arr >= 0).all() and (rows_arr < M).all()
        R, rows_p = rows_arr.size, _ptr(rows_arr)
    y = np.zeros((R, N), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = _load().orc_gemm_rows_ex(_ptr(xb), M, rows_p, R, _ptr(qw), _ptr(sb), _ptr(zw), N, K, g, _dt(dtype),
                                  _ptr(y), int(nthreads))
    if rc != 0:
        raise MemoryError("orc_gemm_rows: allocation failed")
    return y


# ----------------------------------------------------------- epilogues
# Plain fp64 restatements of the two output epilogues, applied to the oracle's unrounded GEMM output.

def silu(v) -> np.ndarray:
    """silu(v) = v * sigmoid(v) = v / (1 + e^-v) in fp64: the gated MLP activation (SiLU / swish)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def silu_mul(y) -> np.ndarray:
    """h [R, N/2] = silu(gate) * up for a fused gate/up output y [R, N] whose columns alternate gate
    (even column 2j) and up (odd column 2j + 1)."""
    y = np.asarray(y, dtype=np.float64)
    assert y.ndim == 2 and y.shape[1] % 2 == 0
    return silu(y[:, 0::2]) * y[:, 1::2]


def qkv_split(y, head_dim: int, q_per_group: int):
    """(q, k, v) from a fused q/k/v output y [R, N] whose columns come in head groups: per group,
    q_per_group query heads, one key head and one value head of head_dim columns each. q is
    [R, groups * q_per_group * head_dim] (the groups' query heads in order), k and v [R, groups * head_dim]."""
    y = np.asarray(y)
    R, N = y.shape
    d, r = head_dim, q_per_group
    span = (r + 2) * d
    assert N % span == 0
    groups = N // span
    yg = y.reshape(R, groups, r + 2, d)
    q = yg[:, :, :r, :].reshape(R, groups * r * d)
    k = yg[:, :, r, :].reshape(R, groups * d)
    v = yg[:, :, r + 1, :].reshape(R, groups * d)
    return q, k, v
