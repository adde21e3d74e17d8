"""Thin Python binding of libw4a16.so (the C ABI in include/w4a16.h).

Argument marshalling only: every step of the quantized linear layer runs in
the library's CUDA kernels. PyTorch supplies device memory and the current
stream. There is no CPU or PyTorch fallback: if the library is missing or a
call fails, a ``W4Error`` is raised.

Names follow the C ABI:

    qw, scales, zeros = w4_pack(W, g)                 # fp16 [N,K] cuda -> canonical packed form
    packed = w4_repack(qw, scales, zeros, N, K, g)    # -> the GEMM's tile layout (uint8 buffer)
    y = w4a16_gemm(x, packed, N, K, g)                # fp16 [M,K] -> fp16 [M,N]

uint32 words are carried in torch.int32 tensors (same bits).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "W4Error", "lib_path", "load", "w4_pack", "w4_repack", "w4_repacked_bytes", "w4a16_gemm",
    "w4a16_gemm_ex", "w4a16_gemm_opts", "w4a16_workspace_bytes", "w4a16_workspace_bytes_ex",
    "w4a16_workspace_bytes_opts", "w4a16_gemm_plan", "w4_last_device_error", "w4_status_string", "Workspace",
    "Options", "STATUS", "KERNEL_DECODE", "KERNEL_TMEM", "FLAG_WEIGHTS_STATIC", "FLAG_TEST_TIMEOUT",
    "Epilogue", "Problem", "EPI_NONE", "EPI_SILU_MUL", "EPI_QKV_SPLIT", "w4a16_gemm_grouped",
    "w4a16_grouped_workspace_bytes", "w4a16_gemm_silu_mul", "w4a16_gemm_qkv", "interleave_gate_up",
    "qkv_head_group_rows",
]

KERNEL_DECODE = 1
KERNEL_TMEM = 2
FLAG_WEIGHTS_STATIC = 1
FLAG_TEST_TIMEOUT = 2


class Options(ctypes.Structure):
    """w4a16_options of the C ABI (all zero: automatic)."""

    _fields_ = [("kernel", ctypes.c_int32), ("block_n", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("cluster", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("wait_limit_cycles", ctypes.c_uint64), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]

EPI_NONE, EPI_SILU_MUL, EPI_QKV_SPLIT = 0, 1, 2


class Epilogue(ctypes.Structure):
    """w4a16_epilogue of the C ABI."""

    _fields_ = [("kind", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("q_per_group", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("k_dev", ctypes.c_void_p), ("v_dev", ctypes.c_void_p)]


class Problem(ctypes.Structure):
    """w4a16_problem of the C ABI."""

    _fields_ = [("x_dev", ctypes.c_void_p), ("packed_dev", ctypes.c_void_p), ("y_dev", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("epilogue", Epilogue)]


_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libw4a16.so")

STATUS = {
    0: "W4_OK", 1: "W4_ERR_INVALID_ARG", 2: "W4_ERR_UNSUPPORTED_SHAPE", 3: "W4_ERR_MISALIGNED",
    4: "W4_ERR_WORKSPACE_TOO_SMALL", 5: "W4_ERR_CUDA", 6: "W4_ERR_TIMEOUT",
}

_lib = None
_lock = threading.Lock()


class W4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {w4_status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Load libw4a16.so (built by ``python -m w4a16_group_quantized_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(lib_path):
            raise ImportError(f"{lib_path} is missing: build it with `python -m w4a16_group_quantized_gb300.build`")
        lib = ctypes.CDLL(lib_path)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        sigs = {
            "w4_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "w4_pack": ([P, I64, I64, I32, P, P, P, P], ctypes.c_int),
            "w4_pack_ex": ([P, I64, I64, I32, I32, I32, P, P, P, P], ctypes.c_int),
            "w4_repacked_bytes": ([I64, I64, I32], SZ),
            "w4_repack": ([P, P, P, I64, I64, I32, P, P], ctypes.c_int),
            "w4a16_workspace_bytes": ([I64, I64, I64, I32], SZ),
            "w4a16_workspace_bytes_ex": ([I64, I64, I64, I32, I32, I32, I32], SZ),
            "w4a16_gemm": ([P, P, I64, I64, I64, I32, P, P, SZ, P], ctypes.c_int),
            "w4a16_gemm_ex": ([P, P, I64, I64, I64, I32, P, P, SZ, I32, I32, I32, P], ctypes.c_int),
            "w4a16_gemm_plan": ([I64, I64, I64, I32, ctypes.POINTER(I32), ctypes.POINTER(I32),
                                 ctypes.POINTER(I32)], ctypes.c_int),
            "w4_last_device_error": ([P, P], ctypes.c_int),
            "w4a16_gemm_opts": ([P, P, I64, I64, I64, I32, P, P, SZ, ctypes.POINTER(Options), P], ctypes.c_int),
            "w4a16_workspace_bytes_opts": ([I64, I64, I64, I32, ctypes.POINTER(Options)], SZ),
            "w4a16_gemm_grouped": ([ctypes.POINTER(Problem), I32, I64, I32, P, SZ, ctypes.POINTER(Options), P],
                                   ctypes.c_int),
            "w4a16_grouped_workspace_bytes": ([ctypes.POINTER(Problem), I32, I64, I32, ctypes.POINTER(Options)], SZ),
        }
        for name, (args, res) in sigs.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def w4_status_string(status: int) -> str:
    return load().w4_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise W4Error(rc, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str) -> ctypes.c_void_p:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _ngroups(K: int, g: int) -> int:
    return -(-K // g)


_DTYPES = {torch.float16: 0, torch.bfloat16: 1}


def w4_pack(W: torch.Tensor, g: int, stream=None, symmetric: bool = False):
    """fp16 or bf16 W [N,K] (cuda) -> (qw int32 [N,ceil(K/8)], scales [N,G] of W's dtype,
    zeros int32 [N,ceil(G/8)]). symmetric: z = 8 and the range +-max|w| (w4_pack_ex)."""
    if W.dtype not in _DTYPES or W.dim() != 2:
        raise ValueError("W must be a 2-D fp16 or bf16 tensor")
    N, K = W.shape
    G = _ngroups(K, g) if g > 0 else 1
    qw = torch.empty((N, -(-K // 8)), dtype=torch.int32, device=W.device)
    scales = torch.empty((N, G), dtype=W.dtype, device=W.device)
    zeros = torch.empty((N, -(-G // 8)), dtype=torch.int32, device=W.device)
    _check(load().w4_pack_ex(_dev(W, "W"), N, K, g, _DTYPES[W.dtype], int(bool(symmetric)), _dev(qw, "qw"),
                             _dev(scales, "scales"), _dev(zeros, "zeros"), _stream(stream)), "w4_pack")
    return qw, scales, zeros


def w4_repacked_bytes(N: int, K: int, g: int) -> int:
    return int(load().w4_repacked_bytes(N, K, g))


def w4_repack(qw: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor, N: int, K: int, g: int,
              out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Canonical packed form -> uint8 buffer in the GEMM's tile layout."""
    nbytes = w4_repacked_bytes(N, K, g)
    if nbytes == 0:
        raise W4Error(1, "w4_repack")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=qw.device)
    elif out.numel() * out.element_size() < nbytes:
        raise ValueError("out is too small")
    _check(load().w4_repack(_dev(qw, "qw"), _dev(scales, "scales"), _dev(zeros, "zeros"), N, K, g,
                            _dev(out, "out"), _stream(stream)), "w4_repack")
    return out


def w4a16_workspace_bytes(M: int, N: int, K: int, g: int) -> int:
    return int(load().w4a16_workspace_bytes(M, N, K, g))


def w4a16_workspace_bytes_ex(M: int, N: int, K: int, g: int, block_n: int, ctas: int, schedule: int) -> int:
    return int(load().w4a16_workspace_bytes_ex(M, N, K, g, block_n, ctas, schedule))


def w4a16_workspace_bytes_opts(M: int, N: int, K: int, g: int, opts: Options) -> int:
    return int(load().w4a16_workspace_bytes_opts(M, N, K, g, ctypes.byref(opts)))


def w4a16_gemm_plan(M: int, N: int, K: int, g: int):
    """(block_n, ctas, schedule) that w4a16_gemm picks on the current device (schedule 1 stream-K, 2 whole tiles)."""
    b, s, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().w4a16_gemm_plan(M, N, K, g, ctypes.byref(b), ctypes.byref(s), ctypes.byref(c)), "w4a16_gemm_plan")
    return b.value, s.value, c.value


class Workspace:
    """A zero-filled device workspace that grows on demand (reuse it across calls on one stream)."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = torch.zeros(256, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 2 * self.buf.numel()), dtype=torch.uint8, device=self.device)
        return self.buf


def _gemm_common(x, packed, N, K, g, y, workspace, block_n, ctas, schedule, stream):
    if x.dtype != torch.float16 or x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x must be fp16 [M, K]")
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    elif y.dtype != torch.float16 or tuple(y.shape) != (M, N):
        raise ValueError("y must be fp16 [M, N]")
    need = w4a16_workspace_bytes_ex(M, N, K, g, block_n, ctas, schedule)
    if need == 0:
        raise W4Error(1, "w4a16_workspace_bytes")
    if workspace is None:
        workspace = Workspace(x.device)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    nbytes = ws.numel() * ws.element_size()
    lib = load()
    if block_n == 0 and ctas == 0 and schedule == 0:
        rc = lib.w4a16_gemm(_dev(x, "x"), _dev(packed, "packed"), M, N, K, g, _dev(y, "y"), _dev(ws, "workspace"),
                            nbytes, _stream(stream))
    else:
        rc = lib.w4a16_gemm_ex(_dev(x, "x"), _dev(packed, "packed"), M, N, K, g, _dev(y, "y"),
                               _dev(ws, "workspace"), nbytes, block_n, ctas, schedule, _stream(stream))
    _check(rc, "w4a16_gemm")
    return y


def w4a16_gemm(x: torch.Tensor, packed: torch.Tensor, N: int, K: int, g: int, y: torch.Tensor | None = None,
               workspace=None, stream=None, weights_static: bool = False) -> torch.Tensor:
    """y [M,N] = x [M,K] . dequant(packed)^T, fp16 or bf16 (x's dtype: the packed scales must be of the
    same type). ``workspace``: a Workspace or a zeroed uint8 tensor. ``weights_static``: the kernel
    launched just before this call on the stream does not write ``packed`` (W4_FLAG_WEIGHTS_STATIC: the
    decode kernel may then fetch weights before that kernel ends)."""
    if weights_static or x.dtype == torch.bfloat16:
        return w4a16_gemm_opts(x, packed, N, K, g, flags=FLAG_WEIGHTS_STATIC if weights_static else 0, y=y,
                               workspace=workspace, stream=stream)
    return _gemm_common(x, packed, N, K, g, y, workspace, 0, 0, 0, stream)


def w4a16_gemm_opts(x: torch.Tensor, packed: torch.Tensor, N: int, K: int, g: int, *, kernel: int = 0,
                    block_n: int = 0, ctas: int = 0, schedule: int = 0, cluster: int = 0, flags: int = 0,
                    wait_limit_cycles: int = 0, y: torch.Tensor | None = None, workspace=None,
                    stream=None) -> torch.Tensor:
    """w4a16_gemm with the options of w4a16_options (see include/w4a16.h); the dtype option follows x."""
    if x.dtype not in _DTYPES or x.dim() != 2 or x.shape[1] != K:
        raise ValueError("x must be fp16 or bf16 [M, K]")
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=x.dtype, device=x.device)
    elif y.dtype != x.dtype or tuple(y.shape) != (M, N):
        raise ValueError("y must be [M, N] of x's dtype")
    o = Options(kernel, block_n, ctas, schedule, cluster, flags, wait_limit_cycles, _DTYPES[x.dtype], 0)
    need = w4a16_workspace_bytes_opts(M, N, K, g, o)
    if need == 0:
        raise W4Error(1, "w4a16_workspace_bytes_opts")
    if workspace is None:
        workspace = Workspace(x.device)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    nbytes = ws.numel() * ws.element_size()
    rc = load().w4a16_gemm_opts(_dev(x, "x"), _dev(packed, "packed"), M, N, K, g, _dev(y, "y"),
                                _dev(ws, "workspace"), nbytes, ctypes.byref(o), _stream(stream))
    _check(rc, "w4a16_gemm_opts")
    return y


def w4a16_gemm_ex(x, packed, N, K, g, block_n: int = 0, ctas: int = 0, schedule: int = 0, y=None, workspace=None,
                  stream=None):
    """w4a16_gemm with the schedule forced: block_n in {8,16,32,64,128} (8: the register-operand decode
    kernel; 16..128: the tensor-memory kernel), ctas >= 1, schedule 1 stream-K or 2 whole tiles (0 = automatic
    for each)."""
    return _gemm_common(x, packed, N, K, g, y, workspace, block_n, ctas, schedule, stream)


def w4_last_device_error(workspace, stream=None) -> int:
    """Reads and clears the workspace's device error word (synchronises the stream). After
    W4_ERR_TIMEOUT the workspace's tile counters are undefined too: zero it before reuse."""
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    return int(load().w4_last_device_error(_dev(ws, "workspace"), _stream(stream)))


# ----------------------------------------------------------------------------- groups and epilogues

def _problem_array(problems, M, dtype, device):
    """(ctypes array of Problem, outputs per problem, tensors to keep alive)."""
    arr = (Problem * len(problems))()
    outs, keep = [], []
    for i, pr in enumerate(problems):
        x, packed, N, K = pr["x"], pr["packed"], int(pr["N"]), int(pr["K"])
        if x.dtype != dtype or x.dim() != 2 or tuple(x.shape) != (M, K):
            raise ValueError(f"problem {i}: x must be [{M}, {K}] of the group's dtype")
        epi = Epilogue()
        if pr.get("silu_mul"):
            epi.kind = EPI_SILU_MUL
            y = pr.get("y")
            if y is None:
                y = torch.empty((M, N // 2), dtype=dtype, device=device)
            elif y.dtype != dtype or tuple(y.shape) != (M, N // 2):
                raise ValueError(f"problem {i}: y must be [{M}, {N // 2}]")
            out = y
        elif pr.get("qkv"):
            head_dim, q_per_group = pr["qkv"]
            span = (q_per_group + 2) * head_dim
            if N % span:
                raise ValueError(f"problem {i}: N must be a multiple of (q_per_group + 2) * head_dim")
            groups = N // span
            epi.kind, epi.head_dim, epi.q_per_group = EPI_QKV_SPLIT, head_dim, q_per_group
            shapes = ((M, groups * q_per_group * head_dim), (M, groups * head_dim), (M, groups * head_dim))
            if pr.get("out") is not None:
                q, k, v = pr["out"]
                if any(t.dtype != dtype or tuple(t.shape) != sh for t, sh in zip((q, k, v), shapes)):
                    raise ValueError(f"problem {i}: out must be q, k, v of shapes {shapes}")
            else:
                q, k, v = (torch.empty(sh, dtype=dtype, device=device) for sh in shapes)
            epi.k_dev, epi.v_dev = k.data_ptr(), v.data_ptr()
            y, out = q, (q, k, v)
            keep += [k, v]
        else:
            y = pr.get("y")
            if y is None:
                y = torch.empty((M, N), dtype=dtype, device=device)
            elif y.dtype != dtype or tuple(y.shape) != (M, N):
                raise ValueError(f"problem {i}: y must be [{M}, {N}]")
            out = y
        arr[i] = Problem(_dev(x, "x").value, _dev(packed, "packed").value, _dev(y, "y").value, N, K, epi)
        outs.append(out)
        keep += [x, packed, y]
    return arr, outs, keep


def w4a16_grouped_workspace_bytes(problems, g: int, **opts) -> int:
    x0 = problems[0]["x"]
    arr, _, _ = _problem_array(problems, x0.shape[0], x0.dtype, x0.device)
    o = Options(opts.get("kernel", 0), opts.get("block_n", 0), opts.get("ctas", 0), opts.get("schedule", 0),
                opts.get("cluster", 0), opts.get("flags", 0), opts.get("wait_limit_cycles", 0), _DTYPES[x0.dtype], 0)
    return int(load().w4a16_grouped_workspace_bytes(arr, len(problems), x0.shape[0], g, ctypes.byref(o)))


def w4a16_gemm_grouped(problems, g: int, *, kernel: int = 0, block_n: int = 0, ctas: int = 0, schedule: int = 0,
                       cluster: int = 0, flags: int = 0, wait_limit_cycles: int = 0, workspace=None, stream=None):
    """Independent GEMMs of one M, g and dtype in one call (w4a16_gemm_grouped). Each problem is a dict
    with x [M, K], packed, N, K, and optionally y (the output), silu_mul=True (y [M, N/2] =
    silu(gate) * up for weight rows alternating gate, up) or qkv=(head_dim, q_per_group) (weight rows in
    head groups; the output is (q, k, v), given as out=(q, k, v) or allocated). Returns the outputs in
    order."""
    if not problems:
        raise ValueError("empty group")
    x0 = problems[0]["x"]
    if x0.dtype not in _DTYPES:
        raise ValueError("x must be fp16 or bf16")
    M = x0.shape[0]
    arr, outs, keep = _problem_array(problems, M, x0.dtype, x0.device)
    o = Options(kernel, block_n, ctas, schedule, cluster, flags, wait_limit_cycles, _DTYPES[x0.dtype], 0)
    need = int(load().w4a16_grouped_workspace_bytes(arr, len(problems), M, g, ctypes.byref(o)))
    if need == 0:
        raise W4Error(1, "w4a16_grouped_workspace_bytes")
    if workspace is None:
        workspace = Workspace(x0.device)
    ws = workspace.get(need) if isinstance(workspace, Workspace) else workspace
    nbytes = ws.numel() * ws.element_size()
    rc = load().w4a16_gemm_grouped(arr, len(problems), M, g, _dev(ws, "workspace"), nbytes, ctypes.byref(o),
                                   _stream(stream))
    _check(rc, "w4a16_gemm_grouped")
    del keep
    return outs


def w4a16_gemm_silu_mul(x, packed, N: int, K: int, g: int, y=None, workspace=None, stream=None, **opts):
    """h [M, N/2] = silu(x . gate^T) * (x . up^T) for packed weight rows alternating gate, up."""
    return w4a16_gemm_grouped([dict(x=x, packed=packed, N=N, K=K, y=y, silu_mul=True)], g, workspace=workspace,
                              stream=stream, **opts)[0]


def w4a16_gemm_qkv(x, packed, N: int, K: int, g: int, head_dim: int, q_per_group: int, workspace=None, stream=None,
                   **opts):
    """(q, k, v) of a fused projection whose weight rows come in head groups (see qkv_head_group_rows)."""
    return w4a16_gemm_grouped([dict(x=x, packed=packed, N=N, K=K, qkv=(head_dim, q_per_group))], g,
                              workspace=workspace, stream=stream, **opts)[0]


def interleave_gate_up(gate: torch.Tensor, up: torch.Tensor) -> torch.Tensor:
    """[2 I, K] weights with row 2j = gate row j and row 2j + 1 = up row j (offline weight preparation)."""
    if gate.shape != up.shape or gate.dim() != 2:
        raise ValueError("gate and up must be [I, K] each")
    return torch.stack([gate, up], dim=1).reshape(2 * gate.shape[0], gate.shape[1])


def qkv_head_group_rows(wq: torch.Tensor, wk: torch.Tensor, wv: torch.Tensor, head_dim: int) -> torch.Tensor:
    """Fused q/k/v weights in head groups (r query heads, one key head, one value head per group), the row
    order W4_EPI_QKV_SPLIT reads (offline weight preparation)."""
    groups = wk.shape[0] // head_dim
    if wk.shape != wv.shape or wk.shape[0] % head_dim or wq.shape[0] % (groups * head_dim):
        raise ValueError("q, k, v rows must be whole heads, with as many key as value heads")
    r = wq.shape[0] // (groups * head_dim)
    K = wq.shape[1]
    q = wq.reshape(groups, r * head_dim, K)
    k = wk.reshape(groups, head_dim, K)
    v = wv.reshape(groups, head_dim, K)
    return torch.cat([q, k, v], dim=1).reshape(-1, K)
