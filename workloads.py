"""Seeded synthetic inputs and the layer shapes they are drawn for.

This module holds no arithmetic of the quantized linear layer itself: it only
draws random numbers and names shapes. Both the CPU oracle (through the tests
and the bench's CPU baseline) and the CUDA path take their inputs from here.

Value distributions follow the workloads that the pages' benchmarks use as
real models (Llama-2-7B / 70B linears, lmdeploy PR #202 "Blazing fast W4A16
inference", throughput table; Marlin post, batch sizes 1..128):

* source weights W: float32 ~ N(0, 0.02^2), cast to fp16 (round to nearest);
* activations x: fp16 ~ N(0, 1);
* prefill-like activations: 1 % of the K channels (chosen by a seeded
  permutation) multiplied by 20 before the fp16 cast (outlier channels).

Seeds: weights use seed 0, activations seed 1, outlier channels seed 2
(numpy PCG64 streams, identical on x86-64 and aarch64).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

SEED_W = 0
SEED_X = 1
SEED_OUTLIER = 2


def weights_f16(n: int, k: int, seed: int = SEED_W, std: float = 0.02) -> np.ndarray:
    """fp16 source weight matrix W [n, k] (row-major, PyTorch nn.Linear order)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n, k), dtype=np.float32)
    w *= np.float32(std)
    return w.astype(np.float16)


def activations_f16(m: int, k: int, seed: int = SEED_X, outliers: bool = False) -> np.ndarray:
    """fp16 activations x [m, k]; with ``outliers`` 1 % of channels are scaled by 20."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float32)
    if outliers:
        n_out = int(math.ceil(0.01 * k))
        cols = np.random.default_rng(SEED_OUTLIER).permutation(k)[:n_out]
        x[:, cols] *= np.float32(20.0)
    return x.astype(np.float16)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 values -> uint16 bits of the nearest bfloat16 (ties to even; inputs finite). Input
    generation only: bf16 weights and activations are drawn as float32 and then cast."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def weights_bf16(n: int, k: int, seed: int = SEED_W, std: float = 0.02) -> np.ndarray:
    """bf16 source weights W [n, k] as uint16 bits (the same normal draw as weights_f16)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n, k), dtype=np.float32)
    w *= np.float32(std)
    return f32_to_bf16_bits(w)


def activations_bf16(m: int, k: int, seed: int = SEED_X, outliers: bool = False) -> np.ndarray:
    """bf16 activations x [m, k] as uint16 bits; with ``outliers`` 1 % of channels are scaled by 20."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k), dtype=np.float32)
    if outliers:
        n_out = int(math.ceil(0.01 * k))
        cols = np.random.default_rng(SEED_OUTLIER).permutation(k)[:n_out]
        x[:, cols] *= np.float32(20.0)
    return f32_to_bf16_bits(x)


@dataclass(frozen=True)
class Layer:
    """One linear layer shape: y[M, N] = x[M, K] . W[N, K]^T, group size g."""

    name: str
    n: int
    k: int
    g: int = 128


# Tiny parity case: M=4, N=256, K=512, g=128.
TINY = Layer("tiny", 256, 512, 128)
TINY_M = 4

# Llama-2-7B-shaped decode linears, g=128.
DECODE_LAYERS = (
    Layer("qkv_fused_12288x4096", 12288, 4096),
    Layer("o_proj_4096x4096", 4096, 4096),
    Layer("gate_up_fused_22016x4096", 22016, 4096),
    Layer("down_proj_4096x11008", 4096, 11008),
)
DECODE_MS = (1, 4, 8, 16, 32, 64, 128)

# Non-multiple group sizes: the last group is 32 wide in both.
PARTIAL_LAYERS = (
    Layer("stories_288x288_g256", 288, 288, 256),
    Layer("k4000_4096x4000_g128", 4096, 4000, 128),
)
PARTIAL_MS = (1, 8, 64)

# Llama-2-70B-shaped prefill linears, g=128, outlier activations.
PREFILL_LAYERS = (
    Layer("qkv_fused_10240x8192", 10240, 8192),
    Layer("o_proj_8192x8192", 8192, 8192),
    Layer("gate_up_fused_57344x8192", 57344, 8192),
    Layer("down_proj_8192x28672", 8192, 28672),
)
PREFILL_MS = (256, 512, 1024, 4096)

# One decoder layer of a 32-layer Llama-2-7B, unfused linears, plus lm_head.
STACK_LAYER = (
    Layer("q_proj", 4096, 4096),
    Layer("k_proj", 4096, 4096),
    Layer("v_proj", 4096, 4096),
    Layer("o_proj", 4096, 4096),
    Layer("gate_proj", 11008, 4096),
    Layer("up_proj", 11008, 4096),
    Layer("down_proj", 4096, 11008),
)
STACK_LAYERS = 32
STACK_HEAD = Layer("lm_head", 32000, 4096)
STACK_MS = (1, 16, 128)
