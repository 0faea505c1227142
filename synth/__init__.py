"""Seeded synthetic inputs for the W4A16 hot path.

This module serves both the CUDA path's tests/benchmark and the CPU oracle.
It holds no arithmetic of the method: it only draws random numbers and lays
them out in the storage format (8 four-bit codes per 32-bit word, lowest
nibble = lowest k; binary16 scales, and biases unless the codes are
symmetric, per group along K: 64 unless stated).

Distributions follow the workloads the pages describe with model shapes:
codes q uniform on 0..15, scale ~ U(0.002, 0.02), bias = -8*scale +
N(0, 1e-3), activations ~ N(0, 1), all rounded to binary16.
"""
from __future__ import annotations

import numpy as np

GROUP = 64

# Projection shapes (name, K in, N out) per transformer layer.
QWEN25_05B_Q = [("q", 896, 896)]
QWEN3_06B = [("q", 1024, 2048), ("k", 1024, 1024), ("v", 1024, 1024), ("o", 2048, 1024),
             ("gate", 1024, 3072), ("up", 1024, 3072), ("down", 3072, 1024)]
QWEN3_06B_LAYERS = 28
QWEN3_06B_LM_HEAD = (1024, 151936)
QWEN25_3B = [("q", 2048, 2048), ("k", 2048, 256), ("v", 2048, 256), ("o", 2048, 2048),
             ("gate", 2048, 11008), ("up", 2048, 11008), ("down", 11008, 2048)]
QWEN25_3B_LAYERS = 36
QWEN25_3B_LM_HEAD = (2048, 151936)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """uint8 codes [N][K] (values 0..15) -> uint32 words [N][K/8], code k%8 in bits 4*(k%8)."""
    q = np.asarray(q, dtype=np.uint32)
    N, K = q.shape
    assert K % 8 == 0
    q = q.reshape(N, K // 8, 8)
    words = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        words |= (q[:, :, i] & 0xF) << np.uint32(4 * i)
    return words


def make_scales_biases(g: np.random.Generator, N: int, K: int, group: int = GROUP):
    s = g.uniform(0.002, 0.02, size=(N, K // group))
    s16 = s.astype(np.float16)
    b = -8.0 * s16.astype(np.float64) + g.normal(0.0, 1e-3, size=(N, K // group))
    return s16, b.astype(np.float16)


def make_linear(seed: int, N: int, K: int, group: int = GROUP):
    """Random int4 affine weight: (qweight uint32 [N][K/8], scales f16, biases f16 [N][K/group]).

    Uniform random 32-bit words are 8 independent uniform 4-bit codes."""
    g = rng(seed)
    qweight = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s16, b16 = make_scales_biases(g, N, K, group)
    return qweight, s16, b16


def make_linear_sym(seed: int, N: int, K: int, group: int = 128):
    """Random int4 symmetric weight (codes read as q - 8, no biases):
    (qweight uint32 [N][K/8], scales f16 [N][K/group], None).  Scales are
    drawn like the affine ones, ~ U(0.002, 0.02)."""
    g = rng(seed)
    qweight = g.integers(0, 2**32, size=(N, K // 8), dtype=np.uint32)
    s16 = g.uniform(0.002, 0.02, size=(N, K // group)).astype(np.float16)
    return qweight, s16, None


def make_x(seed: int, M: int, K: int) -> np.ndarray:
    """Activations fp16 [M][K] ~ N(0, 1); row m drawn from seed + m."""
    rows = [rng(seed + m).standard_normal(K) for m in range(M)]
    return np.stack(rows).astype(np.float16)


def layer_seed(base: int, layer: int, proj: int) -> int:
    return base + 7 * layer + proj


def make_half_matrix(seed: int, rows: int, cols: int, std: float = 1.0) -> np.ndarray:
    """fp16 [rows][cols] ~ N(0, std^2) (dense operands for the half GEMM)."""
    return (rng(seed).standard_normal((rows, cols)) * std).astype(np.float16)
