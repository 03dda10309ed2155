"""Seeded synthetic inputs shared by the oracle tests, the CUDA tests and the bench.

This module only draws numbers.  It holds none of the codec's or the matrix
products' arithmetic: no exponent split, no rank table, no coding, no
summation.  Both sides of every parity check receive the same arrays from here.

Workload shapes follow the pages' models (Binade project README and the
Hugging Face cards for the 3B, 12B and 26B-A4B packed models): random-init
BF16 weights N(0, 0.02), optional 0.1% outliers at 100x, activations N(0, 1).

Seeds: ``numpy.random.SeedSequence([cfg, layer, proj, expert])`` with PCG64;
activations use ``[cfg, 999, step]``; routing uses ``[cfg, 777, layer, step]``.
"""
from __future__ import annotations

import numpy as np

SIGMA = 0.02
OUTLIER_FRAC = 0.001
OUTLIER_SCALE = 100.0


def rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 samples to bf16 bit patterns (nearest, ties to even).

    Used only to turn drawn float samples into bf16 inputs; NaN never occurs
    in drawn samples.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def weights(rows: int, cols: int, key, outliers: bool = False,
            sigma: float = SIGMA) -> np.ndarray:
    """bf16 bit patterns [rows, cols] of N(0, sigma), optionally with outliers.

    Outliers: exactly round(0.001 * n) positions, drawn uniformly without
    replacement, multiplied by 100 in float32 before rounding to bf16.
    """
    g = rng(*key)
    n = rows * cols
    w = g.standard_normal(n, dtype=np.float32)
    w *= np.float32(sigma)
    if outliers and n > 0:
        m = int(round(OUTLIER_FRAC * n))
        if m:
            pos = g.choice(n, size=m, replace=False)
            w[pos] *= np.float32(OUTLIER_SCALE)
    return f32_to_bf16_bits(w).reshape(rows, cols)


def activations(k: int, key, count: int = 1) -> np.ndarray:
    """bf16 bit patterns [count, k] (or [k] when count == 1) of N(0, 1)."""
    g = rng(*key)
    x = g.standard_normal(count * k, dtype=np.float32)
    b = f32_to_bf16_bits(x)
    return b if count == 1 else b.reshape(count, k)


def routing(tokens: int, n_experts: int, topk: int, key):
    """Top-k routing: distinct expert ids per token (uniform without
    replacement) and weights p = softmax of topk N(0, 1) logits (computed in
    double with the C library's exp through numpy, then rounded to float32)."""
    g = rng(*key)
    ids = np.empty((tokens, topk), dtype=np.int32)
    p = np.empty((tokens, topk), dtype=np.float32)
    for t in range(tokens):
        ids[t] = g.choice(n_experts, size=topk, replace=False)
        z = g.standard_normal(topk)
        e = np.exp(z - z.max())
        p[t] = (e / e.sum()).astype(np.float32)
    return ids, p


# Named workloads (shapes of the pages' models; random init).
CFG_SMALL = dict(name="tensor-1024x1024", rows=1024, cols=1024, outliers=True)
CFG_BULK = dict(name="bulk-4096x16384", rows=4096, cols=16384, outliers=True)

DENSE_3B = dict(name="dense-3B", layers=28, hidden=3072, proj=[
    ("q", 3072, 3072), ("k", 1024, 3072), ("v", 1024, 3072), ("o", 3072, 3072),
    ("gate", 8192, 3072), ("up", 8192, 3072), ("down", 3072, 8192)])

DENSE_12B = dict(name="dense-12B", layers=48, hidden=3840, proj=[
    ("q", 4096, 3840), ("k", 2048, 3840), ("v", 2048, 3840), ("o", 3840, 4096),
    ("gate", 15360, 3840), ("up", 15360, 3840), ("down", 3840, 15360)])

MOE = dict(name="moe-30L-128E", layers=30, hidden=2816, experts=128, topk=8,
           expert_proj=[("gate", 704, 2816), ("up", 704, 2816), ("down", 2816, 704)],
           attn_proj=[("q", 2816, 2816), ("k", 1024, 2816), ("v", 1024, 2816),
                      ("o", 2816, 2816)])

GEMM_ROWS = (16, 128, 2048)


# Special-value inputs (the exactness claim covers every bf16 pattern, not
# only the model-like draws above).
def bf16_patterns(count: int, key, finite_only: bool = False) -> np.ndarray:
    """`count` bf16 bit patterns: every pattern of the set (all 65,536, or the
    finite ones) once in a seeded random order, repeated in fresh orders
    until `count` are drawn."""
    g = rng(*key)
    allp = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if finite_only:
        allp = allp[np.isfinite(bf16_bits_to_f32(allp))]
    reps = -(-count // allp.size)
    return np.concatenate([g.permutation(allp) for _ in range(reps)])[:count]


def tiny_weights(rows: int, cols: int, key, log2_scale: int = -128) -> np.ndarray:
    """bf16 bit patterns of N(0, 1) * 2^log2_scale: at the default scale most
    are bf16 subnormals (below 2^-126) and the rest the smallest normals."""
    g = rng(*key)
    w = np.ldexp(g.standard_normal(rows * cols, dtype=np.float32), log2_scale).astype(np.float32)
    return f32_to_bf16_bits(w).reshape(rows, cols)


def scaled_activations(k: int, key, log2_scale: int, count: int = 1) -> np.ndarray:
    """bf16 bit patterns [count, k] (or [k]) of N(0, 1) * 2^log2_scale."""
    g = rng(*key)
    x = np.ldexp(g.standard_normal(count * k, dtype=np.float32), log2_scale).astype(np.float32)
    b = f32_to_bf16_bits(x)
    return b if count == 1 else b.reshape(count, k)
