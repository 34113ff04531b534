"""Seeded synthetic inputs for the BitLinear forward.

This module only draws random numbers; it holds none of the method's
arithmetic. Both the CUDA path and the CPU oracle are fed from here, so the
two see the same bytes. Every generator is a pure function of its seed
(numpy PCG64 via ``np.random.default_rng``) and returns fp32 arrays on the
host (or bf16 bit patterns where the workload is bf16).

The shapes and distributions follow the 2B-class model of the "BitNet b1.58
2B4T Technical Report" (hidden 2560, FFN 6912; the k/v projection 2560->640)
and a 70B-class model (hidden 8192, FFN 28672). The pages print no tensors, so
all values are synthetic.
"""
from __future__ import annotations

import numpy as np

# (K, N) of the four BitLinear projections of one 2B-class layer
SHAPES_2B = {
    "qo": (2560, 2560),      # attention q / o projection
    "kv": (2560, 640),       # attention k / v projection
    "up": (2560, 6912),      # FFN up
    "down": (6912, 2560),    # FFN down
}
# (K, N) of the 70B-class projections
SHAPES_70B = {
    "attn": (8192, 8192),
    "up": (8192, 28672),
    "down": (28672, 8192),
}
DECODE_LAYERS = 30


def gaussian_weights(N: int, K: int, sigma: float, seed: int,
                     outlier_frac: float = 0.0, outlier_scale: float = 10.0) -> np.ndarray:
    """W [N, K] ~ N(0, sigma^2); round(outlier_frac * N * K) entries, chosen
    uniformly without replacement, are multiplied by outlier_scale."""
    rng = np.random.default_rng(seed)
    W = rng.standard_normal((N, K), dtype=np.float32)
    W *= np.float32(sigma)
    n_out = int(round(outlier_frac * N * K))
    if n_out:
        idx = rng.choice(N * K, size=n_out, replace=False)
        W.reshape(-1)[idx] *= np.float32(outlier_scale)
    return W


def student_t(M: int, K: int, seed: int, df: float = 4.0) -> np.ndarray:
    """X [M, K] ~ Student-t(df), fp32."""
    rng = np.random.default_rng(seed)
    return rng.standard_t(df, size=(M, K)).astype(np.float32)


def tiny_case(seed: int = 0):
    """W [256, 256] ~ N(0, 0.02^2); X [4, 256]: rows 0-1 ~ N(0, 1), row 2 all
    zero, row 3 ~ N(0, 1) with one entry (index drawn from the seed) set to a
    50x outlier (+-50)."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((256, 256), dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    X = rng.standard_normal((4, 256), dtype=np.float32)
    X[2, :] = 0.0
    j = int(rng.integers(0, 256))
    X[3, j] = np.float32(50.0) * (np.float32(1.0) if X[3, j] >= 0 else np.float32(-1.0))
    return W, X


def decode_weights(shape: str, layer: int) -> np.ndarray:
    """2B-class decode weights: N(0, 0.02^2) with 0.1% entries x10; seed 1000 + layer
    (+ a per-shape offset so the four projections differ)."""
    K, N = SHAPES_2B[shape]
    off = {"qo": 0, "kv": 100, "up": 200, "down": 300}[shape]
    return gaussian_weights(N, K, 0.02, 1000 + off + layer, outlier_frac=0.001)


def decode_activations(shape: str, layer: int, M: int = 1) -> np.ndarray:
    """X [M, K] ~ Student-t(4); seed 5000 + per-shape offset + layer."""
    K, _ = SHAPES_2B[shape]
    off = {"qo": 0, "kv": 100, "up": 200, "down": 300}[shape]
    return student_t(M, K, 5000 + off + layer)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (ties to even) and return the uint16 bit patterns.
    Input conditioning for the bf16 workloads, not part of the method."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
    return r.astype(np.uint16)


def batched_activations_bf16(M: int, K: int, seed: int) -> np.ndarray:
    """Batched-decode activations as bf16 bit patterns [M, K]: Student-t(4)
    times a per-row multiplier 10^U(-1.5, 1.5), rounded to bf16."""
    rng = np.random.default_rng(seed)
    x = rng.standard_t(4.0, size=(M, K)).astype(np.float32)
    mult = (10.0 ** rng.uniform(-1.5, 1.5, size=(M, 1))).astype(np.float32)
    return f32_to_bf16_bits(x * mult)


def prefill_activations(M: int, K: int, seed: int, heavy_frac: float = 0.01,
                        heavy_scale: float = 20.0) -> np.ndarray:
    """Prefill activations [M, K] ~ N(0, 1); a fixed 1% of the channels (chosen
    from the seed) are multiplied by 20 for every token."""
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K), dtype=np.float32)
    n_heavy = max(1, int(round(heavy_frac * K)))
    ch = rng.choice(K, size=n_heavy, replace=False)
    X[:, ch] *= np.float32(heavy_scale)
    return X


def large_weights(shape: str) -> np.ndarray:
    """70B-class weights: N(0, 0.01^2) with 0.1% entries x10."""
    K, N = SHAPES_70B[shape]
    off = {"attn": 0, "up": 1, "down": 2}[shape]
    return gaussian_weights(N, K, 0.01, 7000 + off, outlier_frac=0.001)


def norm_gain(K: int, seed: int, edge: bool = True) -> np.ndarray:
    """RMSNorm gain [K] ~ U(0.05, 2.5), fp32 (norm gains are mostly positive
    and of order one). With ``edge``, 1% of the entries are negated and 0.5%
    set to zero, so that signs and dropped columns are exercised."""
    rng = np.random.default_rng(seed)
    g = rng.uniform(0.05, 2.5, K).astype(np.float32)
    if edge:
        neg = rng.choice(K, size=max(1, K // 100), replace=False)
        g[neg] = -g[neg]
        g[rng.choice(K, size=max(1, K // 200), replace=False)] = 0.0
    return g
