"""Seeded synthetic inputs shared by the tests, the bench and the CPU baseline.

This module only draws numbers. It holds none of the quantization or GEMM
arithmetic: the kernels and the oracle each receive these arrays as inputs.

Shapes and distributions follow the workloads of the quantization pages:

* the fake-quant weight study of "量化部署实战" (anrans.github.io, section
  精度比较): linear weights ~ N(0, 0.02) with a few outlier channels;
* the Llama-3.1-8B MLP shape of "量化：让每一步搬更少的字节"
  (niuwancheng.cn, 路线一): K = 4096, N = 14336;
* the Qwen3-0.6B linear set (q/k/v/o/gate/up/down) and the K-cache structure
  "constant per-channel bias + small variation" of "量化部署实战"
  (section KV Cache 量化).

N(m, s) means mean m and standard deviation s. All generators use numpy's
PCG64 (`numpy.random.default_rng(seed)`).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "normal_f32", "with_outlier_channels", "to_bf16_bits", "bf16_bits_to_f32",
    "quant_roundtrip_input", "w4a16_decode_inputs", "fp8_block_gemm_inputs",
    "fp4_gemm_inputs", "qwen3_decode_linears", "kv_cache_inputs",
    "QWEN3_LINEARS",
]


def normal_f32(rng: np.random.Generator, shape, std: float, mean: float = 0.0) -> np.ndarray:
    """Draw float32 N(mean, std) of `shape`."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def with_outlier_channels(rng: np.random.Generator, x: np.ndarray, count: int, factor: float,
                          axis: int = -1) -> np.ndarray:
    """Scale `count` distinct seeded channels (indices along `axis`) by `factor`, in place."""
    n = x.shape[axis]
    idx = np.sort(rng.choice(n, size=count, replace=False))
    sl = [slice(None)] * x.ndim
    sl[axis] = idx
    x[tuple(sl)] *= np.float32(factor)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even) and return the uint16 bit patterns.

    This is data generation (the bf16 inputs of the workloads), not part of the
    quantizers. It relies on torch's own fp32 -> bf16 conversion.
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------- workloads

def quant_roundtrip_input(seed: int = 0, rows: int = 1024, cols: int = 1024,
                          n_outlier_cols: int = 8, factor: float = 50.0) -> np.ndarray:
    """fp32 [rows, cols] ~ N(0, 0.02) with `n_outlier_cols` seeded columns x`factor`."""
    rng = np.random.default_rng(seed)
    x = normal_f32(rng, (rows, cols), 0.02)
    return with_outlier_channels(rng, x, n_outlier_cols, factor, axis=1)


def w4a16_decode_inputs(M: int, seed: int = 0, K: int = 4096, N: int = 14336,
                        outlier_frac: float = 0.01, factor: float = 20.0):
    """Decode-GEMM inputs: A bf16 bits [M, K] ~ N(0, 1) with round(1% K) channels x20
    (the same channels in every row) and an fp32 weight W [K, N] ~ N(0, 0.02)."""
    rng = np.random.default_rng(seed)
    a = normal_f32(rng, (M, K), 1.0)
    with_outlier_channels(rng, a, int(round(outlier_frac * K)), factor, axis=1)
    w = normal_f32(rng, (K, N), 0.02)
    return to_bf16_bits(a), w


def fp8_block_gemm_inputs(seed: int = 0, M: int = 2048, K: int = 4096, N: int = 14336,
                          n_outlier: int | None = None, factor: float = 20.0):
    """FP8 block GEMM inputs: A bf16 bits [M, K] ~ N(0,1) with outlier channels, and
    B^T bf16 bits [N, K] where B [K, N] ~ N(0, 0.02) (B is transposed once, K-major)."""
    rng = np.random.default_rng(seed)
    a = normal_f32(rng, (M, K), 1.0)
    with_outlier_channels(rng, a, n_outlier if n_outlier is not None else int(round(0.01 * K)),
                          factor, axis=1)
    b = normal_f32(rng, (K, N), 0.02)
    return to_bf16_bits(a), to_bf16_bits(np.ascontiguousarray(b.T))


def fp4_gemm_inputs(seed: int = 0, M: int = 8192, K: int = 4096, N: int = 4096,
                    outlier_frac: float = 0.005, factor: float = 30.0):
    """NVFP4/MXFP4 GEMM inputs: A bf16 bits [M, K] ~ N(0,1) with 0.5% channels x30,
    B^T bf16 bits [N, K] with B [K, N] ~ N(0, 0.02)."""
    rng = np.random.default_rng(seed)
    a = normal_f32(rng, (M, K), 1.0)
    with_outlier_channels(rng, a, max(1, int(round(outlier_frac * K))), factor, axis=1)
    b = normal_f32(rng, (K, N), 0.02)
    return to_bf16_bits(a), to_bf16_bits(np.ascontiguousarray(b.T))


# Qwen3-0.6B linear set: (name, in_features K, out_features N).
QWEN3_LINEARS = (
    ("q_proj", 1024, 2048), ("k_proj", 1024, 1024), ("v_proj", 1024, 1024),
    ("o_proj", 2048, 1024), ("gate_proj", 1024, 3072), ("up_proj", 1024, 3072),
    ("down_proj", 3072, 1024),
)


def qwen3_decode_linears(layers: int = 28, tokens: int = 64, seed: int = 0):
    """Yield (layer, name, A bf16 bits [tokens, K], W fp32 [K, N]) for every linear of a
    random-init Qwen3-0.6B-shaped decoder. Each (layer, projection) has its own seed, and
    each linear gets an independent N(0, 1) input, so every GEMM checks on its own."""
    for layer in range(layers):
        for p, (name, K, N) in enumerate(QWEN3_LINEARS):
            rng = np.random.default_rng([seed, layer, p])
            w = normal_f32(rng, (K, N), 0.02)
            a = normal_f32(rng, (tokens, K), 1.0)
            yield layer, name, to_bf16_bits(a), w


def kv_cache_inputs(seed: int = 0, B: int = 1, H: int = 8, T: int = 4096, D: int = 128,
                    bias_std: float = 4.0):
    """KV-cache write inputs, bf16 bits [B, H, T, D]: K = N(0,1) + bias[h, d] with a
    per-channel constant bias ~ N(0, 4) (the same for every token), V = N(0, 1)."""
    rng = np.random.default_rng(seed)
    bias = normal_f32(rng, (H, D), bias_std)
    k = normal_f32(rng, (B, H, T, D), 1.0) + bias[None, :, None, :]
    v = normal_f32(rng, (B, H, T, D), 1.0)
    return to_bf16_bits(k), to_bf16_bits(v)
