"""Seeded synthetic inputs for the verify matmul.

This module holds no arithmetic of the method itself (no quantization, no
dequantization, no rotation, no matmul): it only draws the raw fp32 weights and
bf16 activation rows that both the CUDA library and the CPU oracle consume.
The workloads it stands in for are real model weights and real drafted-token
activations, which are not available; the shapes follow a hidden-5120,
27B-class model as served on the pages ("r9k: a from-scratch inference engine
for Qwen3.8-27B on two Radeon AI PRO R9700", opening section).

Recipe (identical on host and device generators):
  * weights: fp32 N(0, 0.02) per element.
  * activations: fp32 N(0, 1); optionally ceil(0.001 K) distinct outlier
    channels k are drawn and column k of every row is scaled by 20 (so exactly
    0.1% of the entries of each row are outliers and the channels persist
    across rows, as outlier channels do in the Hadamard page); then every value
    is rounded to bf16 (round to nearest even).
  * seeds: a workload with base seed b draws weights from b, activations from
    b + 1000 and outlier channels from b + 2000 (numpy PCG64 on the host,
    torch's CUDA generator on the device).

Host generators return numpy arrays; device generators return torch tensors.
"""
from __future__ import annotations

import math

import numpy as np

WEIGHT_SIGMA = 0.02
OUTLIER_FRACTION = 0.001
OUTLIER_FACTOR = 20.0

# Workload shapes (M, N, K lists) used by the tests and the bench.
SHAPES = {
    # Q4_0 single shape, M=8 rows, K=512, N=256, seed 0
    "q4_small": dict(fmt="q4_0", N=256, K=512, Ms=(8,), seed=0, outliers=False),
    # Q4_0 attention-projection-like shape
    "q4_attn": dict(fmt="q4_0", N=5120, K=5120, Ms=(1, 8, 16), seed=1, outliers=True),
    # Q4_0 MLP-like shapes (gate+up fused, down), plus the Hadamard variant
    "q4_gateup": dict(fmt="q4_0", N=2 * 17408, K=5120, Ms=(16,), seed=2, outliers=True),
    "q4_down": dict(fmt="q4_0", N=5120, K=17408, Ms=(16,), seed=2, outliers=True),
    # FP8 E4M3 block-scaled shape
    "fp8_mlp": dict(fmt="fp8", N=17408, K=5120, Ms=(1, 8, 16), seed=3, outliers=True),
    # Q8_0 shapes (the FP8 MLP shape and the attention-projection shape)
    "q8_mlp": dict(fmt="q8_0", N=17408, K=5120, Ms=(1, 8, 16), seed=6, outliers=True),
    "q8_attn": dict(fmt="q8_0", N=5120, K=5120, Ms=(1, 8, 16), seed=7, outliers=True),
    # Q4_0 qkv-projection-like shape of the whole-model sweep (5120 -> 10240)
    "q4_qkv": dict(fmt="q4_0", N=10240, K=5120, Ms=(1, 8, 16), seed=8, outliers=True),
    # Q4_0 output head (vocabulary 151,936 x hidden 5120) for the greedy acceptance step
    "q4_lmhead": dict(fmt="q4_0", N=151936, K=5120, Ms=(1, 8, 16), seed=5, outliers=True),
}

# Whole-model sweep: per layer (N, K) of the four Q4_0 matrices.
MODEL_LAYER = (("qkv", 10240, 5120), ("out", 5120, 5120), ("gateup", 2 * 17408, 5120),
               ("down", 5120, 17408))
MODEL_LAYERS = 64
MODEL_MS = (1, 2, 4, 8, 16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def outlier_channels(K: int, seed: int) -> np.ndarray:
    n = math.ceil(OUTLIER_FRACTION * K)
    g = np.random.Generator(np.random.PCG64(seed))
    return np.sort(g.choice(K, size=n, replace=False)).astype(np.int64)


def weights(N: int, K: int, seed: int, sigma: float = WEIGHT_SIGMA) -> np.ndarray:
    """fp32 [N][K] ~ N(0, sigma^2)."""
    g = np.random.Generator(np.random.PCG64(seed))
    w = g.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(sigma)
    return w


def activations(M: int, K: int, seed: int, outliers: bool = False,
                outlier_seed: int | None = None) -> np.ndarray:
    """bf16 bit patterns [M][K]: N(0,1), optional x20 outlier channels, RNE to bf16."""
    g = np.random.Generator(np.random.PCG64(seed))
    a = g.standard_normal((M, K), dtype=np.float32)
    if outliers:
        ch = outlier_channels(K, seed + 1000 if outlier_seed is None else outlier_seed)
        a[:, ch] *= np.float32(OUTLIER_FACTOR)
    return f32_to_bf16_bits(a)


def workload(name: str, M: int | None = None):
    """Host inputs of a named shape: (fp32 weights [N][K], bf16 act [M][K], spec)."""
    spec = dict(SHAPES[name])
    M = spec["Ms"][-1] if M is None else M
    b = spec["seed"]
    w = weights(spec["N"], spec["K"], b)
    a = activations(M, spec["K"], b + 1000, outliers=spec["outliers"], outlier_seed=b + 2000)
    return w, a, spec


# ------------------------------------------------------------------ device
def weights_cuda(N: int, K: int, seed: int, sigma: float = WEIGHT_SIGMA, device="cuda"):
    """fp32 [N][K] ~ N(0, sigma^2) drawn on the GPU with torch's generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    w.mul_(sigma)
    return w


def activations_cuda(M: int, K: int, seed: int, outliers: bool = True, device="cuda"):
    """bf16 [M][K] tensor with the same recipe as ``activations`` (device RNG)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    a = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    if outliers:
        ch = torch.from_numpy(outlier_channels(K, seed + 1000)).to(device)
        a[:, ch] *= OUTLIER_FACTOR
    return a.to(torch.bfloat16)
