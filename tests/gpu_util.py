"""Helpers shared by the GPU tests (marshalling and the tolerance check only)."""
from __future__ import annotations

import numpy as np

TOL_REL = 1e-3
TOL_ABS = 1e-6


def bf16_cuda(bits: np.ndarray, pad_to: int | None = None):
    """numpy bf16 bit patterns [M, K] -> CUDA bf16 tensor (optionally with lda = pad_to)."""
    import torch
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    M, K = a.shape
    if pad_to is not None and pad_to > K:
        b = np.full((M, pad_to), 0x7FC0, np.uint16)  # NaN padding must never be read
        b[:, :K] = a
        t = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
        return t[:, :K]
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()


def assert_within_tolerance(got, ref, S, what=""):
    """|gpu - oracle| <= 1e-3 * sum_k |a_k w_k| + 1e-6, element by element."""
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = TOL_REL * S + TOL_ABS
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape)
    assert (err <= bound).all(), (
        f"{what}: {int((err > bound).sum())} elements out of tolerance; worst at {worst}: "
        f"gpu {got[worst]!r} oracle {ref[worst]!r} bound {bound[worst]!r}")
    return float(ratio.max())


def f32_bits(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
