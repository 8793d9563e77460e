"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the
CPU oracle.  Holds no FP8 arithmetic: it only draws numbers.

Recipe (the isolated-linear and MLP workloads): X ~ N(0, 1), W ~ N(0, 0.02),
dY ~ N(0, 1e-3) (second parameter = standard deviation), drawn in float32
with torch's seeded CPU generator, multiplied by the standard deviation in
float32, then rounded once to bf16.  Outliers: a seeded permutation (CPU
generator) picks floor(frac * numel) distinct entries, which are multiplied
by `factor` in float32 before the single bf16 rounding.  Every draw happens
on the host and the bytes are then copied to the requested device, so the
same seed gives the same tensor on any machine, with or without a GPU.
"""
from __future__ import annotations

import hashlib

import numpy as np
import torch

SEED_X, SEED_W, SEED_DY, SEED_OUTLIER = 42, 43, 44, 45


def bf16_normal(shape, std: float, seed: int, device="cpu",
                outlier_frac: float = 0.0, outlier_factor: float = 100.0) -> torch.Tensor:
    """bf16 tensor of N(0, std) samples, reproducible from `seed` (drawn on
    the host, then placed on `device`)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32)
    x.mul_(float(std))
    if outlier_frac > 0:
        n = x.numel()
        k = int(np.floor(outlier_frac * n))
        g2 = torch.Generator(device="cpu")
        g2.manual_seed(SEED_OUTLIER)
        idx = torch.randperm(n, generator=g2)[:k]
        flat = x.view(-1)
        flat[idx] = flat[idx] * float(outlier_factor)
    x = x.to(torch.bfloat16)
    return x if torch.device(device).type == "cpu" else x.to(device)


def sha256(t: torch.Tensor) -> str:
    """SHA-256 of a tensor's bytes (row-major, host copy), for recording
    exactly which inputs a measurement used."""
    a = t.detach().contiguous().cpu()
    if a.dtype == torch.bfloat16:
        a = a.view(torch.int16)
    return hashlib.sha256(memoryview(a.numpy()).cast("B")).hexdigest()


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(b: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    arr = np.ascontiguousarray(b, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(arr.copy()).view(torch.bfloat16).to(device)


def linear_inputs(N: int, K: int, O: int, device="cpu", layer: int = 0,
                  outlier_frac: float = 0.0):
    """(X [N,K], W [O,K], dY [N,O]) bf16 for one linear."""
    x = bf16_normal((N, K), 1.0, SEED_X + 100 * layer, device, outlier_frac=outlier_frac)
    w = bf16_normal((O, K), 0.02, SEED_W + layer, device)
    dy = bf16_normal((N, O), 1e-3, SEED_DY + 100 * layer, device)
    return x, w, dy
