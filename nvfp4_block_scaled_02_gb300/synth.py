"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws numbers: it holds none of the quantiser's arithmetic and
is shared by the tests, the oracle runs and ``bench.py`` so that both sides of a
parity check see the same bytes. Values are drawn in float32 with
``numpy.random.Generator(PCG64(seed))`` and rounded to bfloat16 by PyTorch's
round-to-nearest-even cast. Tensors are returned as ``uint16`` arrays holding the
bf16 bit patterns (row-major, C-contiguous).

Workloads (the defaults are the full sizes; every function takes smaller shapes
for tests that the oracle must finish in seconds):

* ``outlier_normal``    N(0,1) with a fraction of entries multiplied by a factor
                        (1024x1024, 0.1 % x20, seed 0).
* ``student_t``         0.5 * Student-t(nu=3) activations (8192 tokens x 4096).
* ``scale_learning``    weight N(0, 0.02), upstream gradient N(0, 1e-3), and the
                        per-block scales initialised to block amax / 6
                        (14336x4096, seed 2).
* ``drifting_gradient`` N(0,1) times per-row lognormal(0, 2) magnitudes, grown
                        by 1.05 per step (16384x4096, seed 3).
* ``moe_experts``       64 experts x 2048x7168 N(0, 0.02) with 0.01 % x50
                        outliers (seed 4).
"""
from __future__ import annotations

import numpy as np
import torch


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (RNE, PyTorch cast) and return the bits."""
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _outliers(rng: np.random.Generator, x: np.ndarray, frac: float, factor: float) -> None:
    n = x.size
    k = int(round(n * frac))
    if k:
        idx = rng.choice(n, size=k, replace=False)
        flat = x.reshape(-1)
        flat[idx] *= np.float32(factor)


def outlier_normal(rows: int = 1024, cols: int = 1024, seed: int = 0,
                   frac: float = 1e-3, factor: float = 20.0) -> np.ndarray:
    rng = _rng(seed)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    _outliers(rng, x, frac, factor)
    return to_bf16_bits(x)


def student_t(rows: int = 8192, cols: int = 4096, seed: int = 1, nu: float = 3.0,
              scale: float = 0.5) -> np.ndarray:
    rng = _rng(seed)
    x = (rng.standard_t(nu, size=(rows, cols)) * scale).astype(np.float32)
    return to_bf16_bits(x)


def scale_learning(rows: int = 14336, cols: int = 4096, seed: int = 2,
                   w_std: float = 0.02, g_std: float = 1e-3):
    """Returns (w_bits, g_bits, s_init) with s_init = block amax / 6 in float32,
    the initialisation of trainable per-block scales (amax parameterisation)."""
    rng = _rng(seed)
    w = (rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(w_std))
    g = (rng.standard_normal((rows, cols), dtype=np.float32) * np.float32(g_std))
    wb = to_bf16_bits(w)
    gb = to_bf16_bits(g)
    amax = np.abs(bf16_bits_to_f32(wb)).reshape(rows, cols // 16, 16).max(axis=2)
    s = (amax / np.float32(6.0)).astype(np.float32)
    s[s == 0] = np.float32(1.0)
    return wb, gb, s


class DriftingGradient:
    """Gradient stream for periodic tensor scaling: x_t = bf16(base * 1.05**t)."""

    def __init__(self, rows: int = 16384, cols: int = 4096, seed: int = 3,
                 sigma: float = 2.0, drift: float = 1.05):
        rng = _rng(seed)
        base = rng.standard_normal((rows, cols), dtype=np.float32)
        mag = np.exp(rng.standard_normal((rows, 1)) * sigma).astype(np.float32)
        self.base = base * mag
        self.drift = drift

    def step(self, t: int) -> np.ndarray:
        return to_bf16_bits(self.base * np.float32(self.drift ** t))


def moe_experts(experts: int = 64, rows: int = 2048, cols: int = 7168, seed: int = 4,
                std: float = 0.02, frac: float = 1e-4, factor: float = 50.0) -> np.ndarray:
    rng = _rng(seed)
    x = rng.standard_normal((experts, rows, cols), dtype=np.float32) * np.float32(std)
    _outliers(rng, x, frac, factor)
    return to_bf16_bits(x)


def uniform_bits(shape, seed: int, lo: float = -8.0, hi: float = 8.0) -> np.ndarray:
    """Plain uniform values, for edge-case tests."""
    rng = _rng(seed)
    return to_bf16_bits(rng.uniform(lo, hi, size=shape).astype(np.float32))
