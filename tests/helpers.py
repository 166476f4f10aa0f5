"""Shared helpers of the GPU parity tests: moving bf16 bit arrays between numpy
and the device, running the CUDA path through the binding, and comparing its
outputs with the oracle's."""
from __future__ import annotations

import numpy as np
import torch

# Floating-point outputs must match within this relative error (dequantised
# values and per-block scale gradients); codes, scale bytes, 4/6 bits and
# random draws must match exactly.
FLOAT_RTOL = 1e-6


def dev_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> device tensor (int16 storage of the bits)."""
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).to(device)


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_exact(got: np.ndarray, want: np.ndarray, what: str) -> None:
    got = np.asarray(got).reshape(-1)
    want = np.asarray(want).reshape(-1)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:5]}: " \
                          f"got {got[bad[:5]]} want {want[bad[:5]]}"


def assert_close_f32(got: np.ndarray, want: np.ndarray, what: str, rtol: float = FLOAT_RTOL):
    g = np.asarray(got, np.float64).reshape(-1)
    w = np.asarray(want, np.float64).reshape(-1)
    assert g.shape == w.shape
    err = np.abs(g - w)
    ok = (err <= rtol * np.abs(w)) | (g == w)
    bad = np.nonzero(~ok)[0]
    assert bad.size == 0, f"{what}: {bad.size} beyond rtol {rtol}, first {bad[:5]}: " \
                          f"got {g[bad[:5]]} want {w[bad[:5]]}"


def assert_close_bf16(got_bits: np.ndarray, want_bits: np.ndarray, what: str,
                      rtol: float = FLOAT_RTOL):
    """Dequantised bf16 values within rtol (one bf16 ulp is 2^-8 relative, so this
    means equal values; +0 and -0 count as equal)."""
    assert_close_f32(bf16_to_f64(got_bits), bf16_to_f64(want_bits), what, rtol)


def compare_encoding(gpu: dict, ref: dict, prefix: str, what: str, fos: bool,
                     dequant: bool = True) -> None:
    assert_exact(host_u8(gpu["codes"]), ref[prefix + "codes"], f"{what} codes")
    assert_exact(host_u8(gpu["scales"]), ref[prefix + "scales"], f"{what} scales")
    if fos:
        assert_exact(host_u32(gpu["choice"]), ref[prefix + "choice"], f"{what} 4/6 bits")
    if dequant:
        assert_close_bf16(host_u16(gpu["dequant"]), ref[prefix + "dq"], f"{what} dequant")
