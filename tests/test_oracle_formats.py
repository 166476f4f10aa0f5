"""Pins of the oracle's number formats against things other than itself:
the grid the pages print, PyTorch's float8 casts (library routines), the
textbook construction of round-to-nearest-even into a small float format
(numpy's half-to-even rounding on the scaled value), and Random123 /
cuRAND known answers for Philox4x32-10."""
import ctypes
import os

import numpy as np
import pytest
import torch

from conftest import golden


def _fp32_range(lo: float, hi: float, stride: int = 1) -> np.ndarray:
    a = np.array([lo], np.float32).view(np.uint32)[0]
    b = np.array([hi], np.float32).view(np.uint32)[0]
    return np.arange(a, b, stride, dtype=np.uint32).view(np.float32)


def _around(values, span: int = 48) -> np.ndarray:
    """All fp32 bit patterns within +-span ulps of each value."""
    bits = np.asarray(values, np.float32).view(np.uint32).astype(np.int64)
    off = np.arange(-span, span + 1, dtype=np.int64)
    allb = (bits[:, None] + off[None, :]).reshape(-1)
    allb = allb[(allb >= 0) & (allb < 0x7F800000)]
    return allb.astype(np.uint32).view(np.float32)


# ------------------------------------------------------------------ E2M1 --

def textbook_minifloat(a: np.ndarray, mbits: int, emin: int, vmax: float) -> np.ndarray:
    """RNE of non-negative a into a float format with mbits mantissa bits and
    minimum normal exponent emin (subnormals below), saturating at vmax:
    the quantum is 2^(max(e, emin) - mbits), and numpy rounds half to even."""
    a = np.asarray(a, np.float64)
    _, e2 = np.frexp(a)  # a = m * 2^e2, m in [0.5, 1)
    e = np.maximum(e2.astype(np.int64) - 1, emin)
    quantum = np.ldexp(1.0, (e - mbits).astype(np.int32))
    v = np.round(a / quantum) * quantum
    return np.minimum(v, vmax)


def test_e2m1_grid_is_the_printed_one(orc):
    g = golden("worked_examples.json")["e2m1_grid"]["magnitudes"]
    vals = orc.e2m1_value(np.arange(16))
    assert list(vals[:8]) == g
    assert list(-vals[8:]) == g
    assert np.all(np.signbit(vals[8:]))


def _e2m1_textbook_codes(y: np.ndarray) -> np.ndarray:
    grid = np.array(golden("worked_examples.json")["e2m1_grid"]["magnitudes"], np.float64)
    v = textbook_minifloat(np.abs(y), mbits=1, emin=0, vmax=6.0)
    code = np.searchsorted(grid, v)
    assert np.all(grid[code] == v)
    return (code | np.where(np.signbit(y), 8, 0)).astype(np.uint8)


def test_e2m1_rne_exhaustive_core_range(orc):
    """Every fp32 value in [2^-3, 8) and its negation, plus a stride below."""
    y = np.concatenate([_fp32_range(0.125, 8.0), _fp32_range(1e-45, 0.125, 4099),
                        _fp32_range(8.0, 3.0e38, 4099),
                        np.array([0.0, np.inf, 6.0, 5.0, 3.5, 2.5, 1.75, 1.25, 0.75, 0.25],
                                 np.float32)])
    y = np.concatenate([y, -y])
    assert np.array_equal(orc.e2m1_rne(y), _e2m1_textbook_codes(y))


def test_e2m1_ties_go_to_even_code(orc):
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    expect = [0, 2, 2, 4, 4, 6, 6]  # codes of 0, 1, 1, 2, 2, 4, 4
    assert list(orc.e2m1_rne(ties)) == expect
    assert list(orc.e2m1_rne(-ties)) == [c | 8 for c in expect]
    assert orc.e2m1_rne(np.float32(-0.0)) == 8 and orc.e2m1_rne(np.float32(-0.1)) == 8


# ------------------------------------------------------------------ E4M3 --

def _torch_e4m3_table() -> np.ndarray:
    codes = torch.arange(127, dtype=torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_matches_torch(orc):
    assert np.array_equal(orc.scale_value(0, np.arange(127)).astype(np.float64),
                          _torch_e4m3_table())


def test_e4m3_encode_matches_torch_cast_below_464(orc):
    table = _torch_e4m3_table()
    mids = (table[:-1] + table[1:]) / 2
    t = np.concatenate([_fp32_range(1e-45, 464.0, 97), _around(mids.astype(np.float32)),
                        table.astype(np.float32), np.zeros(1, np.float32)])
    t = t[t < 464.0]
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.scale_encode(0, t), ref)


def test_e4m3_saturates_at_448(orc):
    t = np.array([464.0, 470.0, 480.0, 1e6, 3.0e38, np.inf], np.float32)
    assert np.all(orc.scale_encode(0, t) == 0x7E)
    assert orc.scale_value(0, 0x7E) == 448.0


def test_e4m3_encode_matches_textbook(orc):
    t = np.concatenate([_fp32_range(1e-45, 600.0, 211),
                        _around(_torch_e4m3_table().astype(np.float32)[1:], 8)])
    v = textbook_minifloat(t, mbits=3, emin=-6, vmax=448.0)
    assert np.array_equal(orc.scale_value(0, orc.scale_encode(0, t)).astype(np.float64), v)


# ----------------------------------------------------------------- UE5M3 --

def test_ue5m3_even_codes_are_e5m2(orc):
    """UE5M3 adds one mantissa bit to E5M2 (same bias 15, same subnormals):
    code 2k decodes like E5M2 code k for every finite E5M2 code."""
    k = np.arange(0x7C)  # E5M2 exponent field < 31: finite
    e5 = torch.from_numpy(k.astype(np.uint8)).view(torch.float8_e5m2).to(torch.float64).numpy()
    assert np.array_equal(orc.scale_value(1, 2 * k).astype(np.float64), e5)


def test_ue5m3_odd_codes_are_midpoints(orc):
    v = orc.scale_value(1, np.arange(256)).astype(np.float64)
    assert np.all(np.diff(v) > 0)
    odd = np.arange(1, 255, 2)
    same_binade = (odd >> 3) == ((odd + 1) >> 3)
    o = odd[same_binade]
    assert np.array_equal(v[o], (v[o - 1] + v[o + 1]) / 2)
    assert v[255] == 1.875 * 2.0 ** 16 and v[1] == 2.0 ** -17


def test_ue5m3_encode_matches_textbook(orc):
    v = orc.scale_value(1, np.arange(256)).astype(np.float32)
    t = np.concatenate([_fp32_range(1e-45, 2.0e5, 1543), _around(v[1:], 8),
                        _around(((v[:-1].astype(np.float64) + v[1:]) / 2).astype(np.float32), 8)])
    ref = textbook_minifloat(t, mbits=3, emin=-14, vmax=122880.0)
    assert np.array_equal(orc.scale_value(1, orc.scale_encode(1, t)).astype(np.float64), ref)


# ------------------------------------------------------------------ bf16 --

def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 0x7F800000, size=200000, dtype=np.uint32)
    bits[:1000] = (bits[:1000] & 0xFFFF0000) | 0x8000  # exact ties
    f = bits.view(np.float32)
    f = np.concatenate([f, -f])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f32_to_bf16(f), ref)


# ---------------------------------------------------------------- Philox --

def test_philox_known_answers(orc):
    for v in golden("philox4x32_10_kat.json")["vectors"]:
        ctr = [int(h, 16) for h in v["ctr"]]
        key = [int(h, 16) for h in v["key"]]
        out = [int(h, 16) for h in v["out"]]
        assert list(orc.philox(ctr, key)) == out


def _curand():
    for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(d, "lib64", "libcurand.so")
        if d and os.path.exists(p):
            return ctypes.CDLL(p)
    return None


def test_philox_matches_curand_host_generator(orc):
    """cuRAND's host-side Philox4_32_10 generator emits, for seed s, block i =
    philox(counter (0, 0, i, 0), key (s mod 2^32, s / 2^32))."""
    cu = _curand()
    if cu is None:
        pytest.skip("libcurand not found")
    gen = ctypes.c_void_p()
    assert cu.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0
    try:
        seed = 0x0123456789ABCDEF
        assert cu.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        n = 4 * 256
        buf = (ctypes.c_uint * n)()
        assert cu.curandGenerate(gen, buf, ctypes.c_size_t(n)) == 0
        got = np.frombuffer(buf, np.uint32).reshape(-1, 4)
    finally:
        cu.curandDestroyGenerator(gen)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in range(got.shape[0]):
        assert list(orc.philox([0, 0, i, 0], key)) == list(got[i]), i
