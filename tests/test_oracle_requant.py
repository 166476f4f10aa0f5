"""Pins of the oracle's re-quantisation (End-to-End 4-Bit Training,
"Re-quantization with stochastic rounding"): the MX shared exponent against
the textbook floor(log2) rule, E4M3 rounding against PyTorch's float8 cast and
table (library), exact stochastic-rounding probabilities, and the pages' claim
that re-quantised tensors equal the forward ones in expectation (their 4.5 ->
2 / 3 example included)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden

W = golden("worked_examples.json")


def _e4m3_table() -> np.ndarray:
    return torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_mx_shared_exponent_is_the_smallest_that_does_not_saturate(orc):
    """e is the smallest integer with amax <= 448 * 2^e (checked exactly in
    float64 on both sides of the boundary)."""
    rng = np.random.default_rng(3)
    vals = np.concatenate([rng.uniform(0, 1, 2000) * 10.0 ** rng.integers(-30, 30, 2000),
                           448.0 * 2.0 ** np.arange(-100, 100),
                           np.nextafter(448.0 * 2.0 ** np.arange(-100, 100), np.inf),
                           2.0 ** np.arange(-120, 120)])
    for a in vals.astype(np.float32):
        if not (a > 0) or not np.isfinite(a):
            continue
        e = orc.mx_shared_exp(float(a))
        if -127 < e < 127:
            assert float(a) <= 448.0 * 2.0 ** e and float(a) > 448.0 * 2.0 ** (e - 1), a
    assert orc.mx_shared_exp(0.0) == -127 and orc.mx_shared_exp(1e-44) == -127
    assert orc.mx_shared_exp(448.0) == 0 and orc.mx_shared_exp(449.0) == 1


def test_e4m3_rne_matches_torch_cast(orc):
    rng = np.random.default_rng(4)
    table = _e4m3_table()
    mids = (table[:-1] + table[1:]) / 2
    y = np.concatenate([rng.uniform(-460, 460, 3000), mids, -mids, table]).astype(np.float32)
    y = y[np.abs(y) < 464]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_rne(y), ref)
    assert list(orc.e4m3_rne(np.array([500.0, -1e9], np.float32))) == [0x7E, 0xFE]


def test_e4m3_sr_probability_is_exact(orc):
    table = _e4m3_table()
    rng = np.random.default_rng(5)
    v = np.arange(0, 65536, 97, dtype=np.uint32)  # 676 evenly spread draws
    for y in np.concatenate([rng.uniform(0, 447, 12), [0.00390625 * 1.3, 300.0, 447.9]]).astype(np.float32):
        a = Fraction(float(y))
        lo = max(t for t in table if Fraction(t) <= a)
        hi = min(t for t in table if Fraction(t) > a)
        p = (a - Fraction(lo)) / (Fraction(hi) - Fraction(lo))
        got = orc.e4m3_signed_value(orc.e4m3_sr(np.full(v.size, y, np.float32), v)).astype(np.float64)
        assert set(np.unique(got)) <= {lo, hi}
        up = got == hi
        for vi, u in zip(v, up):
            assert u == (Fraction(int(vi), 65536) < p)
    assert orc.e4m3_sr(np.float32(-500.0), 0)[0] == 0xFE


def _forward_encode(orc, x: np.ndarray, fos=0):
    xb = orc.f32_to_bf16(x.astype(np.float32))
    gam, _ = orc.global_amax(xb, xb.shape[0])
    q = orc.quantize(xb, gam, four_over_six=fos)
    return q, gam


def test_dequant_matches_forward_dequant(orc):
    rng = np.random.default_rng(6)
    x = (rng.standard_t(3, (2, 48, 64)) * 0.3).astype(np.float32)
    q, gam = _forward_encode(orc, x, fos=1)
    xh, st = orc.dequant(q["row_codes"], q["row_scales"], gam, four_over_six=1)
    assert st == 0
    # the forward dequant is the bf16 rounding of the same fp32 values
    assert np.array_equal(orc.f32_to_bf16(xh), q["row_dq"])


def test_requant_example_from_the_pages(orc):
    """A value 5.4 quantised in a block with scale 9 becomes 4.5; re-quantised
    in a block with scale 2 it is 2 (p 0.75) or 3 (p 0.25) times the scale."""
    ex, sr = W["requant_example"], W["sr_example"]
    x = np.zeros((1, 16, 16), np.float32)
    x[0, 0, 0], x[0, 0, 1] = 54.0, ex["x"]   # forward row block: scale 9
    x[0, 1, 1] = 12.0                        # column 1 block amax 12 -> scale 2
    x[0, 2, 0] = 2688.0                      # global amax 2688 -> g = 1
    q, gam = _forward_encode(orc, x)
    xh, _ = orc.dequant(q["row_codes"], q["row_scales"], gam)
    assert xh[0, 0, 1] == ex["value"] and xh[0, 1, 1] == 12.0
    ups = []
    for seed in range(3000):
        r = orc.requant(q["row_codes"], q["row_scales"], gam, target=1, rounding=1, seed=seed)
        assert orc.scale_value(0, r["scales"][0, 1, 0]) == sr["scale"]
        code = r["codes"][0, 1, 0] & 15  # element (row 0) of column 1, low nibble
        v = orc.e2m1_value(code) * sr["scale"]
        assert v in (sr["lo"] * sr["scale"], sr["hi"] * sr["scale"])
        ups.append(v == sr["hi"] * sr["scale"])
    assert abs(np.mean(ups) - sr["p_hi"]) < 4 * np.sqrt(0.25 * 0.75 / 3000)


@pytest.mark.parametrize("target", [0, 1])
def test_requant_preserves_forward_values_in_expectation(orc, target):
    """E[requant] = the forward values (the transposed de-quantised tensor)."""
    rng = np.random.default_rng(7 + target)
    x = (rng.standard_normal((1, 32, 32)) * 0.05).astype(np.float32)
    q, gam = _forward_encode(orc, x)
    xh, _ = orc.dequant(q["row_codes"], q["row_scales"], gam)
    want = xh[0].T.astype(np.float64)
    acc = np.zeros_like(want)
    n = 600
    for seed in range(n):
        r = orc.requant(q["row_codes"], q["row_scales"], gam, target=target, seed=seed)
        if target == 0:
            e = r["scales"][0].astype(np.int64) - 127
            vals = orc.e4m3_signed_value(r["codes"][0]).astype(np.float64)
            vals *= np.ldexp(1.0, np.repeat(e, 32, axis=1))
        else:
            c = r["codes"][0]
            codes = np.stack([c & 15, c >> 4], axis=-1).reshape(32, 32)
            g = gam[0] / np.float32(2688.0)
            d = (orc.scale_value(0, r["scales"][0]) * np.float32(g)).astype(np.float64)
            vals = orc.e2m1_value(codes).astype(np.float64) * np.repeat(d, 16, axis=1)
        acc += vals
    mean = acc / n
    # per element every draw is one of the two grid neighbours of the value, a
    # grid step apart, so the mean of n draws has std <= step / (2 sqrt(n))
    if target == 0:
        table = _e4m3_table()
        e = orc.requant(q["row_codes"], q["row_scales"], gam, target=0, seed=0)["scales"][0]
        X = np.ldexp(1.0, np.repeat(e.astype(np.int64) - 127, 32, axis=1))
        y = np.abs(want) / X
        hi = table[np.minimum(np.searchsorted(table, y, side="right"), table.size - 1)]
        lo = table[np.maximum(np.searchsorted(table, y, side="right") - 1, 0)]
        step = (hi - lo) * X
    else:
        r = orc.requant(q["row_codes"], q["row_scales"], gam, target=1, seed=0)
        g = gam[0] / np.float32(2688.0)
        d = np.repeat((orc.scale_value(0, r["scales"][0]) * np.float32(g)).astype(np.float64),
                      16, axis=1)
        y = np.abs(want) / np.where(d > 0, d, 1)
        step = np.where(y < 2, 0.5, np.where(y < 4, 1.0, 2.0)) * d
    assert np.all(np.abs(mean - want) <= 6 * step / (2 * np.sqrt(n)) + 1e-12)


def test_mx_block_maximum_lands_in_the_top_octave_without_clipping(orc):
    rng = np.random.default_rng(8)
    v = (rng.standard_normal(32 * 200) * np.exp(rng.uniform(-8, 8, 32 * 200))).astype(np.float32)
    codes, scales = orc.mx_encode(v, rounding=0)
    vals = np.abs(orc.e4m3_signed_value(codes)).reshape(-1, 32).max(axis=1)
    assert np.all((vals >= 224) & (vals <= 448))


def test_e4m3_sr_counts_are_exact_at_dyadic_probabilities(orc):
    """Over all 2^16 random values a value a quarter, a half or three quarters
    of the way between two E4M3 neighbours rounds up for exactly p * 2^16 of
    them (u = v / 2^16 < p), in the subnormal range, across binades and at the
    top of the grid."""
    table = _e4m3_table()
    v = np.arange(65536, dtype=np.uint32)
    for i in (1, 8, 40, 100, 125):
        lo, hi = table[i], table[i + 1]
        for k in (1, 2, 3):
            y = np.float32(lo + (hi - lo) * k / 4)
            assert float(y) == lo + (hi - lo) * k / 4
            got = orc.e4m3_signed_value(orc.e4m3_sr(np.full(65536, y, np.float32), v))
            assert int(np.sum(got == hi)) == k * 16384
            assert int(np.sum(got == lo)) == 65536 - k * 16384


@pytest.mark.parametrize("fmt,scale_max", [(1, 0.0), (0, 300.0), (1, 1000.0)])
def test_requant_reads_the_source_encoding_it_is_told(orc, fmt, scale_max):
    """A UE5M3 or explicit-M forward encoding is de-quantised with that format
    and M (its bf16 rounding is the forward's own dequant output), and the
    re-quantisation starts from exactly those values."""
    rng = np.random.default_rng(11)
    xb = orc.f32_to_bf16((rng.standard_t(3, (1, 32, 64)) * 0.3).astype(np.float32))
    gam, _ = orc.global_amax(xb)
    q = orc.quantize(xb, gam, scale_fmt=fmt, scale_max=scale_max)
    xh, st = orc.dequant(q["row_codes"], q["row_scales"], gam, scale_fmt=fmt,
                         scale_max=scale_max)
    assert st == 0 and np.array_equal(orc.f32_to_bf16(xh), q["row_dq"])
    r = orc.requant(q["row_codes"], q["row_scales"], gam, target=0, rounding=0,
                    src_fmt=fmt, src_scale_max=scale_max)
    xt = np.ascontiguousarray(xh[0].T)
    for c in range(64):
        codes, scales = orc.mx_encode(xt[c], rounding=0)
        assert np.array_equal(r["codes"][0, c], codes) and np.array_equal(r["scales"][0, c], scales)
