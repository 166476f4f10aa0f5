"""Pins of the oracle's FP8-scale side of scale learning (Scale Learning blog,
"How Scale Learning Works": the block scale is itself quantised to FP8 with a
straight-through estimator; "Using Scale Learning": MSE scale setting with an
FP8 sweep, export of the learned post-scale): a float64 brute force of the
sweep, exactly representable blocks, scale invariance, FP8 rounding of the
scales through PyTorch's float8 cast (library), and the export's
de-quantisation against the fake-quant forward."""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_02_gb300 import synth

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e4m3_values() -> np.ndarray:
    return torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _g(gamax: float) -> np.float32:
    g = np.float32(gamax) / np.float32(6.0 * 448.0) if gamax > 0 else np.float32(1.0)
    return np.float32(g)


def _fq_sse64(x: np.ndarray, s: float) -> float:
    """Fake-quantisation SSE of one block in float64: textbook nearest E2M1
    value (ties to the even code), saturating at 6."""
    y = np.abs(x) / s
    idx = np.searchsorted(E2M1, y)  # first grid value >= y
    lo = np.clip(idx - 1, 0, 7)
    hi = np.clip(idx, 0, 7)
    dlo, dhi = y - E2M1[lo], E2M1[hi] - y
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(y >= 6.0, 7, pick)
    q = np.sign(x) * E2M1[pick]
    return float(np.sum((x - s * q) ** 2))


def test_mse_sweep_against_float64_brute_force(orc):
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((8, 64)) * np.exp(rng.uniform(-3, 3, (8, 1)))).astype(np.float32)
    x[2, 5] *= 40  # an outlier block
    xb = orc.f32_to_bf16(x)
    gam, _ = orc.global_amax(xb)
    r = orc.scale_init_mse(xb, gam[0])
    assert r["status"] == 0
    g = float(_g(gam[0]))
    vals = _e4m3_values()
    xf = synth.bf16_bits_to_f32(xb).astype(np.float64)
    for rb in range(8):
        for j in range(4):
            blk = xf[rb, 16 * j:16 * j + 16]
            sses = np.array([_fq_sse64(blk, vals[c] * g) for c in range(1, 127)])
            chosen = _fq_sse64(blk, vals[r["codes"][rb, j]] * g)
            assert chosen <= sses.min() * (1 + 1e-5) + 1e-30, (rb, j)
            assert r["s"][rb, j] == np.float32(vals[r["codes"][rb, j]]) * np.float32(g)


def test_mse_sweep_finds_exactly_representable_blocks(orc):
    """x = s* q with q on the E2M1 grid (±6 included) has zero error at s*."""
    rng = np.random.default_rng(12)
    vals = _e4m3_values()
    gam = np.float32(2688.0)  # g = 1
    xs = []
    for c in (40, 56, 72, 90, 110):
        q = E2M1[rng.integers(0, 8, 16)] * rng.choice([-1.0, 1.0], 16)
        q[3] = 6.0
        xs.append(q * vals[c])
    x = np.stack(xs).astype(np.float32)
    xb = orc.f32_to_bf16(x)
    assert np.array_equal(synth.bf16_bits_to_f32(xb), x)  # exact in bf16
    r = orc.scale_init_mse(xb, gam)
    assert np.all(r["sse"] == 0.0)
    # the chosen scale reproduces the block exactly
    for i in range(5):
        s = r["s"][i, 0]
        xq, st = orc.fakequant_fwd(xb[i:i + 1], np.array([[s]], np.float32))
        assert st == 0 and np.array_equal(xq, xb[i:i + 1])


def test_mse_sweep_zero_block_and_scale_invariance(orc):
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((4, 32)) * 0.01).astype(np.float32)
    x[1, :16] = 0.0
    xb = orc.f32_to_bf16(x)
    gam, _ = orc.global_amax(xb)
    r = orc.scale_init_mse(xb, gam[0])
    assert r["codes"][1, 0] == 1 and r["sse"][1, 0] == 0.0
    # doubling x (exact in bf16) and its amax doubles g: same codes
    x2 = orc.f32_to_bf16(synth.bf16_bits_to_f32(xb) * 2)
    r2 = orc.scale_init_mse(x2, gam[0] * 2)
    assert np.array_equal(r["codes"], r2["codes"])


def test_mse_sweep_never_worse_than_the_amax_scale(orc):
    wb, _, _ = synth.scale_learning(32, 256, seed=14)
    gam, _ = orc.global_amax(wb)
    r = orc.scale_init_mse(wb, gam[0])
    q = orc.quantize(wb, gam, scale_max=448.0)  # amax-derived E4M3 scales, same g
    g = _g(gam[0])
    vals = _e4m3_values()
    xf = synth.bf16_bits_to_f32(wb).astype(np.float64)
    worse = 0
    for rb in range(32):
        for j in range(16):
            blk = xf[rb, 16 * j:16 * j + 16]
            a = _fq_sse64(blk, vals[q["row_scales"][0, rb, j]] * float(g))
            worse += _fq_sse64(blk, vals[r["codes"][rb, j]] * float(g)) > a * (1 + 1e-5)
    assert worse == 0


def _q8_torch(s: np.ndarray, gamax: float) -> np.ndarray:
    """FP8 rounding of scales through PyTorch's float8_e4m3fn cast (RNE)."""
    g = _g(gamax)
    rg = np.float32(np.float32(1.0) / g)
    t = (s.astype(np.float32) * rg).astype(np.float32)
    assert np.all(t < 448)
    c = torch.from_numpy(t).to(torch.float8_e4m3fn).to(torch.float32).numpy()
    return (c * g).astype(np.float32)


@pytest.mark.parametrize("tied", [False, True])
def test_fp8_scale_ste_is_the_plain_ste_at_the_rounded_scales(orc, tied):
    wb, gb, s = synth.scale_learning(16, 64, seed=15)
    gam, _ = orc.global_amax(wb)
    gam = gam * np.float32(2.0)  # keeps the rounded scales below the E4M3 maximum
    rng = np.random.default_rng(15)
    sp = (s * rng.uniform(0.8, 1.25, s.shape)).astype(np.float32)
    so = None if tied else (s * rng.uniform(0.8, 1.25, s.shape)).astype(np.float32)
    spq, soq = _q8_torch(sp, gam[0]), None if tied else _q8_torch(so, gam[0])
    xq8, st8 = orc.fakequant_fwd_fp8(wb, sp, so, gam[0])
    xq, st = orc.fakequant_fwd(wb, spq, soq)
    assert st8 == st == 0 and np.array_equal(xq8, xq)
    b8 = orc.scale_grad_bwd_fp8(wb, gb, sp, so, gam[0])
    b = orc.scale_grad_bwd(wb, gb, spq, soq)
    for k in ("gx", "gs_pre", "gs_post"):
        if b[k] is not None:
            assert np.array_equal(b8[k], b[k]), k
    # scales already on the FP8 grid: identical to the plain path
    xq_on, _ = orc.fakequant_fwd_fp8(wb, spq, soq, gam[0])
    assert np.array_equal(xq_on, xq)


def test_fp8_scale_bad_scales_are_flagged(orc):
    wb, gb, s = synth.scale_learning(4, 32, seed=16)
    gam, _ = orc.global_amax(wb)
    so = s.copy()
    so[0, 0] = -s[0, 0]
    assert orc.fakequant_fwd_fp8(wb, s, so, gam[0])[1] & orc.ST_BAD_SCALE
    sp = s.copy()
    sp[1, 1] = 1e-30  # rounds to the zero code
    assert orc.fakequant_fwd_fp8(wb, sp, None, gam[0])[1] & orc.ST_BAD_SCALE


@pytest.mark.parametrize("tied", [False, True])
def test_export_dequantises_to_the_fake_quant_forward(orc, tied):
    wb, _, s = synth.scale_learning(32, 128, seed=17)
    gam, _ = orc.global_amax(wb)
    gam = gam * np.float32(2.0)
    rng = np.random.default_rng(17)
    sp = (s * rng.uniform(0.7, 1.4, s.shape)).astype(np.float32)
    so = None if tied else (s * rng.uniform(0.7, 1.4, s.shape)).astype(np.float32)
    ex = orc.export_scales(wb, sp, so, gam[0])
    assert ex["status"] == 0
    xh, st = orc.dequant(ex["codes"][None], ex["scales"][None], gam, scale_max=448.0)
    assert st == 0
    xq, st = orc.fakequant_fwd_fp8(wb, sp, so, gam[0])
    assert st == 0
    assert np.array_equal(orc.f32_to_bf16(xh[0]), xq)
    # the scale bytes are the float8 codes of the post-scales
    t = ((sp if tied else so) * np.float32(np.float32(1.0) / _g(gam[0]))).astype(np.float32)
    want = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ex["scales"], want)


def test_export_flags_a_pre_scale_that_rounds_to_the_zero_code(orc):
    """A pre-scale that is a normal fp32 number but rounds to the FP8 zero
    code gives no usable forward scale: the export reports it like the
    fake-quant forward does."""
    wb, _, s = synth.scale_learning(4, 32, seed=18)
    gam, _ = orc.global_amax(wb)
    assert orc.export_scales(wb, s, None, gam[0])["status"] == 0
    sp = s.copy()
    sp[2, 1] = 1e-30
    assert orc.export_scales(wb, sp, None, gam[0])["status"] & orc.ST_BAD_SCALE
    assert orc.fakequant_fwd_fp8(wb, sp, None, gam[0])[1] & orc.ST_BAD_SCALE
