"""Pins of the oracle's scale-learning forward and STE backward: central
finite differences (float64) of the straight-through surrogate, the tied/dual
identity, and the link between fake quantisation and the quantiser's dequant."""
import numpy as np
import pytest


def _f(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _setup(seed, R=4, C=64, scale_jitter=0.3):
    rng = np.random.default_rng(seed)
    import oracle as O
    x = O.f32_to_bf16((rng.standard_normal((R, C)) * 0.02).astype(np.float32))
    g = O.f32_to_bf16((rng.standard_normal((R, C)) * 1e-3).astype(np.float32))
    amax = np.abs(_f(x)).reshape(R, C // 16, 16).max(axis=2)
    s = (amax / np.float32(6.0)).astype(np.float32)
    sp = (s * np.exp(rng.uniform(-scale_jitter, scale_jitter, s.shape))).astype(np.float32)
    so = (s * np.exp(rng.uniform(-scale_jitter, scale_jitter, s.shape))).astype(np.float32)
    return x, g, sp, so


def _surrogate(x, g, sp0, sp, so, q0, in0):
    """Straight-through surrogate of sum_i g_i * x~_i for one block: with the
    rounding offset c_i = q0_i - x_i/sp0 frozen, x~_i = so * (x_i/sp + c_i) for
    in-range elements and so * q0_i for clamped ones."""
    c = q0 - x / sp0
    xt = np.where(in0, so * (x / sp + c), so * q0)
    return float(np.sum(g * xt))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dual_scale_gradients_match_finite_differences(orc, seed):
    x, g, sp, so = _setup(seed)
    out = orc.scale_grad_bwd(x, g, sp, so)
    xf, gf = _f(x).astype(np.float64), _f(g).astype(np.float64)
    R, C = x.shape
    for r in range(R):
        for b in range(C // 16):
            xs, gs = xf[r, 16 * b:16 * b + 16], gf[r, 16 * b:16 * b + 16]
            p, o = float(sp[r, b]), float(so[r, b])
            q0 = orc.e2m1_value(orc.e2m1_rne((xs / p).astype(np.float32))).astype(np.float64)
            in0 = np.abs(xs / p) <= 6
            h = p * 1e-6
            fd_pre = (_surrogate(xs, gs, p, p + h, o, q0, in0)
                      - _surrogate(xs, gs, p, p - h, o, q0, in0)) / (2 * h)
            fd_post = (_surrogate(xs, gs, p, p, o + h, q0, in0)
                       - _surrogate(xs, gs, p, p, o - h, q0, in0)) / (2 * h)
            tol = 1e-4 * np.sum(np.abs(gs * q0)) + 1e-12
            assert abs(out["gs_post"][r, b] - fd_post) <= tol
            tolp = 1e-4 * np.sum(np.abs(gs * xs)) * o / p ** 2 + 1e-12
            assert abs(out["gs_pre"][r, b] - fd_pre) <= tolp


@pytest.mark.parametrize("seed", [3, 4])
def test_tied_scale_gradient_matches_finite_differences(orc, seed):
    x, g, sp, _ = _setup(seed, scale_jitter=0.6)  # jitter pushes some |x/s| past 6
    out = orc.scale_grad_bwd(x, g, sp, None)
    xf, gf = _f(x).astype(np.float64), _f(g).astype(np.float64)
    R, C = x.shape
    clamped = 0
    for r in range(R):
        for b in range(C // 16):
            xs, gs = xf[r, 16 * b:16 * b + 16], gf[r, 16 * b:16 * b + 16]
            s = float(sp[r, b])
            q0 = orc.e2m1_value(orc.e2m1_rne((xs / s).astype(np.float32))).astype(np.float64)
            in0 = np.abs(xs / s) <= 6
            clamped += int(np.sum(~in0))
            h = s * 1e-6
            fd = (_surrogate(xs, gs, s, s + h, s + h, q0, in0)
                  - _surrogate(xs, gs, s, s - h, s - h, q0, in0)) / (2 * h)
            tol = 1e-4 * np.sum(np.abs(gs) * 6) + 1e-12
            assert abs(out["gs_pre"][r, b] - fd) <= tol
    assert clamped > 0


def test_input_gradient_is_clamp_masked_ratio(orc):
    """dL/dx = g * d x~/d x = g * s_post / s_pre inside the clamp range, 0 outside
    (finite difference of the surrogate in x)."""
    x, g, sp, so = _setup(5, scale_jitter=0.6)
    out = orc.scale_grad_bwd(x, g, sp, so)
    xf, gf = _f(x).astype(np.float64), _f(g).astype(np.float64)
    R, C = x.shape
    for r in range(R):
        for i in range(C):
            p, o = float(sp[r, i // 16]), float(so[r, i // 16])
            inside = abs(xf[r, i] / p) <= 6
            h = abs(xf[r, i]) * 1e-6 + 1e-12
            q0 = float(orc.e2m1_value(orc.e2m1_rne(np.float32(xf[r, i] / p))))
            c = q0 - xf[r, i] / p
            f = (lambda xx: o * (xx / p + c)) if inside else (lambda xx: o * q0)
            dx = (f(xf[r, i] + h) - f(xf[r, i] - h)) / (2 * h)
            want = gf[r, i] * dx
            got = float(_f(out["gx"][r, i]))
            assert abs(got - want) <= 2 ** -7 * abs(want) + 1e-30


def test_tied_equals_sum_of_dual_partials_at_equal_scales(orc):
    x, g, sp, _ = _setup(6)
    tied = orc.scale_grad_bwd(x, g, sp, None)["gs_pre"]
    dual = orc.scale_grad_bwd(x, g, sp, sp.copy())
    both = dual["gs_pre"].astype(np.float64) + dual["gs_post"].astype(np.float64)
    scale = np.abs(dual["gs_pre"]).astype(np.float64) + np.abs(dual["gs_post"]) + 1e-30
    assert np.all(np.abs(tied - both) <= 1e-5 * scale)


def test_fakequant_matches_quantiser_dequant(orc):
    """With s_pre = s_post = the quantiser's decoded block scale, the fake
    quantisation is the quantiser's dequantised output."""
    rng = np.random.default_rng(12)
    x = orc.f32_to_bf16(rng.standard_normal((8, 128)).astype(np.float32))
    gam, _ = orc.global_amax(x)
    q = orc.quantize(x, gam)
    g = gam[0] / np.float32(6.0 * 448.0)
    d = (orc.scale_value(0, q["row_scales"][0]) * g).astype(np.float32)
    ok = d > 0
    xq, st = orc.fakequant_fwd(x, np.where(ok, d, 1.0).astype(np.float32))
    assert st == 0
    mask = np.repeat(ok, 16, axis=1)
    assert np.array_equal(xq[mask], q["row_dq"][0][mask])
    assert np.array_equal(orc.fakequant_fwd(x, d.clip(1e-30), d.clip(1e-30))[0][mask], xq[mask])


def test_bad_scales_are_flagged(orc):
    x, g, sp, so = _setup(7)
    for bad in (0.0, -1.0, np.nan, np.inf, 1e-40):
        s = sp.copy()
        s[1, 2] = bad
        assert orc.fakequant_fwd(x, s)[1] & orc.ST_BAD_SCALE
        assert orc.scale_grad_bwd(x, g, s, so)["status"] & orc.ST_BAD_SCALE
    assert orc.scale_grad_bwd(x, g, sp, so)["status"] == 0


def test_clamp_bounds_belong_to_the_middle_case(orc):
    """Scale Learning blog, "How Scale Learning Works": the STE's middle case
    holds for q_min <= x/s <= q_max, bounds included. At x/s = +-6 the tied
    term round(x/s) - x/s is 0 and the dual s_pre term is -s_post x / s_pre^2;
    beyond the bound the term is q_max (tied) or 0 (s_pre), and dL/dx is
    masked by the same interval. The expected values are the case formulas
    evaluated by hand."""
    s = np.float32(0.25)
    x = np.zeros((1, 16), np.float32)
    x[0, :3] = [6 * s, -6 * s, 7 * s]  # on both bounds, and beyond the upper one
    g = np.zeros((1, 16), np.float32)
    g[0, :3] = [1.0, 2.0, 4.0]
    xb, gb = orc.f32_to_bf16(x), orc.f32_to_bf16(g)
    tied = orc.scale_grad_bwd(xb, gb, np.array([[s]], np.float32), None)
    assert tied["status"] == 0
    assert tied["gs_pre"][0, 0] == 4.0 * 6.0  # bounds contribute 0, the clamped value q_max
    assert list(_f(tied["gx"][0, :3])) == [1.0, 2.0, 0.0]
    so = np.array([[0.5]], np.float32)  # s_post / s_pre = 2
    dual = orc.scale_grad_bwd(xb, gb, np.array([[s]], np.float32), so)
    # dL/ds_pre = -(s_post/s_pre) * sum g * x/s_pre over the middle case
    assert dual["gs_pre"][0, 0] == -2.0 * (1.0 * 6.0 + 2.0 * -6.0)
    assert dual["gs_post"][0, 0] == 1.0 * 6.0 + 2.0 * -6.0 + 4.0 * 6.0
    assert list(_f(dual["gx"][0, :3])) == [2.0, 4.0, 0.0]
