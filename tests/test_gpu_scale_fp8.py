"""CUDA FP8-scale side of scale learning against the oracle: the MSE scale
sweep over every E4M3 scale (codes and scales bit-exact), the fake-quant
forward and STE backward at FP8-rounded scales, export of learned scales, bad
scales and a bad global amax, and the sweep at the full weight size on
sampled rows (blocks are independent given the tensor's global amax)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_close_bf16, assert_close_f32, assert_exact, dev_bits, host_u16, host_u8
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _case(R, Cc, seed, jitter=0.3):
    wb, gb, s = synth.scale_learning(R, Cc, seed=seed)
    gam, _ = oracle.global_amax(wb)
    gam = (gam * np.float32(1.5)).astype(np.float32)  # rounded scales below the E4M3 maximum
    rng = np.random.default_rng(seed)
    sp = (s * np.exp(rng.uniform(-jitter, jitter, s.shape))).astype(np.float32)
    so = (s * np.exp(rng.uniform(-jitter, jitter, s.shape))).astype(np.float32)
    return wb, gb, sp, so, gam


def _d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


SHAPES = [(1, 16), (3, 48), (37, 272), (128, 4096), (1000, 160)]


@pytest.mark.parametrize("shape", SHAPES)
def test_mse_scale_sweep(shape):
    wb, _, _, _, _ = _case(*shape, seed=shape[0] + 1)
    gam, _ = oracle.global_amax(wb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_scale_init_mse(dev_bits(wb), _d(gam), status=st)
    want = oracle.scale_init_mse(wb, gam[0])
    assert int(st.item()) == want["status"] == 0
    assert_exact(host_u8(got["codes"]), want["codes"], "scale codes")
    assert_exact(got["s"].cpu().numpy().view(np.uint32), want["s"].view(np.uint32), "scales")


def test_mse_scale_sweep_outliers_zeros_and_tiny_amax():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-6, 6, (64, 1)))).astype(np.float32)
    x[5, :16] = 0.0
    x[9, 7] = 3.0e4
    wb = oracle.f32_to_bf16(x)
    for gam in (oracle.global_amax(wb)[0], np.array([0.0], np.float32),
                np.array([1e-30], np.float32)):
        got = nv.nvfp4_scale_init_mse(dev_bits(wb), _d(gam))
        want = oracle.scale_init_mse(wb, gam[0])
        assert_exact(host_u8(got["codes"]), want["codes"], f"codes (gamax {gam[0]})")
        assert_exact(got["s"].cpu().numpy().view(np.uint32), want["s"].view(np.uint32), "scales")


def _sweep_stress_blocks(rng, n):
    """n blocks of 16 of many kinds: Gaussian over 12 decades, one large
    outlier (the best scale may saturate it), a single spike, constant,
    sparse, two-level, bf16 subnormal, and values near the top of bf16."""
    kinds = []
    for k in range(n):
        t = k % 9
        if t == 0:
            b = rng.standard_normal(16) * np.exp(rng.uniform(-14, 14))
        elif t == 1:
            b = rng.standard_normal(16) * 0.1
            b[rng.integers(16)] = rng.uniform(2, 60) * rng.choice([-1, 1])
        elif t == 2:
            b = np.zeros(16)
            b[rng.integers(16)] = np.exp(rng.uniform(-20, 20))
        elif t == 3:
            b = np.full(16, np.exp(rng.uniform(-10, 10)))
        elif t == 4:
            b = rng.standard_normal(16) * (rng.uniform(size=16) < 0.2)
        elif t == 5:
            b = np.where(rng.uniform(size=16) < 0.5, 1.0, rng.uniform(0.001, 0.3, 16))
            b *= np.exp(rng.uniform(-5, 5)) * rng.choice([-1, 1], 16)
        elif t == 6:
            b = rng.standard_normal(16) * 1e-39
        elif t == 7:
            b = rng.uniform(-1, 1, 16) * 3.0e38
        else:
            b = rng.standard_normal(16) * np.exp(rng.uniform(-3, 3, 16))
        kinds.append(b)
    return np.concatenate(kinds).astype(np.float32).reshape(-1, 256)


def test_mse_scale_sweep_stress_against_the_full_oracle_sweep():
    """The kernel evaluates only the candidates that can win; the oracle
    evaluates all 126. Codes and scales must agree on every kind of block,
    under slice amaxes from far below to far above the blocks' own."""
    rng = np.random.default_rng(77)
    wb = oracle.f32_to_bf16(_sweep_stress_blocks(rng, 9 * 400))
    # 1e-6 .. 1e12 give 25 to 126 distinct winning codes; the tensor's own
    # amax (set by the blocks near the top of bf16), 1e-30 and 3e38 make every
    # candidate of most blocks tie (code 1 wins)
    own = oracle.global_amax(wb)[0]
    for g in (1e-6, 1e-3, 1.0, 1e3, 1e6, 1e12, own[0], 1e-30, 3.0e38):
        gam = np.array([g], np.float32)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = nv.nvfp4_scale_init_mse(dev_bits(wb), _d(gam), status=st)
        want = oracle.scale_init_mse(wb, gam[0])
        assert int(st.item()) == want["status"]
        assert_exact(host_u8(got["codes"]), want["codes"], f"codes (gamax {gam[0]})")
        assert_exact(got["s"].cpu().numpy().view(np.uint32), want["s"].view(np.uint32),
                     f"scales (gamax {gam[0]})")


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dual", [False, True])
def test_fp8_scale_fakequant_forward(shape, dual):
    wb, _, sp, so, gam = _case(*shape, seed=shape[1])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_fakequant_fwd_fp8scale(dev_bits(wb), _d(sp), _d(so) if dual else None, _d(gam),
                                          status=st)
    want, wst = oracle.fakequant_fwd_fp8(wb, sp, so if dual else None, gam[0])
    assert int(st.item()) == wst == 0
    assert_close_bf16(host_u16(got), want, "x~")


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dual", [False, True])
@pytest.mark.parametrize("want_gx", [False, True])
def test_fp8_scale_ste_backward(shape, dual, want_gx):
    wb, gb, sp, so, gam = _case(*shape, seed=shape[0] + shape[1])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_scale_grad_bwd_fp8scale(dev_bits(wb), dev_bits(gb), _d(sp),
                                           _d(so) if dual else None, _d(gam), want_gx=want_gx,
                                           status=st)
    want = oracle.scale_grad_bwd_fp8(wb, gb, sp, so if dual else None, gam[0], want_gx=want_gx)
    assert int(st.item()) == want["status"] == 0
    assert_close_f32(got["gs_pre"].cpu().numpy(), want["gs_pre"], "dL/ds_pre")
    if dual:
        assert_close_f32(got["gs_post"].cpu().numpy(), want["gs_post"], "dL/ds_post")
    if want_gx:
        assert_close_bf16(host_u16(got["gx"]), want["gx"], "dL/dx")


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dual", [False, True])
def test_export_scales(shape, dual):
    wb, _, sp, so, gam = _case(*shape, seed=shape[0] * 3 + 1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_export_scales(dev_bits(wb), _d(sp), _d(so) if dual else None, _d(gam),
                                 status=st)
    want = oracle.export_scales(wb, sp, so if dual else None, gam[0])
    assert int(st.item()) == want["status"] == 0
    assert_exact(host_u8(got["codes"]).reshape(want["codes"].shape), want["codes"], "codes")
    assert_exact(host_u8(got["scales"]).reshape(want["scales"].shape), want["scales"], "scales")


def test_fp8_scale_status_bits():
    wb, gb, sp, so, gam = _case(8, 64, seed=9)
    so = so.copy()
    so[1, 2] = -so[1, 2]
    sp2 = sp.copy()
    sp2[3, 0] = 1e-30  # rounds to the zero code
    for s_pre, s_post in ((sp, so), (sp2, None)):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        nv.nvfp4_fakequant_fwd_fp8scale(dev_bits(wb), _d(s_pre), None if s_post is None else _d(s_post),
                                        _d(gam), status=st)
        _, wst = oracle.fakequant_fwd_fp8(wb, s_pre, s_post, gam[0])
        assert int(st.item()) & nv.DEV_BAD_SCALE and wst & oracle.ST_BAD_SCALE
        st.zero_()
        nv.nvfp4_export_scales(dev_bits(wb), _d(s_pre), None if s_post is None else _d(s_post),
                               _d(gam), status=st)
        assert int(st.item()) & nv.DEV_BAD_SCALE
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = np.array([np.nan], np.float32)
    nv.nvfp4_scale_init_mse(dev_bits(wb), _d(bad), status=st)
    assert int(st.item()) & nv.DEV_BAD_AMAX and oracle.scale_init_mse(wb, bad[0])["status"] & oracle.ST_BAD_AMAX


def test_full_size_weight_sweep_on_sampled_rows():
    """The sweep on the 14336x4096 scale-learning weight, rows sampled."""
    wb, _, _ = synth.scale_learning(14336, 4096, seed=2)
    gam, _ = oracle.global_amax(wb)
    got = nv.nvfp4_scale_init_mse(dev_bits(wb), _d(gam))
    codes, s = host_u8(got["codes"]), got["s"].cpu().numpy()
    rows = np.random.default_rng(4).choice(14336, 24, replace=False)
    rows[:2] = (0, 14335)
    want = oracle.scale_init_mse(wb[rows], gam[0])
    assert_exact(codes[rows], want["codes"], "codes (sampled rows)")
    assert_exact(s[rows].view(np.uint32), want["s"].view(np.uint32), "scales (sampled rows)")
