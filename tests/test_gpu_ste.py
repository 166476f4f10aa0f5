"""CUDA scale-learning kernels against the oracle: fake-quant forward and the
STE backward, tied and dual scales, with and without dL/dx, ragged sizes and
bad-scale detection."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_close_bf16, assert_close_f32, dev_bits, host_u16
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _case(R, Cc, seed, jitter=0.5):
    wb, gb, s = synth.scale_learning(R, Cc, seed=seed)
    rng = np.random.default_rng(seed)
    sp = (s * np.exp(rng.uniform(-jitter, jitter, s.shape))).astype(np.float32)
    so = (s * np.exp(rng.uniform(-jitter, jitter, s.shape))).astype(np.float32)
    return wb, gb, sp, so


@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (37, 272), (128, 4096), (1000, 160)])
@pytest.mark.parametrize("dual", [False, True])
def test_fakequant_forward(shape, dual):
    wb, _, sp, so = _case(*shape, seed=shape[0])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_fakequant_fwd(dev_bits(wb), torch.from_numpy(sp).cuda(),
                                 torch.from_numpy(so).cuda() if dual else None, status=st)
    want, wst = oracle.fakequant_fwd(wb, sp, so if dual else None)
    assert int(st.item()) == wst == 0
    assert_close_bf16(host_u16(got), want, "x~")


@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (37, 272), (128, 4096), (1000, 160)])
@pytest.mark.parametrize("dual", [False, True])
@pytest.mark.parametrize("want_gx", [False, True])
def test_ste_backward(shape, dual, want_gx):
    wb, gb, sp, so = _case(*shape, seed=shape[1])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_scale_grad_bwd(dev_bits(wb), dev_bits(gb), torch.from_numpy(sp).cuda(),
                                  torch.from_numpy(so).cuda() if dual else None,
                                  want_gx=want_gx, status=st)
    want = oracle.scale_grad_bwd(wb, gb, sp, so if dual else None, want_gx=want_gx)
    assert int(st.item()) == want["status"] == 0
    assert_close_f32(got["gs_pre"].cpu().numpy(), want["gs_pre"], "dL/ds_pre")
    if dual:
        assert_close_f32(got["gs_post"].cpu().numpy(), want["gs_post"], "dL/ds_post")
    if want_gx:
        assert_close_bf16(host_u16(got["gx"]), want["gx"], "dL/dx")


def test_clamped_elements_present():
    """With shrunken scales many |x/s| exceed 6: the clamp branch is exercised."""
    wb, gb, sp, so = _case(64, 256, seed=5, jitter=0.0)
    sp = (sp * np.float32(0.5)).astype(np.float32)
    xs = synth.bf16_bits_to_f32(wb).reshape(64, 16, 16) / sp[:, :, None]
    assert (np.abs(xs) > 6).mean() > 0.05
    for dual in (False, True):
        got = nv.nvfp4_scale_grad_bwd(dev_bits(wb), dev_bits(gb), torch.from_numpy(sp).cuda(),
                                      torch.from_numpy(so).cuda() if dual else None)
        want = oracle.scale_grad_bwd(wb, gb, sp, so if dual else None)
        assert_close_f32(got["gs_pre"].cpu().numpy(), want["gs_pre"], "dL/ds_pre")
        assert_close_bf16(host_u16(got["gx"]), want["gx"], "dL/dx")


@pytest.mark.parametrize("bad", [0.0, -1.0, np.nan, np.inf, 1e-40])
def test_bad_scale_flagged(bad):
    wb, gb, sp, so = _case(8, 64, seed=1)
    sp[3, 1] = bad
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nvfp4_fakequant_fwd(dev_bits(wb), torch.from_numpy(sp).cuda(), status=st)
    nv.nvfp4_scale_grad_bwd(dev_bits(wb), dev_bits(gb), torch.from_numpy(sp).cuda(),
                            torch.from_numpy(so).cuda(), status=st)
    assert int(st.item()) & nv.DEV_BAD_SCALE
    assert oracle.fakequant_fwd(wb, sp)[1] & oracle.ST_BAD_SCALE


def test_nonfinite_gradient_flagged():
    wb, gb, sp, so = _case(8, 64, seed=2)
    gb[2, 5] = 0x7F80
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nvfp4_scale_grad_bwd(dev_bits(wb), dev_bits(gb), torch.from_numpy(sp).cuda(), status=st)
    assert int(st.item()) & nv.DEV_NONFINITE_INPUT


def test_clamp_bounds_match_the_oracle():
    """Values exactly on the clamp bounds (x/s = +-6, s a power of two, so the
    quotient is exact) belong to the middle case of the STE; neighbours just
    inside and beyond them too."""
    rng = np.random.default_rng(21)
    R, Cc = 16, 256
    s = np.ldexp(1.0, rng.integers(-8, 2, (R, Cc // 16))).astype(np.float32)
    k = rng.choice(np.array([6.0, -6.0, 5.5, -5.5, 7.0, -7.0, 6.5, 0.25]), (R, Cc))
    x = (k * np.repeat(s, 16, axis=1)).astype(np.float32)
    wb = synth.to_bf16_bits(x)
    assert np.array_equal(synth.bf16_bits_to_f32(wb), x)
    gb = synth.to_bf16_bits(rng.standard_normal((R, Cc)).astype(np.float32))
    so = (s * np.float32(1.25)).astype(np.float32)
    for post in (None, so):
        got = nv.nvfp4_scale_grad_bwd(dev_bits(wb), dev_bits(gb), torch.from_numpy(s).cuda(),
                                      None if post is None else torch.from_numpy(post).cuda())
        want = oracle.scale_grad_bwd(wb, gb, s, post)
        assert_close_f32(got["gs_pre"].cpu().numpy(), want["gs_pre"], "dL/ds_pre")
        if post is not None:
            assert_close_f32(got["gs_post"].cpu().numpy(), want["gs_post"], "dL/ds_post")
        assert_close_bf16(host_u16(got["gx"]), want["gx"], "dL/dx")
        fq = nv.nvfp4_fakequant_fwd(dev_bits(wb), torch.from_numpy(s).cuda(),
                                    None if post is None else torch.from_numpy(post).cuda())
        assert_close_bf16(host_u16(fq), oracle.fakequant_fwd(wb, s, post)[0], "x~")
