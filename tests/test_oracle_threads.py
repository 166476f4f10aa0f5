"""The oracle's OpenMP build (used only to time the oracle on all host cores)
returns the same bytes as its single-threaded build for every entry point,
on shapes whose 4/6 bitmap words straddle rows and slices."""
import numpy as np
import pytest

from nvfp4_block_scaled_02_gb300 import synth


@pytest.fixture
def both(orc):
    """Run fn once on one thread and once on four; return both results."""
    def run(fn):
        orc.set_threads(1)
        a = fn()
        assert orc.set_threads(4) == 4
        try:
            b = fn()
        finally:
            orc.set_threads(1)
        return a, b
    return run


def _same(a, b):
    if a is None:
        assert b is None
    elif isinstance(a, dict):
        assert a.keys() == b.keys()
        for k in a:
            _same(a[k], b[k])
    elif isinstance(a, tuple):
        for u, v in zip(a, b):
            _same(u, v)
    else:
        a, b = (np.ascontiguousarray(np.atleast_1d(np.asarray(t))) for t in (a, b))
        assert a.dtype == b.dtype and a.shape == b.shape
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


@pytest.mark.parametrize("blocks,fos,rounding", [(1, 1, 0), (2, 1, 1), (3, 1, 0), (3, 0, 1)])
def test_quantize(orc, both, blocks, fos, rounding):
    x = synth.student_t(3 * 48, 80, seed=11).reshape(3, 48, 80)  # 5 blocks per row
    a, _ = orc.global_amax(x, 3)
    _same(*both(lambda: orc.quantize(x, a, blocks=blocks, four_over_six=fos, rounding=rounding,
                                     seed=5, step=2)))


def test_amax(orc, both):
    x = synth.student_t(64, 112, seed=12)
    x[17, 33] = 0x7F80  # +Inf: the status bit is OR-reduced
    _same(*both(lambda: orc.global_amax(x.reshape(4, 16, 112), 4)))


def test_ste(orc, both):
    wb, gb, s = synth.scale_learning(rows=32, cols=96, seed=2)
    so = (s * np.float32(1.25)).astype(np.float32)
    _same(*both(lambda: orc.fakequant_fwd(wb, s, so)))
    _same(*both(lambda: orc.scale_grad_bwd(wb, gb, s, so)))
    _same(*both(lambda: orc.scale_grad_bwd(wb, gb, s)))
    gam = float(np.abs(synth.bf16_bits_to_f32(wb)).max()) * 1.5
    _same(*both(lambda: orc.fakequant_fwd_fp8(wb, s, so, gam)))
    _same(*both(lambda: orc.scale_grad_bwd_fp8(wb, gb, s, so, gam)))
    _same(*both(lambda: orc.scale_init_mse(wb, gam)))
    _same(*both(lambda: orc.export_scales(wb, s, so, gam)))


@pytest.mark.parametrize("target", [0, 1])
def test_requant(orc, both, target):
    x = synth.student_t(64, 48, seed=13)
    a, _ = orc.global_amax(x)
    q = orc.quantize(x, a, four_over_six=1, dequant=False)
    _same(*both(lambda: orc.requant(q["row_codes"], q["row_scales"], a, target=target,
                                    rounding=1, seed=7, src_fos=1, dst_fos=target)))


def test_mx_and_tile16(orc, both):
    x = synth.student_t(64, 96, seed=14)
    a, _ = orc.global_amax(x)
    _same(*both(lambda: orc.mx_quantize(x, blocks=3, rounding=1, seed=12, step=1)))
    _same(*both(lambda: orc.quantize_tile16(x, a, rounding=1, seed=3)))
