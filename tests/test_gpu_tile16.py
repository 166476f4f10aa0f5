"""CUDA 16x16 tile-scale quantiser against the oracle: row encoding and its
transposed column encoding bit-exact (codes, scales, dequant), both scale
formats, RNE and stochastic rounding, several slices, bad amax, and the
activation-size tensor on sampled row bands."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_exact, dev_bits, host_u16, host_u8
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def run_both(xb, gamax, *, fmt=0, rounding=0, seed=0, step=0, scale_max=0.0, dequant=True):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = nv.Config(blocks=nv.BLOCKS_TILE16, scale_fmt=fmt, rounding=rounding, seed=seed,
                    step=step, scale_max=scale_max)
    out = nv.nvfp4_quantize(dev_bits(xb), torch.from_numpy(np.asarray(gamax, np.float32)).cuda(),
                            cfg, status=st, dequant=dequant)
    torch.cuda.synchronize()
    ref = oracle.quantize_tile16(xb, gamax, scale_fmt=fmt, rounding=rounding, seed=seed, step=step,
                                 scale_max=scale_max, dequant=dequant)
    return out, ref, int(st.item())


def _check(out, ref, st, dequant=True):
    assert st == ref["status"]
    for side in ("row", "col"):
        o = out[side]
        assert_exact(host_u8(o["codes"]), ref[side + "_codes"], side + " codes")
        assert_exact(host_u8(o["scales"]), ref[side + "_scales"], side + " scales")
        if dequant:
            assert_exact(host_u16(o["dequant"]), ref[side + "_dq"], side + " dequant")


SHAPES = [(1, 16, 16), (2, 48, 80), (3, 64, 272), (1, 512, 1024)]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_tile16_matches_oracle(shape, fmt, rounding):
    S, R, Cc = shape
    xb = synth.outlier_normal(S * R, Cc, seed=R + Cc).reshape(shape)
    gamax, _ = oracle.global_amax(xb, S)
    out, ref, st = run_both(xb, gamax, fmt=fmt, rounding=rounding, seed=5, step=7)
    _check(out, ref, st)


def test_tile16_without_dequant_and_stale_amax():
    xb = synth.student_t(96, 160, seed=3).reshape(1, 96, 160)
    gamax, _ = oracle.global_amax(xb)
    out, ref, st = run_both(xb, gamax * np.float32(0.1), dequant=False)  # saturating scales
    _check(out, ref, st, dequant=False)


def test_tile16_bad_amax_is_flagged():
    xb = synth.outlier_normal(32, 32, seed=1).reshape(1, 32, 32)
    _, _, st = run_both(xb, np.array([np.nan], np.float32))
    assert st & nv.DEV_BAD_AMAX


def test_tile16_column_is_transposed_row_on_device():
    xb = synth.student_t(128, 256, seed=4).reshape(1, 128, 256)
    gamax, _ = oracle.global_amax(xb)
    out, _, _ = run_both(xb, gamax, rounding=1, seed=3)
    rd = host_u16(out["row"]["dequant"]).reshape(128, 256)
    cd = host_u16(out["col"]["dequant"]).reshape(256, 128)
    assert np.array_equal(cd, rd.T)


def test_tile16_activation_size_sampled_bands():
    """8192 x 4096 in one launch (RNE); 6 row bands of 16 re-encoded by the
    oracle on their own (tiles are independent given the slice's global
    amax). Stochastic rounding is compared at the smaller sizes, where the
    oracle sees the same flat indices."""
    xb = synth.student_t(8192, 4096, seed=1)
    gamax, _ = oracle.global_amax(xb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = nv.nvfp4_quantize(dev_bits(xb), torch.from_numpy(gamax).cuda(),
                            nv.Config(blocks=nv.BLOCKS_TILE16), status=st)
    rc = host_u8(out["row"]["codes"]).reshape(8192, 2048)
    rs = host_u8(out["row"]["scales"]).reshape(8192, 256)
    cc = host_u8(out["col"]["codes"]).reshape(4096, 4096)
    cs = host_u8(out["col"]["scales"]).reshape(4096, 512)
    bands = np.random.default_rng(2).choice(512, 6, replace=False)
    bands[:2] = (0, 511)
    for b in bands:
        ref = oracle.quantize_tile16(xb[16 * b:16 * b + 16], gamax, dequant=False)
        assert_exact(rc[16 * b:16 * b + 16], ref["row_codes"][0], f"band {b} codes")
        assert_exact(rs[16 * b:16 * b + 16], ref["row_scales"][0], f"band {b} scales")
        assert_exact(cc[:, 8 * b:8 * b + 8], ref["col_codes"][0], f"band {b} column codes")
        assert_exact(cs[:, b], ref["col_scales"][0][:, 0], f"band {b} column scales")
    assert int(st.item()) == 0


@pytest.mark.parametrize("shape", [(1, 80, 144), (2, 64, 128)])
def test_tile16_row_encoding_alone(shape):
    """The column encoding is optional at the ABI: a call with no column
    outputs writes the same row encoding."""
    import ctypes as C
    S, R, Cc = shape
    xb = synth.student_t(S * R, Cc, seed=R).reshape(shape)
    gamax, _ = oracle.global_amax(xb, S)
    row = nv.alloc_encoding(S, R, Cc, "cuda", False, True)
    x = dev_bits(xb)
    gam = torch.from_numpy(np.asarray(gamax, np.float32)).cuda()
    cfg = nv.Config(blocks=nv.BLOCKS_TILE16, rounding=1, seed=2, step=1).c()
    ro = nv._out(row)
    rc = nv.lib().nvfp4_quantize(C.byref(cfg), x.data_ptr(), S, R, Cc, gam.data_ptr(),
                                 C.byref(ro), None, None,
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ref = oracle.quantize_tile16(xb, gamax, rounding=1, seed=2, step=1)
    assert_exact(host_u8(row["codes"]), ref["row_codes"], "row codes")
    assert_exact(host_u8(row["scales"]), ref["row_scales"], "row scales")
    assert_exact(host_u16(row["dequant"]), ref["row_dq"], "row dequant")


def test_tile16_nonfinite_input_flags_and_other_tiles_exact():
    """A NaN and an Inf in two tiles set the non-finite status bit; every other
    tile of both encodings matches the oracle."""
    xb = synth.student_t(64, 96, seed=8).reshape(1, 64, 96).copy()
    xb[0, 3, 5] = 0x7FC0    # NaN in tile (0, 0)
    xb[0, 40, 70] = 0xFF80  # -Inf in tile (2, 4)
    gamax = np.array([4.0], np.float32)
    out, ref, st = run_both(xb, gamax)
    assert st & nv.DEV_NONFINITE_INPUT
    bad = {(0, 0), (2, 4)}
    rc = host_u8(out["row"]["codes"]).reshape(64, 48)
    rs = host_u8(out["row"]["scales"]).reshape(64, 6)
    cc = host_u8(out["col"]["codes"]).reshape(96, 32)
    cs = host_u8(out["col"]["scales"]).reshape(96, 4)
    wrc, wrs = ref["row_codes"].reshape(64, 48), ref["row_scales"].reshape(64, 6)
    wcc, wcs = ref["col_codes"].reshape(96, 32), ref["col_scales"].reshape(96, 4)
    for tr in range(4):
        for tc in range(6):
            if (tr, tc) in bad:
                continue
            rows, cols = slice(16 * tr, 16 * tr + 16), slice(16 * tc, 16 * tc + 16)
            assert_exact(rc[rows, 8 * tc:8 * tc + 8], wrc[rows, 8 * tc:8 * tc + 8], f"row codes {tr},{tc}")
            assert_exact(rs[rows, tc], wrs[rows, tc], f"row scales {tr},{tc}")
            assert_exact(cc[cols, 8 * tr:8 * tr + 8], wcc[cols, 8 * tr:8 * tr + 8], f"col codes {tr},{tc}")
            assert_exact(cs[cols, tr], wcs[cols, tr], f"col scales {tr},{tc}")


@pytest.mark.parametrize("gam", [1e-45, 1e-40])
def test_tile16_zero_tiles_under_a_tiny_slice_amax(gam):
    xb = np.zeros((1, 64, 128), np.uint16)
    xb[0, 3, 5] = synth.to_bf16_bits(np.array([2e-39], np.float32))[0]
    for fmt in (0, 1):
        out, ref, st = run_both(xb, np.array([gam], np.float32), fmt=fmt)
        _check(out, ref, st)
        sc = host_u8(out["row"]["scales"]).reshape(64, 8)  # the 16 row blocks of a tile share its scale
        assert np.all(sc[:16, 0] == sc[0, 0]) and sc[16:].max() == 0 and sc[:, 1:].max() == 0
