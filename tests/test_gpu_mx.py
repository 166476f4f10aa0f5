"""CUDA MXFP8 quantisation of bf16 tensors against the oracle (End-to-End
4-Bit Training, quantised-linear-layer figure: bf16 gradients quantised to
MXFP8 with stochastic rounding, row-wise and transposed): E4M3 codes and E8M0
scale bytes bit-exact for rows, columns and both from one read, RNE and
stochastic rounding, ragged tiles, column-only calls on unaligned widths,
special values, non-finite blocks, several slices, and the full 16384 x 4096
gradient on sampled rows and columns."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_exact, dev_bits, host_u8
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(xb, blocks, rounding, seed=0, step=0):
    x = xb if xb.ndim == 3 else xb[None]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_mx_quantize(dev_bits(x), nv.Config(blocks=blocks, rounding=rounding, seed=seed,
                                                      step=step), status=st)
    want = oracle.mx_quantize(x, blocks=blocks, rounding=rounding, seed=seed, step=step)
    return got, want, int(st.item())


def _compare(got, want, blocks, what=""):
    if blocks & 1:
        assert_exact(host_u8(got["row"]["codes"]), want["row_codes"], f"row codes {what}")
        assert_exact(host_u8(got["row"]["scales"]), want["row_scales"], f"row scales {what}")
    if blocks & 2:
        assert_exact(host_u8(got["col"]["codes"]), want["col_codes"], f"col codes {what}")
        assert_exact(host_u8(got["col"]["scales"]), want["col_scales"], f"col scales {what}")


# (slices, rows, cols): one tile, several tiles, ragged row and column tiles
SHAPES = [(1, 32, 32), (1, 64, 128), (1, 96, 160), (2, 64, 96), (1, 160, 4096), (3, 32, 288)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("blocks", [1, 2, 3])
@pytest.mark.parametrize("rounding", [0, 1])
def test_mx_quantize_matches_oracle(shape, blocks, rounding):
    S, R, Cc = shape
    xb = synth.student_t(S * R, Cc, seed=R + Cc).reshape(S, R, Cc)
    got, want, st = _run(xb, blocks, rounding, seed=11, step=5)
    assert st == want["status"] == 0
    _compare(got, want, blocks, str(shape))


@pytest.mark.parametrize("shape", [(1, 17, 64), (1, 70, 96), (2, 5, 32)])
def test_rows_only_any_row_count(shape):
    S, R, Cc = shape
    xb = synth.student_t(S * R, Cc, seed=3).reshape(S, R, Cc)
    for rounding in (0, 1):
        got, want, st = _run(xb, 1, rounding, seed=2)
        assert st == 0
        _compare(got, want, 1, str(shape))


@pytest.mark.parametrize("cols", [40, 44, 7, 130])
def test_columns_only_any_width(cols):
    """Column blocks need rows % 32 only; widths that are not multiples of 8
    take the unvectorised load."""
    xb = synth.student_t(64, cols, seed=cols).reshape(1, 64, cols)
    for rounding in (0, 1):
        got, want, st = _run(xb, 2, rounding, seed=4, step=1)
        assert st == 0
        _compare(got, want, 2, f"cols {cols}")


def test_special_values():
    """Zero blocks, signed zeros, values whose scaled form lands in the E4M3
    subnormal range, bf16 subnormals, the largest bf16 values, and block
    maxima exactly on the 1.75 * 2^k boundary of the shared exponent."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[0, :32] = 0.0
    x[1, :32] = -0.0
    x[2, :32] = rng.standard_normal(32) * 1e-3
    x[2, 0] = 300.0                                     # tiny neighbours of a large max
    x[3, :32] = 1.75 * 2.0 ** 10
    x[3, 1:32] *= rng.uniform(-1, 1, 31)
    x[4, :32] = 1.0e-39                                 # bf16 subnormals
    x[5, :32] = 3.0e38 * np.sign(rng.standard_normal(32))
    x[6, 32:64] = 448.0
    x[7, 64:96] = -2.0 ** -20
    x[:, 100] = 0.0                                     # a zero column
    # smallest value exactly at / just below E4M3's normal range after scaling
    # (block max 448 gives e = 0): the two sides of the stand-in pattern
    x[8, :32] = rng.standard_normal(32) * 100
    x[8, 0], x[8, 5] = 448.0, 2.0 ** -6
    x[9, :32] = rng.standard_normal(32) * 100
    x[9, 0], x[9, 5] = 448.0, 2.0 ** -6 - 2.0 ** -14
    x[32:64, 102] = rng.standard_normal(32) * 100
    x[32, 102], x[40, 102] = -448.0, -(2.0 ** -6)
    x[32:64, 103] = rng.standard_normal(32) * 100
    x[32, 103], x[41, 103] = 448.0, 2.0 ** -6 - 2.0 ** -14
    x[:, 101] = 1.75 * 2.0 ** -30                       # a constant column on the boundary
    xb = synth.to_bf16_bits(x).reshape(1, 64, 256)
    for rounding in (0, 1):
        got, want, st = _run(xb, 3, rounding, seed=9)
        assert st == want["status"] == 0
        _compare(got, want, 3, f"rounding {rounding}")


def test_nonfinite_blocks_raise_status_and_leave_others_exact():
    xb = synth.student_t(64, 128, seed=5).reshape(1, 64, 128).copy()
    xb[0, 3, 5] = 0x7FC0   # NaN in row block (3, 0); column blocks (5, 0)
    xb[0, 40, 70] = 0xFF80  # -Inf in row block (40, 2); column blocks (70, 1)
    got, want, st = _run(xb, 3, 1, seed=1)
    assert st & nv.DEV_NONFINITE_INPUT and want["status"] & oracle.ST_NONFINITE_INPUT
    rc, rs = host_u8(got["row"]["codes"])[0], host_u8(got["row"]["scales"])[0]
    cc, cs = host_u8(got["col"]["codes"])[0], host_u8(got["col"]["scales"])[0]
    rmask = np.ones((64, 4), bool)
    rmask[3, 0] = rmask[40, 2] = False
    cmask = np.ones((128, 2), bool)
    cmask[5, 0] = cmask[70, 1] = False
    wrc, wrs = want["row_codes"][0], want["row_scales"][0]
    wcc, wcs = want["col_codes"][0], want["col_scales"][0]
    assert_exact(rs[rmask], wrs[rmask], "row scales of finite blocks")
    assert_exact(rc.reshape(64, 4, 32)[rmask], wrc.reshape(64, 4, 32)[rmask], "row codes")
    assert_exact(cs[cmask], wcs[cmask], "col scales of finite blocks")
    assert_exact(cc.reshape(128, 2, 32)[cmask], wcc.reshape(128, 2, 32)[cmask], "col codes")


def test_draws_depend_on_seed_step_and_direction():
    xb = synth.student_t(64, 128, seed=8).reshape(1, 64, 128)
    a, _, _ = _run(xb, 3, 1, seed=1, step=0)
    b, _, _ = _run(xb, 3, 1, seed=1, step=0)
    c, _, _ = _run(xb, 3, 1, seed=1, step=1)
    ra, rb, rc = (host_u8(o["row"]["codes"]) for o in (a, b, c))
    assert np.array_equal(ra, rb)
    assert not np.array_equal(ra, rc)
    # the column encoding draws its own bits: on a symmetric tensor (X = X^T)
    # the two encodings see the same values but round some differently
    xs = synth.student_t(64, 64, seed=2).reshape(64, 64)
    upper = np.arange(64)[:, None] <= np.arange(64)[None, :]
    sym = np.where(upper, xs, xs.T)
    got, want, _ = _run(sym[None], 3, 1, seed=3)
    _compare(got, want, 3, "symmetric")
    assert not np.array_equal(host_u8(got["row"]["codes"]), host_u8(got["col"]["codes"]))


def test_outputs_written_into_caller_buffers_twice_in_a_row():
    xb = synth.student_t(96, 192, seed=6).reshape(1, 96, 192)
    row, col = nv.alloc_mx(1, 96, 192, "cuda"), nv.alloc_mx(1, 192, 96, "cuda")
    for t in (0, 1):
        for d in (row, col):
            d["codes"].fill_(0xAB)
            d["scales"].fill_(0xCD)
        nv.nvfp4_mx_quantize(dev_bits(xb), nv.Config(blocks=3, rounding=1, seed=4, step=t),
                             row=row, col=col)
        want = oracle.mx_quantize(xb, blocks=3, rounding=1, seed=4, step=t)
        _compare({"row": row, "col": col}, want, 3, f"step {t}")


def test_full_size_gradient_on_sampled_rows_and_columns():
    """The 16384 x 4096 gradient, both encodings with stochastic rounding in
    one launch (as timed); sampled rows and columns re-encoded by the oracle's
    MX encoder at their flat indices in the full layouts."""
    R, Cc, seed, step = 16384, 4096, 12, 3
    xb = synth.DriftingGradient(R, Cc, seed=3).step(0)
    got = nv.nvfp4_mx_quantize(dev_bits(xb), nv.Config(blocks=3, rounding=1, seed=seed,
                                                       step=step))
    rc, rs = host_u8(got["row"]["codes"])[0], host_u8(got["row"]["scales"])[0]
    cc, cs = host_u8(got["col"]["codes"])[0], host_u8(got["col"]["scales"])[0]
    x = synth.bf16_bits_to_f32(xb)
    rng = np.random.default_rng(5)
    rows = np.concatenate([[0, R - 1], rng.choice(R, 14, replace=False)])
    cols = np.concatenate([[0, Cc - 1], rng.choice(Cc, 14, replace=False)])
    for r in rows:
        codes, scales = oracle.mx_encode(x[r], 1, seed, step, 0, int(r) * Cc)
        assert_exact(rc[r], codes, f"row {r} codes")
        assert_exact(rs[r], scales, f"row {r} scales")
    for c in cols:
        codes, scales = oracle.mx_encode(np.ascontiguousarray(x[:, c]), 1, seed, step, 1,
                                         int(c) * R)
        assert_exact(cc[c], codes, f"column {c} codes")
        assert_exact(cs[c], scales, f"column {c} scales")
