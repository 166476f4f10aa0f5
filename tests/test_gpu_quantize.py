"""CUDA quantiser against the oracle, element by element: global amax, row
(1x16), column (16x1) and dual encodings, every scale format / rounding / 4/6
combination, on shapes that span several tiles with ragged tails, plus the
edge cases (empty, zeros, saturation by a stale amax, non-finite input, bad
amax)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import (assert_exact, compare_encoding, dev_bits, host_u16, host_u8)
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def run_both(xb, gamax, *, blocks=1, fmt=0, rounding=0, fos=0, scale_max=0.0, seed=0, step=0,
             dequant=True, check=True):
    x = dev_bits(xb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = nv.Config(blocks=blocks, scale_fmt=fmt, rounding=rounding, four_over_six=fos,
                    scale_max=scale_max, seed=seed, step=step)
    out = nv.nvfp4_quantize(x, torch.from_numpy(np.asarray(gamax, np.float32)).cuda(), cfg,
                            status=st, dequant=dequant)
    torch.cuda.synchronize()
    ref = oracle.quantize(xb, gamax, blocks=blocks, scale_fmt=fmt, rounding=rounding,
                          four_over_six=fos, scale_max=scale_max, seed=seed, step=step,
                          dequant=dequant)
    if check:
        assert int(st.item()) == ref["status"]
        what = f"blocks={blocks} fmt={fmt} sr={rounding} fos={fos}"
        if blocks & 1:
            compare_encoding(out["row"], ref, "row_", what + " row", bool(fos), dequant)
        if blocks & 2:
            compare_encoding(out["col"], ref, "col_", what + " col", bool(fos), dequant)
    return out, ref, int(st.item())


# ------------------------------------------------------------------ amax --

@pytest.mark.parametrize("shape", [(1, 1024, 1024), (3, 5, 7), (2, 33, 48), (1, 1, 9),
                                   (64, 16, 32), (1, 3000, 4096)])
def test_amax_matches_oracle(shape):
    xb = synth.uniform_bits(shape, seed=sum(shape), lo=-3, hi=3)
    xb.reshape(-1)[np.random.default_rng(1).integers(0, xb.size, 3)] = synth.to_bf16_bits(
        np.array([-7.5, 11.0, 0.5], np.float32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_amax(dev_bits(xb), status=st).cpu().numpy()
    want, wst = oracle.global_amax(xb, shape[0])
    assert_exact(got.view(np.uint32), want.view(np.uint32), "amax")
    assert int(st.item()) == wst == 0


def test_amax_flags_nonfinite():
    xb = synth.uniform_bits((2, 16, 64), seed=3)
    xb[1, 3, 5] = 0xFF80  # -inf
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nvfp4_amax(dev_bits(xb), status=st)
    assert int(st.item()) & nv.DEV_NONFINITE_INPUT


# ------------------------------------------------------------- row blocks --

SHAPES = [(1, 48, 80), (3, 64, 160), (2, 129, 4096), (1, 1024, 1024), (5, 16, 16)]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("fos", [0, 1])
@pytest.mark.parametrize("shape", SHAPES)
def test_row_blocks(shape, fmt, rounding, fos):
    xb = synth.outlier_normal(shape[0] * shape[1], shape[2], seed=7).reshape(shape)
    gamax, _ = oracle.global_amax(xb, shape[0])
    run_both(xb, gamax, blocks=1, fmt=fmt, rounding=rounding, fos=fos, seed=11, step=3)


@pytest.mark.parametrize("blocks", [2, 3])
@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("fos", [0, 1])
@pytest.mark.parametrize("shape", [(1, 48, 80), (2, 160, 272), (1, 64, 128), (3, 208, 144)])
def test_column_and_dual_blocks(shape, blocks, fmt, rounding, fos):
    xb = synth.student_t(shape[0] * shape[1], shape[2], seed=8).reshape(shape)
    gamax, _ = oracle.global_amax(xb, shape[0])
    run_both(xb, gamax, blocks=blocks, fmt=fmt, rounding=rounding, fos=fos, seed=5, step=9)


@pytest.mark.parametrize("blocks", [2, 3])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("shape", [(19, 16, 48), (11, 80, 32), (9, 64, 128)])
def test_dual_runs_across_many_slices(shape, blocks, rounding):
    """Slices of one or a few tiles each, every slice a different magnitude:
    a CTA's run of consecutive tiles crosses slices (each needs its own outer
    scale and scale table) and most tiles are partial."""
    S, R, C = shape
    f = synth.bf16_bits_to_f32(synth.student_t(S * R, C, seed=12)).reshape(S, R, C)
    f = f * (2.0 ** (np.arange(S, dtype=np.float32) - S // 2))[:, None, None]
    xb = synth.to_bf16_bits(f)
    gamax, _ = oracle.global_amax(xb, S)
    run_both(xb, gamax, blocks=blocks, fos=1, rounding=rounding, seed=3, step=4)


@pytest.mark.parametrize("shape", [(1, 32, 24), (2, 48, 40), (1, 16, 7)])
def test_column_blocks_with_unaligned_rows(shape):
    """Column-only encoding needs rows % 16 only; rows of the input may be any
    length (here not a multiple of 8 values)."""
    xb = synth.uniform_bits(shape, seed=4)
    gamax, _ = oracle.global_amax(xb, shape[0])
    run_both(xb, gamax, blocks=2, fos=1)


def test_row_without_dequant_and_explicit_scale_max():
    xb = synth.student_t(64, 512, seed=2)
    gamax, _ = oracle.global_amax(xb)
    run_both(xb, gamax, fos=1, scale_max=300.0, dequant=False)
    run_both(xb[None], gamax, blocks=3, fos=1, scale_max=200.0, dequant=False)


# ------------------------------------------------------------- edge cases --

def test_zero_tensor_and_zero_amax():
    xb = np.zeros((1, 32, 64), np.uint16)
    xb[0, 1, 3] = 0x8000  # -0
    for blocks in (1, 3):
        out, ref, st = run_both(xb, np.zeros(1, np.float32), blocks=blocks, fos=1)
        assert st == 0
        assert host_u8(out["row"]["scales"]).max() == 0


def test_stale_amax_saturates_scales():
    xb = synth.outlier_normal(64, 256, seed=9)
    stale = np.array([0.05], np.float32)  # far below the current amax
    for fmt in (0, 1):
        for blocks in (1, 3):
            out, ref, _ = run_both(xb[None], stale, blocks=blocks, fmt=fmt, fos=0)
            top = 0x7E if fmt == 0 else 0xFF
            assert (host_u8(out["row"]["scales"]) == top).any()


def test_tiny_and_huge_magnitudes():
    vals = np.array([1e-38, 3e-39, 9.2e-41, 1e-30, 1e30, 3e38, -3e38, 1.0, -1e-40],
                    np.float32)
    xb = synth.to_bf16_bits(np.resize(vals, (16, 16 * 9))).reshape(1, 16, -1)
    for gam in (None, np.array([1e-36], np.float32), np.array([3.0e38], np.float32)):
        g = oracle.global_amax(xb)[0] if gam is None else gam
        for fmt in (0, 1):
            run_both(xb, g, blocks=3, fmt=fmt, fos=1, rounding=1, seed=2)


def test_nonfinite_input_is_flagged():
    xb = synth.uniform_bits((1, 32, 64), seed=6)
    xb[0, 7, 9] = 0x7FC0  # NaN
    gamax = np.array([8.0], np.float32)
    for blocks in (1, 2, 3):
        _, ref, st = run_both(xb, gamax, blocks=blocks, fos=1, check=False)
        assert st & nv.DEV_NONFINITE_INPUT and ref["status"] & oracle.ST_NONFINITE_INPUT


@pytest.mark.parametrize("bad", [np.nan, np.inf, -1.0])
def test_bad_amax_is_flagged(bad):
    xb = synth.uniform_bits((1, 16, 32), seed=6)
    for blocks in (1, 3):
        _, ref, st = run_both(xb, np.array([bad], np.float32), blocks=blocks, check=False)
        assert st & nv.DEV_BAD_AMAX and ref["status"] & oracle.ST_BAD_AMAX


def test_empty_inputs():
    for shape in ((0, 16, 32), (1, 0, 32), (1, 16, 0)):
        x = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        out = nv.nvfp4_quantize(x, torch.zeros(max(shape[0], 1), device="cuda"),
                                nv.Config(blocks=3, four_over_six=1))
        assert out["row"]["codes"].numel() == 0 or shape[0] == 0
    assert nv.nvfp4_amax(torch.zeros((0, 4, 4), dtype=torch.bfloat16, device="cuda")).numel() == 0
    a = nv.nvfp4_amax(torch.zeros((2, 0, 4), dtype=torch.bfloat16, device="cuda"))
    assert a.cpu().tolist() == [0.0, 0.0]


def test_guard_bytes_untouched():
    """Outputs are written exactly where the layout says and nowhere else."""
    S, R, Cc = 2, 80, 96
    xb = synth.student_t(S * R, Cc, seed=12).reshape(S, R, Cc)
    gamax, _ = oracle.global_amax(xb, S)
    for blocks in (1, 3):
        encs = {}
        views = {}
        for tag, (rr, cc) in (("row", (R, Cc)), ("col", (Cc, R))):
            if not (blocks & (1 if tag == "row" else 2)):
                continue
            nb = S * rr * cc // 16
            w = S * ((rr * cc // 16 + 31) // 32)
            pad = 64
            raw = {
                "codes": torch.full((nb * 8 + pad,), 0xA5, dtype=torch.uint8, device="cuda"),
                "scales": torch.full((nb + pad,), 0xA5, dtype=torch.uint8, device="cuda"),
                "choice": torch.full((w + pad,), -0x5A5A5A5B, dtype=torch.int32, device="cuda"),
                "dequant": torch.full((nb * 16 + pad,), 0x5A5A, dtype=torch.int16, device="cuda"),
            }
            views[tag] = raw
            encs[tag] = {"codes": raw["codes"][:nb * 8], "scales": raw["scales"][:nb],
                         "choice": raw["choice"][:w], "dequant": raw["dequant"][:nb * 16]}
        cfg = nv.Config(blocks=blocks, four_over_six=1)
        nv.nvfp4_quantize(dev_bits(xb), torch.from_numpy(gamax).cuda(), cfg,
                          row=encs.get("row"), col=encs.get("col"))
        torch.cuda.synchronize()
        ref = oracle.quantize(xb, gamax, blocks=blocks, four_over_six=1)
        for tag, raw in views.items():
            assert (raw["codes"][-64:] == 0xA5).all() and (raw["scales"][-64:] == 0xA5).all()
            assert (raw["choice"][-64:] == -0x5A5A5A5B).all()
            assert (raw["dequant"][-64:] == 0x5A5A).all()
            assert_exact(host_u8(encs[tag]["codes"]), ref[tag + "_codes"], tag + " codes")


def test_periodic_helper_refreshes_on_schedule():
    xs = [synth.uniform_bits((8, 64), seed=t, lo=-(t + 1), hi=t + 1) for t in range(5)]
    pa = nv.PeriodicAmax(period=2)
    seen = []
    for t, xb in enumerate(xs):
        seen.append(pa(dev_bits(xb), t).item())
    want = [oracle.global_amax(xs[t - t % 2])[0][0] for t in range(5)]
    assert seen == [float(w) for w in want] and pa.refreshes == 3


@pytest.mark.parametrize("rule", [1, 2])
@pytest.mark.parametrize("blocks", [1, 3])
@pytest.mark.parametrize("rounding", [0, 1])
def test_alternative_four_over_six_rules(rule, blocks, rounding):
    xb = synth.student_t(160, 272, seed=13 + rule)[None]
    gamax, _ = oracle.global_amax(xb)
    x = dev_bits(xb)
    cfg = nv.Config(blocks=blocks, four_over_six=1, rounding=rounding, seed=7,
                    four_over_six_rule=rule)
    out = nv.nvfp4_quantize(x, torch.from_numpy(gamax).cuda(), cfg)
    torch.cuda.synchronize()
    ref = oracle.quantize(xb, gamax, blocks=blocks, four_over_six=1, rounding=rounding, seed=7,
                          rule=rule)
    compare_encoding(out["row"], ref, "row_", f"rule {rule} row", True)
    if blocks & 2:
        compare_encoding(out["col"], ref, "col_", f"rule {rule} col", True)
    tok = nv.nvfp4_quantize_per_token(x[0], cfg if blocks == 1 else nv.Config(
        four_over_six=1, rounding=rounding, seed=7, four_over_six_rule=rule))
    s = xb[0].reshape(-1, 1, 272)
    a, _ = oracle.global_amax(s, s.shape[0])
    rt = oracle.quantize(s, a, four_over_six=1, rounding=rounding, seed=7, rule=rule)
    compare_encoding(tok, rt, "row_", f"rule {rule} per-token", True)


def test_more_slices_than_one_grid_dimension_holds():
    """70000 slices of one 16-value row each: the per-slice launches split the
    slices over several grids (at most 65535 per grid dimension)."""
    S = 70000
    xb = synth.outlier_normal(S, 16, seed=12).reshape(S, 1, 16)
    x = dev_bits(xb)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    amax = nv.nvfp4_amax(x, status=st)
    out = nv.nvfp4_quantize(x, amax, nv.Config(four_over_six=1), status=st)["row"]
    ref_amax, _ = oracle.global_amax(xb, S)
    ref = oracle.quantize(xb, ref_amax, four_over_six=1)
    assert int(st.item()) == ref["status"] == 0
    assert_exact(amax.cpu().numpy().view(np.uint32), ref_amax.view(np.uint32), "amaxes")
    assert_exact(host_u8(out["codes"]), ref["row_codes"], "codes")
    assert_exact(host_u8(out["scales"]), ref["row_scales"], "scales")
    assert_exact(out["choice"].cpu().numpy().view(np.uint32), ref["row_choice"], "4/6 choices")
    assert_exact(host_u16(out["dequant"]), ref["row_dq"], "dequant")


@pytest.mark.parametrize("gam", [1e-45, 1e-40, 1e-30])
def test_zero_blocks_under_a_tiny_slice_amax(gam):
    """A tiny slice amax makes 1/(k g) overflow fp32 (clamped to FLT_MAX):
    zero blocks still encode to scale 0, the others as the oracle does, in
    every encoding."""
    xb = np.zeros((2, 32, 64), np.uint16)
    rng = np.random.default_rng(int(-np.log10(gam)))
    xb[:, ::5, ::7] = synth.to_bf16_bits(rng.standard_normal(xb[:, ::5, ::7].shape) * 1e-38)
    g = np.full(2, gam, np.float32)
    for blocks in (1, 3):
        for fmt in (0, 1):
            for fos in (0, 1):
                out, ref, st = run_both(xb, g, blocks=blocks, fmt=fmt, fos=fos, rounding=fos,
                                        seed=4)
                assert st == 0
