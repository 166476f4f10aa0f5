"""Per-token (per-row outer scale) single-pass quantiser against the oracle:
per-token scaling is the row encoding of the tensor taken as `rows` slices of
one row each, with every slice's global amax its own row amax."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
import oracle
from helpers import assert_exact, compare_encoding, dev_bits
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def run_token(xb, *, fmt=0, rounding=0, fos=0, scale_max=0.0, seed=0, step=0, dequant=True):
    R, Cc = xb.shape
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cfg = nv.Config(scale_fmt=fmt, rounding=rounding, four_over_six=fos, scale_max=scale_max,
                    seed=seed, step=step)
    out = nv.nvfp4_quantize_per_token(dev_bits(xb), cfg, status=st, dequant=dequant)
    torch.cuda.synchronize()
    slices = xb.reshape(R, 1, Cc)
    amax, ast = oracle.global_amax(slices, R)
    ref = oracle.quantize(slices, amax, scale_fmt=fmt, rounding=rounding, four_over_six=fos,
                          scale_max=scale_max, seed=seed, step=step, dequant=dequant)
    return out, ref, amax, int(st.item()), ref["status"] | ast


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rounding", [0, 1])
@pytest.mark.parametrize("fos", [0, 1])
@pytest.mark.parametrize("shape", [(1, 16), (7, 80), (33, 528), (130, 4096), (5, 4112),
                                   (9, 8192), (3, 16384), (2, 16400), (2, 40000)])
def test_per_token_matches_oracle(shape, fmt, rounding, fos):
    xb = synth.student_t(*shape, seed=sum(shape))
    out, ref, amax, st, wst = run_token(xb, fmt=fmt, rounding=rounding, fos=fos, seed=9, step=4)
    assert st == wst == 0
    assert_exact(out["row_amax"].cpu().numpy().view(np.uint32), amax.view(np.uint32), "row amax")
    compare_encoding(out, ref, "row_", f"per-token fmt={fmt} sr={rounding} fos={fos}", bool(fos))


def test_per_token_equals_two_pass_api():
    """The fused kernel gives the same bytes as nvfp4_amax + nvfp4_quantize with
    one slice per row."""
    xb = synth.outlier_normal(64, 1024, seed=5)
    R, Cc = xb.shape
    x = dev_bits(xb)
    cfg = nv.Config(four_over_six=1)
    fused = nv.nvfp4_quantize_per_token(x, cfg)
    x3 = x.view(R, 1, Cc)
    two = nv.nvfp4_quantize(x3, nv.nvfp4_amax(x3), cfg)["row"]
    for k in ("codes", "scales", "choice", "dequant"):
        assert torch.equal(fused[k].reshape(-1).view(torch.uint8), two[k].reshape(-1).view(torch.uint8)), k


def test_per_token_zero_rows_and_nonfinite():
    xb = synth.uniform_bits((4, 64), seed=2)
    xb[1] = 0
    out, ref, amax, st, wst = run_token(xb, fos=1)
    assert st == 0 and amax[1] == 0
    compare_encoding(out, ref, "row_", "zero row", True)
    xb[2, 5] = 0x7FC0
    st_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    nv.nvfp4_quantize_per_token(dev_bits(xb), nv.Config(), status=st_t)
    assert int(st_t.item()) & nv.DEV_NONFINITE_INPUT
