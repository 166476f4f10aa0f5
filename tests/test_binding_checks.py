"""The Python binding refuses buffers the kernels would read or write past
(too few elements or the wrong element type) before anything reaches the
library; run with CPU tensors, since the checks come first."""
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv


def _x(s, r, c):
    return torch.zeros((s, r, c), dtype=torch.bfloat16)


def test_quantize_output_and_amax_sizes():
    x = _x(2, 32, 64)
    amax = torch.zeros(2)
    row = nv.alloc_encoding(2, 32, 64, "cpu", False)
    row["codes"] = row["codes"][:1]
    with pytest.raises(ValueError, match="row codes"):
        nv.nvfp4_quantize(x, amax, nv.Config(), row=row)
    with pytest.raises(ValueError, match="global_amax"):
        nv.nvfp4_quantize(x, torch.zeros(1), nv.Config())
    with pytest.raises(TypeError, match="global_amax"):
        nv.nvfp4_quantize(x, torch.zeros(2, dtype=torch.float64), nv.Config())
    col = nv.alloc_encoding(2, 64, 32, "cpu", True)
    col["choice"] = None
    with pytest.raises(ValueError, match="choice"):
        nv.nvfp4_quantize(x, amax, nv.Config(blocks=2, four_over_six=1), col=col)
    small_dq = nv.alloc_encoding(2, 32, 64, "cpu", False)
    small_dq["dequant"] = small_dq["dequant"][:, :16]
    with pytest.raises(ValueError, match="row dequant"):
        nv.nvfp4_quantize(x, amax, nv.Config(), row=small_dq)


def test_scale_learning_buffer_sizes():
    x = torch.zeros((16, 64), dtype=torch.bfloat16)
    s = torch.ones((16, 4))
    with pytest.raises(ValueError, match="s_pre"):
        nv.nvfp4_fakequant_fwd(x, s[:8])
    with pytest.raises(TypeError, match="s_post"):
        nv.nvfp4_fakequant_fwd(x, s, s.double())
    with pytest.raises(ValueError, match="gq"):
        nv.nvfp4_scale_grad_bwd(x, x[:8], s)
    with pytest.raises(ValueError, match="gs_pre"):
        nv.nvfp4_scale_grad_bwd(x, x, s, gs_pre=s[:2])
    with pytest.raises(ValueError, match="global_amax"):
        nv.nvfp4_scale_init_mse(x, torch.zeros(0))


def test_requant_mx_and_token_output_sizes():
    codes = torch.zeros((1, 64, 32), dtype=torch.uint8)
    scales = torch.zeros((1, 64, 4), dtype=torch.uint8)
    out = nv.alloc_requant(1, 64, 64, "cpu", nv.TARGET_MXFP8)
    out["scales"] = out["scales"][:, :1]
    with pytest.raises(ValueError, match="out scales"):
        nv.nvfp4_requant_transpose(codes, scales, torch.zeros(1), out=out)
    x = _x(1, 64, 64)
    row = nv.alloc_mx(1, 64, 64, "cpu")
    row["codes"] = row["codes"][:, :32]
    with pytest.raises(ValueError, match="row codes"):
        nv.nvfp4_mx_quantize(x, nv.Config(blocks=1), row=row)
    with pytest.raises(ValueError, match="row_amax"):
        nv.nvfp4_quantize_per_token(x[0], row_amax=torch.zeros(3))
    with pytest.raises(TypeError, match="status"):
        nv.nvfp4_amax(x, status=torch.zeros(1))
