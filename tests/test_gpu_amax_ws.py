"""The one-launch global amax (nvfp4_amax_ws, End-to-End 4-Bit Training,
"Low-precision formats on Blackwell": the FP32 outer scale per tensor or
expert) against the oracle and against nvfp4_amax, bit for bit, with the
workspace back at zero after every call."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


@pytest.mark.parametrize("S,R,C", [(1, 37, 41), (3, 64, 100), (5, 1, 8), (4, 2048, 7168),
                                   (2, 0, 16)])
def test_amax_ws_matches_oracle(orc, S, R, C):
    xb = synth.student_t(max(S * R, 1), C, seed=21)[:S * R].reshape(S, R, C)
    x = _dev(xb) if S * R * C else torch.empty((S, R, C), dtype=torch.int16, device="cuda")
    ws = nv.amax_workspace(S, "cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    want, _ = orc.global_amax(xb, S) if S * R * C else (np.zeros(S, np.float32), 0)
    for _ in range(2):  # a second call finds the workspace as the first left it
        got = nv.nvfp4_amax_ws(x, ws, status=st)
        torch.cuda.synchronize()
        assert np.array_equal(got.cpu().numpy().view(np.uint32),
                              np.asarray(want, np.float32).view(np.uint32))
        assert int(ws.abs().sum().item()) == 0
    assert int(st.item()) == 0
    if S * R * C:
        assert torch.equal(got, nv.nvfp4_amax(x))


def test_amax_ws_many_slices(orc):
    """More slices than one launch's grid can hold in y (65535)."""
    S, R, C = 65537, 1, 16
    xb = synth.student_t(S, C, seed=22).reshape(S, R, C)
    ws = nv.amax_workspace(S, "cuda")
    got = nv.nvfp4_amax_ws(_dev(xb), ws)
    want, _ = orc.global_amax(xb, S)
    assert np.array_equal(got.cpu().numpy(), want)
    assert int(ws.abs().sum().item()) == 0


def test_amax_ws_flags_non_finite(orc):
    xb = synth.student_t(64, 96, seed=23).reshape(2, 32, 96)
    xb[1, 5, 7] = 0x7F80  # +Inf in slice 1
    ws = nv.amax_workspace(2, "cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = nv.nvfp4_amax_ws(_dev(xb), ws, status=st)
    want, ost = orc.global_amax(xb, 2)
    assert int(st.item()) == nv.DEV_NONFINITE_INPUT == ost
    assert np.array_equal(got.cpu().numpy(), want)
    assert int(ws.abs().sum().item()) == 0
