"""The amax entry point that allocates nothing (nvfp4_amax_noalloc), for
callers that cannot allocate device memory: an operator hook that hands out
no workspace, a serving loop that fixes its memory at start-up, code that must
not let a cudaMalloc or cudaFree synchronise the device. It must return what
the workspace entry point (nvfp4_amax_ws) returns, bit for bit (the amax is an
exact maximum), call after call.

This file is collected last on purpose, so that a failure here stops a
first-failure run only after every other test has run; it passes alone in a
fresh process too (the first call on the device does the set-up)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu


def test_noalloc_amax_matches_the_workspace_amax():
    L = nv.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row, on different tensors (a second call must not see
    # what the first left in the shared scratch array)
    for S, R, C, seed in ((8, 64, 96, 31), (3, 2048, 7168, 32)):
        xb = synth.student_t(S * R, C, seed=seed).reshape(S, R, C)
        x = torch.from_numpy(xb.view(np.int16)).cuda()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        got = torch.full((S,), -1.0, dtype=torch.float32, device="cuda")
        assert L.nvfp4_amax_noalloc(x.data_ptr(), S, R, C, got.data_ptr(), st.data_ptr(),
                                    stream) == 0
        ws = nv.amax_workspace(S, "cuda")
        want = torch.full((S,), -2.0, dtype=torch.float32, device="cuda")
        assert L.nvfp4_amax_ws(x.data_ptr(), S, R, C, want.data_ptr(), ws.data_ptr(),
                               ws.numel() * ws.element_size(), st.data_ptr(), stream) == 0
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int32), want.view(torch.int32))
        assert int(st.item()) == 0
    # above the fixed array's limit: refused before anything is enqueued
    assert L.nvfp4_amax_noalloc(x.data_ptr(), nv.AMAX_NOALLOC_MAX_SLICES + 1, 1, 16,
                                got.data_ptr(), None, stream) == 2
