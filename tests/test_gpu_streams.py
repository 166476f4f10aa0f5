"""Stream semantics of the C ABI. Every entry point is ordered on the stream it
is handed and makes no host-synchronous or allocating CUDA call, so a whole
step (amax, dual 4/6 encoding, 16x16 tiles, per-token encoding,
re-quantisation, MXFP8, the scale-learning forward and backward) can be
captured in a CUDA graph and replayed on new data, and independent steps on
two streams, or from two host threads, can overlap. Each case compares its
outputs, byte for byte, with the same calls run eagerly on the default
stream."""
import threading

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_02_gb300 as nv
from helpers import dev_bits
from nvfp4_block_scaled_02_gb300 import synth

pytestmark = pytest.mark.gpu

R, C = 512, 1024
NB = R * C // 16


def _alloc(dev):
    """Every output of one step, allocated once (a graph replays into them)."""
    return {
        "amax": torch.empty(1, dtype=torch.float32, device=dev),
        "row": nv.alloc_encoding(1, R, C, dev, True),
        "col": nv.alloc_encoding(1, C, R, dev, True),
        "t16_row": nv.alloc_encoding(1, R, C, dev, False),
        "t16_col": nv.alloc_encoding(1, C, R, dev, False),
        "tok": nv.alloc_encoding(R, 1, C, dev, True),
        "tok_amax": torch.empty(R, dtype=torch.float32, device=dev),
        "rq": nv.alloc_requant(1, R, C, dev, nv.TARGET_MXFP8),
        "mx_row": nv.alloc_mx(1, R, C, dev),
        "mx_col": nv.alloc_mx(1, C, R, dev),
        "fq": torch.empty((R, C), dtype=torch.bfloat16, device=dev),
        "gx": torch.empty((R, C), dtype=torch.bfloat16, device=dev),
        "gs_pre": torch.empty(NB, dtype=torch.float32, device=dev),
        "gs_post": torch.empty(NB, dtype=torch.float32, device=dev),
        "status": torch.zeros(1, dtype=torch.int32, device=dev),
    }


def _step(x, gq, s_pre, s_post, o, seed):
    st = o["status"]
    nv.nvfp4_amax(x, amax=o["amax"], status=st)
    nv.nvfp4_quantize(x, o["amax"], nv.Config(blocks=nv.BLOCKS_BOTH, four_over_six=1),
                      row=o["row"], col=o["col"], status=st)
    nv.nvfp4_quantize(x, o["amax"], nv.Config(blocks=nv.BLOCKS_TILE16, rounding=nv.ROUND_SR,
                                              seed=seed, step=1),
                      row=o["t16_row"], col=o["t16_col"], status=st)
    nv.nvfp4_quantize_per_token(x, nv.Config(four_over_six=1), out=o["tok"],
                                row_amax=o["tok_amax"], status=st)
    nv.nvfp4_requant_transpose(o["row"]["codes"], o["row"]["scales"], o["amax"],
                               src=nv.Config(four_over_six=1),
                               dst=nv.Config(rounding=nv.ROUND_SR, seed=seed, step=2),
                               target=nv.TARGET_MXFP8, out=o["rq"], status=st)
    nv.nvfp4_mx_quantize(x, nv.Config(blocks=nv.BLOCKS_BOTH, rounding=nv.ROUND_SR, seed=seed,
                                      step=3),
                         row=o["mx_row"], col=o["mx_col"], status=st)
    nv.nvfp4_fakequant_fwd(x, s_pre, s_post, out=o["fq"], status=st)
    nv.nvfp4_scale_grad_bwd(x, gq, s_pre, s_post, gx=o["gx"], gs_pre=o["gs_pre"],
                            gs_post=o["gs_post"], status=st)


def _flat(o):
    out = []
    for k in sorted(o):
        v = o[k]
        if isinstance(v, dict):
            out += [(f"{k}.{j}", v[j]) for j in sorted(v) if v[j] is not None]
        else:
            out.append((k, v))
    return out


def _same(got, want):
    for (name, a), (_, b) in zip(_flat(got), _flat(want)):
        ab = a.contiguous().view(-1).view(torch.uint8)
        bb = b.contiguous().view(-1).view(torch.uint8)
        assert torch.equal(ab, bb), f"{name}: {int((ab != bb).sum())} bytes differ"


def _inputs(seed, dev):
    x = dev_bits(synth.student_t(R, C, seed=seed)).view(torch.bfloat16)
    gq = dev_bits(synth.student_t(R, C, seed=seed + 100)).view(torch.bfloat16)
    blk = x.float().abs().view(-1, 16).amax(1)
    s_pre = (blk / 6.0).clamp_min(1e-3).contiguous()
    s_post = (s_pre * 1.03125).contiguous()
    return x, gq, s_pre, s_post


def test_whole_step_captured_in_a_cuda_graph_replays_exactly():
    dev = torch.device("cuda")
    x, gq, s_pre, s_post = _inputs(21, dev)
    o = _alloc(dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up off the capture
        _step(x, gq, s_pre, s_post, o, seed=9)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(x, gq, s_pre, s_post, o, seed=9)
    for seed in (22, 23):  # new data into the captured buffers, then replay
        nx, ngq, ns_pre, ns_post = _inputs(seed, dev)
        x.copy_(nx)
        gq.copy_(ngq)
        s_pre.copy_(ns_pre)
        s_post.copy_(ns_post)
        o["status"].zero_()
        g.replay()
        ref = _alloc(dev)
        _step(nx, ngq, ns_pre, ns_post, ref, seed=9)
        torch.cuda.synchronize()
        _same(o, ref)
        assert int(o["status"].item()) == 0


def test_independent_steps_on_two_streams():
    dev = torch.device("cuda")
    ins = [_inputs(31, dev), _inputs(32, dev)]
    outs = [_alloc(dev), _alloc(dev)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main = torch.cuda.current_stream()
    for s in streams:
        s.wait_stream(main)
    for _ in range(3):  # interleaved launches, so the two streams' kernels overlap
        for i in (0, 1):
            with torch.cuda.stream(streams[i]):
                _step(*ins[i], outs[i], seed=40 + i)
    for s in streams:
        main.wait_stream(s)
    for i in (0, 1):
        ref = _alloc(dev)
        _step(*ins[i], ref, seed=40 + i)
        torch.cuda.synchronize()
        _same(outs[i], ref)
    assert not np.array_equal(outs[0]["row"]["codes"].cpu().numpy(),
                              outs[1]["row"]["codes"].cpu().numpy())


def test_steps_from_two_host_threads():
    """The binding's foreign calls release the GIL, so two host threads enter
    the C ABI at the same time, each with its own stream."""
    dev = torch.device("cuda")
    ins = [_inputs(51, dev), _inputs(52, dev)]
    outs = [_alloc(dev), _alloc(dev)]
    torch.cuda.synchronize()
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream(device=dev)
            with torch.cuda.stream(s):
                for _ in range(4):
                    _step(*ins[i], outs[i], seed=60 + i)
            s.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in (0, 1)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in (0, 1):
        ref = _alloc(dev)
        _step(*ins[i], ref, seed=60 + i)
        torch.cuda.synchronize()
        _same(outs[i], ref)
