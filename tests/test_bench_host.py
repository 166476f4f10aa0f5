"""Host-side pieces of bench.py: the reference arm reports the same workload
text as the CUDA arm (built from the workloads' own constructor arguments)."""
import importlib.util
import os
import sys
import types

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_every_workload_has_a_description(bench):
    args = types.SimpleNamespace(experts=64, sr_steps=32)
    for c in bench.WORKLOADS:
        text = bench.describe_workload(c, args)
        assert isinstance(text, str) and len(text) > 40, c


def test_descriptions_follow_constructor_arguments(bench):
    args = types.SimpleNamespace(experts=64, sr_steps=32)
    assert bench.describe_workload(1, args).startswith("1024x1024")
    assert "8192x4096" in bench.describe_workload(2, args)
    assert "Four-Over-Six on" in bench.describe_workload(2, args)
    assert "over 32 steps" in bench.describe_workload(4, args)
    assert "64 x 2048x7168" in bench.describe_workload(5, args)
    assert "MXFP8" in bench.describe_workload(7, args)
    assert "to NVFP4" in bench.describe_workload(8, args)
    small = types.SimpleNamespace(experts=4, sr_steps=8)
    assert "4 x 2048x7168" in bench.describe_workload(5, small)
    assert "over 8 steps" in bench.describe_workload(4, small)


@pytest.mark.gpu
@pytest.mark.parametrize("config", [1, 2, 8])
def test_description_matches_the_built_workload(bench, config):
    import torch
    args = types.SimpleNamespace(experts=64, sr_steps=32)
    wl = bench.WORKLOADS[config](torch.device("cuda"))
    assert wl.workload == bench.describe_workload(config, args)
    # every call's bytes are its elements times the per-call table's figure
    bpe = wl.call_bpe(bench._wl_kw(wl))
    for kern in wl.kernels(0, 0):
        assert kern.nbytes == pytest.approx(wl.elements * bpe[kern.name], rel=1e-12)
    assert wl.bytes_per_elem == pytest.approx(sum(bpe.values()), rel=1e-12)


@pytest.mark.parametrize("config", list(range(1, 13)))
def test_reference_arm_charges_the_calls_it_runs(bench, config):
    """Each reference-arm step names the calls it ran, and those calls are
    the ones the CUDA arm's workload charges bytes for."""
    args = types.SimpleNamespace(config=config, ref_rows=32, experts=64, sr_steps=32)
    _, sample, step = bench._reference_sample(args)
    bpe = bench.WORKLOADS[config].call_bpe(bench._ctor_args(config, args))
    e, calls, dt = step(0)
    assert e > 0 and dt > 0 and calls and set(calls) <= set(bpe), (calls, bpe)
    if config == 4:  # periodic scaling: the amax runs on refresh steps only
        assert "amax" not in step(1)[1]


def test_reference_arm_counts_the_dequant(bench):
    """The activation step writes the bf16 dequant: amax (2) + x (2) + codes
    (1/2) + scales (1/16) + 4/6 bitmap (1/128) + dequant (2) bytes."""
    args = types.SimpleNamespace(config=2, ref_rows=32, experts=64, sr_steps=32)
    bpe = bench.WORKLOADS[2].call_bpe(bench._ctor_args(2, args))
    _, _, step = bench._reference_sample(args)
    calls = step(0)[1]
    assert sum(bpe[c] for c in calls) == pytest.approx(2 + 2 + 0.5 + 1 / 16 + 1 / 128 + 2)


def test_host_description(bench):
    assert bench.host_cores() >= 1
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
    t = bench.ClockSampler._when("2026/12/02 15:31:00.123")
    assert t is not None and bench.ClockSampler._when("garbage") is None


def test_default_workload_is_the_largest(bench):
    """Without --config the benchmark times the MoE dual pass (the largest
    workload that fits one GPU)."""
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert '"--config", type=int, default=5' in src
    args = types.SimpleNamespace(experts=64, sr_steps=32)
    assert "64 x 2048x7168" in bench.describe_workload(5, args)


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = importlib.util.spec_from_file_location("bench_rank", os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        sys.argv = ["bench.py"]
        spec.loader.exec_module(mod)
        mod.barrier(world)
        out[rank] = mod.max_over_ranks(1.5 + rank, world)
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_maximum_over_ranks():
    """bench.py's timing reduction on two CPU ranks (gloo): every rank gets the
    slowest rank's time."""
    import torch.multiprocessing as mp
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_sweep_candidate_count_edges(bench):
    """The MSE sweep's work count: an all-zero block encodes code 1 only; every
    count lies between 1 and 126; in a constant block the codes well below
    amax / 6 are pruned."""
    import numpy as np
    z = np.zeros((1, 16), np.uint16)
    assert bench.sweep_candidates_per_block(z, 1.0) == 1.0
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    for gam in (1e-3, 1.0, 1e3):
        n = bench.sweep_candidates_per_block(bits, gam)
        assert 1.0 <= n <= 126.0
    # A = 0.75 with g = 0.75: the codes with 6 s_c well short of A go
    v = np.full((1, 16), 0.75, np.float32)
    assert bench.sweep_candidates_per_block((v.view(np.uint32) >> 16).astype(np.uint16),
                                            2688.0 * 0.75) < 60


def test_committed_counts_match_the_sources(bench):
    """Every instruction count and traffic figure under profiles/ was taken
    from the sources the kernels are built from now (a kernel changed since
    its capture would report no issue or traffic figure)."""
    import json
    for fname in ("inst.json", "traffic.json"):
        with open(os.path.join(ROOT, "profiles", fname)) as f:
            d = json.load(f)
        for cfg, kernels in d["workloads"].items():
            for kernel, e in kernels.items():
                assert e["source_sha"] == bench.kernel_source_hash(kernel), (fname, cfg, kernel)


def test_link_bound_takes_the_slowest_copy_arrangement(bench):
    """The end-to-end ceiling: the larger one-way copy, or both copies at the
    rate the two directions reach together, whichever takes longer (the MoE
    step's 1.9 GB in and 4.8 GB out on a 211 / 193 GB/s link)."""
    bi, bo, step = 1879048192, 4829741056, 8.592e9
    duplex = {"copy_in_gbs": 211.2, "copy_out_gbs": 193.4, "copy_both_gbs": 342.0}
    half = dict(duplex, copy_both_gbs=255.3)
    # full duplex: the copy-out alone sets the step (24.97 ms)
    assert abs(bench.link_bound_gbs(step, bi, bo, duplex) - step / (bo / 193.4e9) / 1e9) < 1e-6
    # both directions at 255.3 GB/s together: 26.28 ms, longer than the copy-out alone
    want = step / ((bi + bo) / 255.3e9) / 1e9
    assert abs(bench.link_bound_gbs(step, bi, bo, half) - want) < 1e-6
    assert bench.link_bound_gbs(step, bi, bo, half) < bench.link_bound_gbs(step, bi, bo, duplex)
