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
