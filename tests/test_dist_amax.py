"""Sharded global amax on CPU ranks (gloo, world size 2): each rank takes its
row shard, computes the local per-slice amax, and the MAX all-reduce must give
every rank exactly the amax of the whole tensor; the quantisation of a shard
with that amax then equals the same rows of the single-process quantisation."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from nvfp4_block_scaled_02_gb300 import dist as nvdist
from nvfp4_block_scaled_02_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = synth.moe_experts(3, 80, 64, seed=4)  # [S=3, R=80, C=64]
        r0, r1 = nvdist.shard_rows(80, rank, world)
        shard = np.ascontiguousarray(x[:, r0:r1])

        def local_amax(t):
            a, _ = oracle.global_amax(t.numpy().view(np.uint16), t.shape[0])
            return torch.from_numpy(a.copy())

        g = nvdist.sharded_global_amax(torch.from_numpy(shard.view(np.int16)), amax_fn=local_amax)
        full, _ = oracle.global_amax(x, 3)
        q_shard = oracle.quantize(shard, g.numpy(), four_over_six=1)
        q_full = oracle.quantize(x, full, four_over_six=1)
        ok = bool(np.array_equal(g.numpy().view(np.uint32), full.view(np.uint32)))
        ok &= bool(np.array_equal(q_shard["row_codes"], q_full["row_codes"][:, r0:r1]))
        ok &= bool(np.array_equal(q_shard["row_dq"], q_full["row_dq"][:, r0:r1]))
        out[rank] = 1 if ok else 0
    finally:
        dist.destroy_process_group()


def test_sharded_amax_is_exact_on_two_cpu_ranks():
    world = 2
    out = mp.get_context("spawn").Array("i", [0] * world)
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn")
    assert list(out) == [1, 1]


def test_shard_rows_cover_and_align():
    for rows in (16, 80, 2048, 48):
        for world in (1, 2, 3, 8):
            spans = [nvdist.shard_rows(rows, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == rows
            for (a, b), (c, d) in zip(spans, spans[1:]):
                assert b == c
            assert all(a % 16 == 0 for a, _ in spans)
