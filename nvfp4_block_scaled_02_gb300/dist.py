"""Multi-GPU use of the quantiser.

Every 16-value block is encoded independently, so a tensor split across ranks
(rows, experts or slices) needs no exchange except one: under current
per-tensor scaling the FP32 outer scale depends on the amax of the WHOLE
tensor. Each rank runs nvfp4_amax on its shard and the per-slice results are
combined with an all-reduce MAX before nvfp4_quantize. MAX is exact and
independent of order, so every rank gets the same bits as a single-GPU run on
the unsplit tensor. Periodic scaling does this only on refresh steps; per-expert
or per-token outer scales need no exchange at all.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def allreduce_amax_(amax: torch.Tensor, group=None) -> torch.Tensor:
    """In-place MAX all-reduce of a per-slice amax vector (fp32, >= 0)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(amax, op=dist.ReduceOp.MAX, group=group)
    return amax


def sharded_global_amax(x_shard: torch.Tensor, group=None, amax_fn=None) -> torch.Tensor:
    """Global amax of a tensor whose rows are split across the ranks of
    `group`: the local amax of this rank's shard, then MAX over ranks.
    `amax_fn(x) -> fp32 [slices]` computes the local part (nvfp4_amax on a GPU)."""
    if amax_fn is None:
        from . import nvfp4_amax as amax_fn
    return allreduce_amax_(amax_fn(x_shard), group)


def shard_rows(rows: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of this rank's rows; boundaries on multiples of 16 so that
    column (16x1) blocks never straddle two ranks."""
    blocks = (rows + 15) // 16
    per, extra = divmod(blocks, world)
    start = (rank * per + min(rank, extra)) * 16
    stop = min(rows, start + (per + (1 if rank < extra else 0)) * 16)
    return start, stop
