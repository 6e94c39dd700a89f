"""Batch-sharded data-parallel step: one process per GPU, weights replicated.

The pages describe a single-GPU operator library ("Contribution Tasks —
JeffreyXiang/FlexGEMM", §一); across GPUs the convolution shards by batch
element with no halo, because the neighbour map never links two batch
elements.  Each rank builds the map of its own batch elements, runs the
forward and both gradients locally through the C ABI, and the ranks then sum
their weight and bias gradients in rank order (an all-gather followed by
``vg_sum_ordered``), so every rank holds the same bits, run after run.

Only the bookkeeping lives here (which rows and batch elements a rank owns,
how their batch indices are relabelled, the rank-ordered exchange); all
arithmetic of the step runs in the library's kernels.  The exchange takes the
summing function as an argument so that the same code runs on CPU ranks
(``gloo``) in the tests.
"""
from __future__ import annotations

from typing import Callable, Tuple

import numpy as np


def batch_range(B: int, rank: int, world: int) -> Tuple[int, int]:
    """The contiguous block [b0, b1) of the B batch elements that `rank` owns."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return rank * B // world, (rank + 1) * B // world


def shard_rows(coords: np.ndarray, B: int, rank: int, world: int):
    """Rows of a global (b,x,y,z) coordinate list owned by `rank`, and their local coordinates.

    Returns (rows, local_coords, local_B): ``rows`` index the global rows (in
    their global order), ``local_coords`` has the batch index shifted so the
    rank's first batch element is 0.  A voxel's neighbours are in its own batch
    element, so the local neighbour map is the global one restricted to ``rows``
    and renumbered."""
    b0, b1 = batch_range(B, rank, world)
    b = coords[:, 0]
    rows = np.nonzero((b >= b0) & (b < b1))[0]
    local = coords[rows].copy()
    local[:, 0] -= b0
    return rows, local, b1 - b0


def rank_coords(wl, rank: int) -> np.ndarray:
    """Coordinates of rank `rank`'s own batch element(s) in the weak-scaling
    benchmark: every rank holds a batch of the workload's shape (the global
    batch is world x wl.B); the geometry is the workload's, the features differ."""
    from . import synth
    return synth.make_coords(wl)


def ordered_sum_over_ranks(local, world: int, sum_fn: Callable, group=None):
    """All-gather `local` (a tensor of the same shape on every rank) into
    [world, *local.shape] and return sum_fn(parts), which must add the parts in
    index (= rank) order."""
    import torch
    import torch.distributed as dist
    flat = torch.empty(world * local.numel(), dtype=local.dtype, device=local.device)
    dist.all_gather_into_tensor(flat, local.contiguous().view(-1), group=group)
    return sum_fn(flat.view((world,) + tuple(local.shape)))


class GradientSum:
    """The exchange step of the data-parallel training step on GPU ranks: dW and db
    replaced in place by their rank-ordered sums over all ranks (NCCL all-gather,
    then the library's vg_sum_ordered kernel)."""

    launches = 2  # vg_sum_ordered for dW and for db

    def __init__(self, world: int, dW, db, device):
        import torch
        self.world = world
        self.dW, self.db = dW, db
        # flat [world * numel] buffers viewed as [world, *shape] (the layout every
        # backend's all-gather accepts)
        self.pW = torch.empty(world * dW.numel(), dtype=dW.dtype, device=device).view((world,) + tuple(dW.shape))
        self.pb = torch.empty(world * db.numel(), dtype=db.dtype, device=device).view((world,) + tuple(db.shape))

    def __call__(self, stream):
        import torch
        import torch.distributed as dist
        from . import ops
        with torch.cuda.stream(stream):
            dist.all_gather_into_tensor(self.pW.view(-1), self.dW.view(-1))
            dist.all_gather_into_tensor(self.pb.view(-1), self.db.view(-1))
            ops.vg_sum_ordered(self.pW, self.dW, stream=stream)
            ops.vg_sum_ordered(self.pb, self.db, stream=stream)
