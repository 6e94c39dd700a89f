"""The batch-sharded data-parallel step on CPU ranks (gloo, world size 2; no GPU).

Each rank takes its block of batch elements (``shard.shard_rows``), computes the
forward and both gradients of its local problem (here with the oracle, standing
in for the GPU library), and the ranks sum their weight and bias gradients in
rank order through ``shard.ordered_sum_over_ranks``.  The result must equal the
single-rank oracle on the whole batch: rows of out and dX exactly, dW and db to
fp64 rounding, and every rank must hold the same dW/db bits.
"""
import os
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GRID = (4, 9, 7, 8)  # four batch elements, anisotropic extents


def _problem(B):
    sys.path.insert(0, ROOT)
    from voxel_gemm_gb300 import synth
    grid = (B,) + GRID[1:]
    coords = synth.random_coords(31 + B, 700, *grid)
    rng = np.random.default_rng(5 + B)
    f = rng.standard_normal((coords.shape[0], 3))
    W = rng.standard_normal((27, 3, 5))
    b = rng.standard_normal(5)
    dY = rng.standard_normal((coords.shape[0], 5))
    return coords, grid, f, W, b, dY


def _rank(rank, world, B, port, q):
    sys.path.insert(0, ROOT)
    import torch
    import oracle
    from voxel_gemm_gb300 import shard
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        coords, grid, f, W, b, dY = _problem(B)
        rows, local, lb = shard.shard_rows(coords, B, rank, world)
        nbr, _ = oracle.nbrmap(local, lb, *grid[1:]) if lb > 0 else (np.zeros((0, 27), np.uint32), None)
        out = oracle.fwd(nbr, f[rows], W, b)
        dX = oracle.dgrad_scatter(nbr, dY[rows], W)
        dW, db = oracle.wgrad(nbr, f[rows], dY[rows])

        def in_rank_order(parts):  # the test's own fixed-order sum (fp64)
            acc = parts[0].clone()
            for p in range(1, parts.shape[0]):
                acc += parts[p]
            return acc

        dW_sum = shard.ordered_sum_over_ranks(torch.from_numpy(dW), world, in_rank_order)
        db_sum = shard.ordered_sum_over_ranks(torch.from_numpy(db), world, in_rank_order)
        q.put((rank, rows, out, dX, dW_sum.numpy(), db_sum.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(B, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29700 + (os.getpid() + B) % 1000
    procs = [ctx.Process(target=_rank, args=(r, world, B, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, *res = q.get(timeout=180)
        got[r] = res
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("B", [4, 3])
def test_sharded_step_matches_single_rank_oracle(B):
    sys.path.insert(0, ROOT)
    import oracle
    coords, grid, f, W, b, dY = _problem(B)
    nbr, _ = oracle.nbrmap(coords, *grid)
    out_ref = oracle.fwd(nbr, f, W, b)
    dX_ref = oracle.dgrad_scatter(nbr, dY, W)
    dW_ref, db_ref = oracle.wgrad(nbr, f, dY)
    got = _run(B)
    seen = np.concatenate([got[r][0] for r in sorted(got)])
    assert np.array_equal(np.sort(seen), np.arange(coords.shape[0]))  # the ranks partition the rows
    for r, (rows, out, dX, dW, db) in got.items():
        assert _rel(out, out_ref[rows]) < 1e-14, r
        assert _rel(dX, dX_ref[rows]) < 1e-14, r
        assert _rel(dW, dW_ref) < 1e-12 and _rel(db, db_ref) < 1e-12, r
    # the rank-ordered sum leaves the same bits on every rank
    assert np.array_equal(got[0][3], got[1][3]) and np.array_equal(got[0][4], got[1][4])


def test_batch_range_partitions_the_batch():
    sys.path.insert(0, ROOT)
    from voxel_gemm_gb300 import shard
    for B in range(0, 9):
        for world in range(1, 5):
            blocks = [shard.batch_range(B, r, world) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == B
            assert all(blocks[i][1] == blocks[i + 1][0] for i in range(world - 1))
    with pytest.raises(ValueError):
        shard.batch_range(4, 2, 2)
