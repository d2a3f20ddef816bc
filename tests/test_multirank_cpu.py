"""Multi-rank host logic on CPU with two gloo ranks (no GPU).

* lpt_partition covers every sequence exactly once and balances length;
* sequence shards, each run through the oracle on its own rank, give the
  unsharded batch's outputs, and their parameter gradients summed across the
  ranks (the one exchange step of data-parallel training) equal the
  unsharded gradients;
* timing_over_ranks combines per-rank times as bench.py reports them:
  frames summed over ranks, time of the slowest rank.
"""
import os
import socket

import numpy as np
import pytest

from padding_free_variable_gb300 import sharding, synthetic


def test_lpt_partition_covers_and_balances():
    rng = np.random.default_rng(0)
    lengths = rng.integers(1, 1000, 128)
    for world in (1, 2, 3, 4, 8):
        shares = sharding.lpt_partition(lengths, world)
        got = np.sort(np.concatenate(shares))
        assert np.array_equal(got, np.arange(len(lengths)))
        loads = [int(lengths[s].sum()) for s in shares]
        # greedy longest-first: no share exceeds another by more than the longest sequence
        assert max(loads) - min(loads) <= int(lengths.max())
    # hand case: lengths 5 4 3 3 -> shares {5, 3} and {4, 3}
    shares = sharding.lpt_partition([5, 4, 3, 3], 2)
    assert [list(s) for s in shares] == [[0, 3], [1, 2]]


def test_shard_rows():
    rows = sharding.shard_rows([2, 0, 3], [0, 2])
    assert list(rows) == [0, 1, 2, 3, 4]
    assert list(sharding.shard_rows([2, 0, 3], [2])) == [2, 3, 4]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        w = synthetic.custom(2, 2, 6, 5, [9, 3, 0, 7, 7, 1, 12, 4], seed=21)
        share = sharding.lpt_partition(w.lengths, world)[rank]
        rows = sharding.shard_rows(w.lengths, share)
        res = oracle.lstm_stack(w.lengths[share], w.x[rows], w.layers, 2, 5, G=w.G[rows])
        flat = np.concatenate([res["grads"][l][k].ravel() for l in range(2) for k in ("W", "R", "b", "peep")])
        t = torch.from_numpy(flat.copy())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        fps, max_ms = sharding.timing_over_ranks(10.0 + rank, 100 * (rank + 1), 5, dist)
        out[rank] = {"share": share, "y": res["y"], "dx": res["dx"], "grads": t.numpy(),
                     "fps": fps, "max_ms": max_ms}
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_unsharded_batch():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    import oracle
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    w = synthetic.custom(2, 2, 6, 5, [9, 3, 0, 7, 7, 1, 12, 4], seed=21)
    full = oracle.lstm_stack(w.lengths, w.x, w.layers, 2, 5, G=w.G)
    flat = np.concatenate([full["grads"][l][k].ravel() for l in range(2) for k in ("W", "R", "b", "peep")])
    for r in range(world):
        np.testing.assert_allclose(res[r]["grads"], flat, rtol=1e-12, atol=1e-14)
        rows = sharding.shard_rows(w.lengths, res[r]["share"])
        np.testing.assert_allclose(res[r]["y"], full["y"][rows], rtol=1e-13)
        np.testing.assert_allclose(res[r]["dx"], full["dx"][rows], rtol=1e-12, atol=1e-14)
        # frames 100 + 200 per step over the slowest rank's 11 ms, 5 steps
        assert res[r]["max_ms"] == 11.0
        assert res[r]["fps"] == pytest.approx(300 * 5 / 0.011)
