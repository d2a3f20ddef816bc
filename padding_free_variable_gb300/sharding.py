"""Host-side logic for running the packed LSTM on several ranks.

Sequences are independent through the whole layer stack, so a batch can be
split by sequence: each rank builds its own plan (its own length sort and
step tables) over its share and runs the unchanged kernels.  The split
balances the recurrent work, which is proportional to sequence length:
"Multi-Lane Capsule Networks", Sec. IV, assigns independent lanes to GPUs
with a greedy number partition (largest remaining item into the least
loaded bin); here the items are sequences and their cost is their length.

Every run in this repository has one GPU, so nothing here launches work on
several devices; ``timing_over_ranks`` is what bench.py uses to combine the
per-rank times of independent replicas.
"""
from __future__ import annotations

import numpy as np


def lpt_partition(lengths, world: int):
    """Greedy longest-first partition of sequence indices into `world` shares.

    Sequences are taken in decreasing length (ties: lower index first) and each
    goes to the share with the smallest total length so far (ties: lower rank).
    Returns a list of `world` index arrays, each in ascending index order.
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    if world < 1:
        raise ValueError("world must be >= 1")
    order = sorted(range(len(lengths)), key=lambda i: (-int(lengths[i]), i))
    load = [0] * world
    shares = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        shares[r].append(i)
        load[r] += int(lengths[i])
    return [np.array(sorted(s), dtype=np.int64) for s in shares]


def shard_rows(lengths, share):
    """Rows of the caller-order frame matrix that belong to the sequences in `share`."""
    lengths = np.asarray(lengths, dtype=np.int64)
    start = np.concatenate([[0], np.cumsum(lengths)])
    if len(share) == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(start[i], start[i + 1]) for i in share])


def timing_over_ranks(local_ms: float, local_frames: int, steps: int, dist=None):
    """Whole-job throughput of independent ranks: frames summed over ranks, time = slowest rank.

    Returns (frames_per_second, max_ms).  `dist` is torch.distributed (or None for one rank).
    """
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return local_frames * steps / (local_ms / 1e3), local_ms
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(local_ms), float(local_frames)], dtype=torch.float64, device=dev)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    sm = t.clone()
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    max_ms, frames = float(mx[0].item()), float(sm[1].item())
    return frames * steps / (max_ms / 1e3), max_ms
