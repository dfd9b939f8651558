"""Data-parallel split of a packed batch across GPUs, one process per GPU.

Every step of the block works on one row at a time except attention, and
attention only looks at keys of the query's own sequence ("cortiq-engine
0.8.39 src/gpu_metal/egemma2.rs", att_plan: per-sequence spans in the packed
rows).  A packed batch therefore splits along sequence boundaries into
independent shares: a rank needs no row of another rank, weights are
replicated, and the forward has no exchange step.  The only collectives are
on the host side of a measurement (the slowest rank's time, the summed work).

The split balances the forward's work, not the row count: a sequence of
length n costs c_lin * n (the projections, per row) plus c_attn * pairs(n)
(the attention, per visible (query, key) pair, windowed layers counted with
their window).  Shares are built by longest-processing-time-first greedy
assignment, which keeps the largest share within max(cost) of the mean.
"""
from __future__ import annotations

import numpy as np


def visible_pairs_one(n: int, window: int) -> int:
    """(query, key) pairs attention computes inside one sequence of length n:
    all n*n without a window, else those with |i - j| <= window."""
    n = int(n)
    if window == 0 or window >= n - 1:
        return n * n
    i = np.arange(n)
    return int(np.sum(np.minimum(n - 1, i + window) - np.maximum(0, i - window) + 1))


def sequence_costs(cfg, lens) -> np.ndarray:
    """Forward flops of each sequence of the batch over all layers of cfg."""
    d, hd, H, KV, F = cfg.d, cfg.hd, cfg.heads, cfg.kv_heads, cfg.ffn
    c_lin = 2 * cfg.layers * (d * (H + 2 * KV) * hd + H * hd * d
                              + d * F * (2 if cfg.gated else 1) + F * d
                              + 3 * d * getattr(cfg, "ple_dim", 0))
    windows = [cfg.window_of(i) for i in range(cfg.layers)]
    out = np.empty(len(lens), dtype=np.float64)
    for s, n in enumerate(lens):
        pairs = sum(visible_pairs_one(n, w) for w in windows)
        out[s] = c_lin * int(n) + 4 * hd * H * pairs
    return out


def partition(costs, world: int) -> list[np.ndarray]:
    """Split sequence indices into `world` shares of near-equal total cost.

    Deterministic (every rank computes the same plan): sequences are taken in
    order of decreasing cost (ties by index) and each goes to the share with
    the least cost so far (ties to the lowest rank).  Each share lists its
    sequences in ascending index order, so packing keeps their relative order.
    A share may be empty when there are fewer sequences than ranks."""
    if world < 1:
        raise ValueError("world must be >= 1")
    costs = np.asarray(costs, dtype=np.float64)
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    load = [0.0] * world
    shares: list[list[int]] = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda k: (load[k], k))
        shares[r].append(i)
        load[r] += float(costs[i])
    return [np.asarray(sorted(s), dtype=np.int64) for s in shares]


def global_lens(cfg, world: int, draw) -> np.ndarray:
    """The packed batch of a weak-scaling run on `world` GPUs: `world` draws of
    one GPU's batch, the first with the base seed (so one GPU runs exactly the
    single-GPU workload) and draw r with seed offset r."""
    return np.concatenate([draw(cfg, r) for r in range(world)]).astype(np.int32)


def max_over_ranks(value: float, dist) -> float:
    """The largest `value` over all ranks (the slowest rank's time)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist) -> float:
    """The sum of `value` over all ranks (the work all ranks did)."""
    import torch
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())
