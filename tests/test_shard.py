"""The multi-GPU split (one process per GPU): host logic only, on CPU.

The forward has no exchange step, so what a multi-rank run adds is the split
of the packed batch along sequence boundaries and the two host-side
reductions of a measurement (slowest rank's time, summed work).  The gloo
test runs them in two real processes with world_size 2.
"""
import os
import socket

import numpy as np
import pytest

from transformer_encoder_forward_gb300 import shard, synth


def _brute_pairs(n, w):
    return sum(1 for i in range(n) for j in range(n) if w == 0 or abs(i - j) <= w)


@pytest.mark.parametrize("n,w", [(1, 0), (1, 5), (7, 0), (7, 2), (7, 6), (7, 9), (40, 3), (130, 64)])
def test_visible_pairs_match_brute_force(n, w):
    assert shard.visible_pairs_one(n, w) == _brute_pairs(n, w)


def test_sequence_costs_add_up_to_the_forward_flops():
    # per-sequence costs must sum to the whole batch's flops, counted the
    # plain way: GEMM 2*T*params per layer, attention 4*hd*H*pairs per layer
    cfg = synth.CONFIGS["c2"]
    lens = synth.draw_lens(cfg)
    T = int(lens[:6].sum())
    params = (cfg.d * (cfg.heads + 2 * cfg.kv_heads) * cfg.hd + cfg.heads * cfg.hd * cfg.d
              + cfg.d * cfg.ffn * 2 + cfg.ffn * cfg.d)
    per_window = {w: sum(_brute_pairs(int(n), w) for n in lens[:6])
                  for w in {cfg.window_of(i) for i in range(cfg.layers)}}
    pairs = [per_window[cfg.window_of(i)] for i in range(cfg.layers)]
    want = 2 * T * params * cfg.layers + 4 * cfg.hd * cfg.heads * sum(pairs)
    assert shard.sequence_costs(cfg, lens[:6]).sum() == pytest.approx(want, rel=1e-12)


def test_partition_covers_every_sequence_once_and_balances():
    rng = np.random.default_rng(5)
    for world in (1, 2, 3, 4, 8):
        costs = rng.uniform(1.0, 100.0, 61)
        parts = shard.partition(costs, world)
        assert len(parts) == world
        allidx = np.concatenate(parts)
        assert sorted(allidx.tolist()) == list(range(61))
        for p in parts:
            assert np.all(np.diff(p) > 0)            # ascending, packing keeps order
        loads = [costs[p].sum() for p in parts]
        # greedy LPT bound: no share exceeds the mean by more than the largest item
        assert max(loads) <= costs.sum() / world + costs.max() + 1e-9


def test_partition_one_rank_is_the_identity_and_is_deterministic():
    costs = [3.0, 1.0, 3.0, 2.0]
    assert shard.partition(costs, 1)[0].tolist() == [0, 1, 2, 3]
    a = shard.partition(costs, 2)
    b = shard.partition(list(costs), 2)
    assert [x.tolist() for x in a] == [x.tolist() for x in b]
    # equal costs: ties go by index, lowest rank first
    assert [x.tolist() for x in shard.partition([1.0] * 4, 2)] == [[0, 2], [1, 3]]


def test_partition_with_fewer_sequences_than_ranks_leaves_empty_shares():
    parts = shard.partition([5.0, 1.0], 4)
    assert [p.tolist() for p in parts] == [[0], [1], [], []]
    with pytest.raises(ValueError):
        shard.partition([1.0], 0)


def test_global_batch_starts_with_the_one_gpu_batch():
    cfg = synth.CONFIGS["c2"]
    draw = lambda c, r: synth.draw_lens(c, synth.BASE_SEED + r)
    one = shard.global_lens(cfg, 1, draw)
    assert one.tolist() == synth.draw_lens(cfg).tolist() and int(one.sum()) == 16238
    four = shard.global_lens(cfg, 4, draw)
    assert len(four) == 4 * cfg.n_seqs and four[: cfg.n_seqs].tolist() == one.tolist()
    parts = shard.partition(shard.sequence_costs(cfg, four), 4)
    loads = [shard.sequence_costs(cfg, four[p]).sum() for p in parts]
    assert max(loads) / min(loads) < 1.05           # weak scaling: about one batch per rank


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = synth.CONFIGS["c2"]
        allv = shard.global_lens(cfg, world, lambda c, r: synth.draw_lens(c, synth.BASE_SEED + r))
        mine = shard.partition(shard.sequence_costs(cfg, allv), world)[rank]
        got = [None] * world
        dist.all_gather_object(got, mine.tolist())
        t_ms = 10.0 + 5.0 * rank                      # a per-rank "step time"
        work = float(shard.sequence_costs(cfg, allv[mine]).sum())
        res = {"plans": got, "max_ms": shard.max_over_ranks(t_ms, dist),
               "sum_work": shard.sum_over_ranks(work, dist), "n": len(allv),
               "total": float(shard.sequence_costs(cfg, allv).sum())}
        np.save(os.path.join(out_dir, f"r{rank}.npy"), np.array([res], dtype=object))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_the_batch_and_reduce_the_timing(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [np.load(tmp_path / f"r{r}.npy", allow_pickle=True)[0] for r in range(world)]
    plans = res[0]["plans"]
    assert res[1]["plans"] == plans                   # every rank sees the same plan
    flat = sorted(i for p in plans for i in p)
    assert flat == list(range(res[0]["n"]))           # disjoint, and covers the batch
    for r in res:
        assert r["max_ms"] == 15.0                    # the slowest rank's time
        assert r["sum_work"] == pytest.approx(r["total"], rel=1e-12)
