"""The data-parallel path across ranks, on CPU: the sharding plan, the slicing and merge
of a packed batch, and a two-rank gloo run in which each rank computes its own
sequences (float64 oracle standing in for the GPU layer) and the merged result equals
the single-process result bit for bit -- the split needs no data-path exchange."""
import os
import socket

import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from gated_deltanet_linear_05_gb300 import shard


def test_plan_covers_every_sequence_once_and_balances_tokens():
    lengths = [5577, 6806, 8032, 5712, 3790, 7512, 7600, 7900]
    for world in (1, 2, 3, 4, 8):
        owned = shard.plan(lengths, world)
        flat = sorted(n for o in owned for n in o)
        assert flat == list(range(len(lengths)))
        loads = [sum(lengths[n] for n in o) for o in owned]
        # greedy longest-first: the spread is at most the longest sequence
        assert max(loads) - min(loads) <= max(lengths)
    assert shard.plan([3, 0, 7], 5)[0] == [2]


def test_slice_and_merge_round_trip():
    wl = gi.Workload("s", [40, 0, 17, 64, 5], 1, 2, chunk=16, dtype="f32", s0_scale=0.1)
    x = gi.make_inputs(wl, seed=3)
    owned = shard.plan(wl.lengths, 3)
    parts = [shard.slice_inputs(x, seqs) for seqs in owned]
    for seqs, pt in zip(owned, parts):
        assert int(pt["cu_seqlens"][-1]) == sum(wl.lengths[n] for n in seqs)
        assert pt["state0"].shape[0] == len(seqs)
    o, s = shard.merge(x["cu_seqlens"], owned, [pt["v"] for pt in parts],
                       [pt["state0"] for pt in parts])
    assert np.array_equal(o, x["v"]) and np.array_equal(s, x["state0"])


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = gi.Workload("dp", [70, 33, 129, 16, 90], 2, 4, chunk=64, dtype="bf16", s0_scale=0.1)
        x = gi.make_inputs(wl, seed=17)
        owned = shard.plan(wl.lengths, world)
        mine = shard.slice_inputs(x, owned[rank])
        o, s = oracle.recurrent(mine["q"], mine["k"], mine["v"], mine["g"], mine["beta"],
                                mine["state0"], mine["cu_seqlens"], threads=1)
        gathered = [None] * world
        dist.all_gather_object(gathered, (o, s))
        slowest = shard.max_over_ranks(float(rank + 1))
        if rank == 0:
            o_m, s_m = shard.merge(x["cu_seqlens"], owned, [g_[0] for g_ in gathered],
                                   [g_[1] for g_ in gathered])
            o_ref, s_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                            x["state0"], x["cu_seqlens"], threads=1)
            queue.put((bool(np.array_equal(o_m, o_ref) and np.array_equal(s_m, s_ref)),
                       slowest))
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_split_equals_single_process():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    codes = [p.exitcode for p in procs]
    assert codes == [0, 0], codes
    exact, slowest = queue.get(timeout=5)
    assert exact
    assert slowest == 2.0
