"""Multi-rank host logic on CPU: two gloo ranks, each owning its shard of units.

The decode path shards into independent (layer, batch, KV head) units (HashEvict
paper, technical framework: every step is per head and per sequence), so a
rank's results must not depend on which other units exist or where they run.
Each rank runs the oracle on its shard of a small workload; the gathered
results must equal a one-process run over every unit, the shards must
partition the units, and max_over_ranks must return the slowest rank's time.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import synth
from lsh_pre_attention_decode_b300.shard import batch_shard, layer_shard, max_over_ranks
from tests.gpu_harness import run_oracle_unit

WORKLOAD = synth.WORKLOADS["llama8b_b8"].with_(batch=3, budget=40, kv_heads=2, heads=8)
STEPS = 6


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _unit_result(layer: int, b: int, j: int):
    r = run_oracle_unit(WORKLOAD, b, j, WORKLOAD.budget, STEPS, out_steps=range(STEPS),
                        layer=layer)
    return r.evicted.copy(), np.asarray(r.outs).copy()


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = {}
        for layer in layer_shard(rank, world, 1):
            for b in batch_shard(rank, world, WORKLOAD.batch):
                for j in range(WORKLOAD.kv_heads):
                    mine[(layer, b, j)] = _unit_result(layer, b, j)
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        slowest = max_over_ranks(10.0 + rank)
        if rank == 0:
            q.put((gathered, slowest))
    finally:
        dist.destroy_process_group()


def test_shard_partitions():
    for world in (1, 2, 3, 8):
        rows = [r for k in range(world) for r in batch_shard(k, world, 13)]
        assert rows == list(range(13))
        layers = [x for k in range(world) for x in layer_shard(k, world, 4)]
        assert layers == list(range(4 * world))
    with pytest.raises(ValueError):
        layer_shard(2, 2, 1)
    with pytest.raises(ValueError):
        batch_shard(0, 0, 4)
    assert max_over_ranks(3.5) == 3.5  # no process group: identity


def test_two_gloo_ranks_match_one_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    gathered, slowest = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert slowest == 11.0
    keys = [set(g) for g in gathered]
    assert not (keys[0] & keys[1])
    # rank r owns layer r and its batch rows; every (layer, b, j) of its shard appears once
    for r in range(2):
        want = {(r, b, j) for b in batch_shard(r, 2, WORKLOAD.batch)
                for j in range(WORKLOAD.kv_heads)}
        assert keys[r] == want
    for g in gathered:
        for (layer, b, j), (ev, outs) in g.items():
            ev1, outs1 = _unit_result(layer, b, j)
            assert np.array_equal(ev, ev1)
            assert np.array_equal(outs, outs1)
