"""Multi-rank host logic on CPU (gloo, world size 2).

The hot path shards by request with no exchange step: each rank owns its own
sequences and KV caches ("Hosting Qwen on Blackwell", section "Decoders":
decoders use data parallelism, each device keeps its own KV caches and
requests). These tests cover what runs on the host for N > 1: the
max-over-ranks timing reduction, the per-rank seeds, and that splitting one
batch over ranks and concatenating the shards' results reproduces the
unsharded result exactly (computed here with the float64 oracle).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from gqa_attention_softmax_gb300 import runner, workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # timing reduction: every rank sees the slowest rank's time
        assert runner.max_over_ranks(1.5 * (rank + 1)) == 1.5 * world

        # per-rank seeds give independent batches of the same shape
        w = workloads.Workload("t", "decode", 8, 2, 64, True, batch=5, q_len=2,
                               kv_range=(3, 40), sink_dist="uniform2", seed=9)
        mine = workloads.make_inputs(w, seed=runner.rank_seed(w.seed, rank))
        shapes = [None] * world
        dist.all_gather_object(shapes, (mine["q"].shape[1:], float(mine["q"].float().sum())))
        assert all(s[0] == shapes[0][0] for s in shapes)
        assert len({s[1] for s in shapes}) == world

        # shard one batch by sequence, run each shard, concatenate on rank 0
        full = workloads.make_inputs(w)
        seqs = runner.shard_sequences(full["batch"], rank, world)
        sub = runner.slice_sequences(full, w.num_kv_heads, seqs)
        out, lse = oracle.attend(sub["q"], sub["k"], sub["v"], sub["sinks"], sub["cu_q"],
                                 sub["cu_k"], 8, 2, 64, w.scale, True, 0)
        parts = [None] * world
        dist.all_gather_object(parts, (list(seqs), out, lse))
        if rank == 0:
            ref_out, ref_lse = oracle.attend(full["q"], full["k"], full["v"], full["sinks"],
                                             full["cu_q"], full["cu_k"], 8, 2, 64, w.scale, True, 0)
            cat_out = np.concatenate([p[1] for p in parts])
            cat_lse = np.concatenate([p[2] for p in parts])
            assert sum(len(p[0]) for p in parts) == full["batch"]
            assert np.array_equal(cat_out, ref_out) and np.array_equal(cat_lse, ref_lse)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_host_path(oracle_lib):
    mp.spawn(_worker, args=(2, _free_port()), nprocs=2, join=True)


def test_shard_sequences_partition():
    from gqa_attention_softmax_gb300 import runner
    for B in (1, 2, 5, 64, 257):
        for world in (1, 2, 3, 8):
            if world > B:
                continue
            got = [list(runner.shard_sequences(B, r, world)) for r in range(world)]
            assert sum(got, []) == list(range(B))
            assert max(map(len, got)) - min(map(len, got)) <= 1
