"""The multi-process path of bench.py on CPU: two gloo ranks (world size 2).
Sequences are sharded across ranks with no exchange on the data path; the
only collective is the timing's barrier and max over ranks."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import gdn_inputs as gi


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench._dist() == (ws, rank, rank)
        # the slowest rank's time decides the step time on every rank
        t = bench._barrier_max(1e-3 * (rank + 1), ws)
        # each rank's own sequences: a first state value per rank
        wl = gi.workload_batched_decode(batch=2, sets=1, shard=rank)
        first = float(wl["state"].reshape(-1)[0])
        out[rank] = (t, first)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_max_time_and_own_distinct_sequences():
    ws = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(ws, _free_port(), out), nprocs=ws, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    assert res[0][0] == res[1][0] == 2e-3  # max over ranks, seen by both
    assert res[0][1] != res[1][1]  # distinct sequences per rank
    single = gi.workload_batched_decode(batch=2, sets=1)
    assert res[0][1] == float(single["state"].reshape(-1)[0])  # rank 0 = one-process data


def test_reference_arm_runs_on_rank_zero_only():
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=3, cpu_seconds=0.1, batch=64)
    assert bench.run_reference(args, 2, 1) is None  # other ranks exit without work


def test_shards_are_reproducible():
    a = gi.workload_batched_decode(batch=2, sets=1, shard=3)
    b = gi.workload_batched_decode(batch=2, sets=1, shard=3)
    assert np.array_equal(a["state"].numpy(), b["state"].numpy())
    assert torch.equal(a["steps"][0].mixed_qkv, b["steps"][0].mixed_qkv)
