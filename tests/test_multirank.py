"""The benchmark's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own problem (weak scaling, no collective on the data
path); the only cross-rank step is the max over ranks of the timed region."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from head_attention_fwd_gb300.inputs import WORKLOADS


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_local = 1.25 + rank  # rank 1 is the slow one
        bench.barrier(world)
        t = bench.max_over_ranks(t_local, world)
        w = WORKLOADS["mha_f16_s4096"]
        seeds = [bench.rank_seed(w, rank, i) for i in range(8)]
        value = bench.aggregate_tflops(w.attn_flops, 100, world, t)
        out[rank] = (t, tuple(seeds), value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max_time_and_draw_distinct_problems():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    (t0, s0, v0), (t1, s1, v1) = out[0], out[1]
    assert t0 == t1 == 2.25                      # max over ranks
    assert not set(s0) & set(s1)                 # each rank its own inputs
    w = WORKLOADS["mha_f16_s4096"]
    assert v0 == v1 == pytest.approx(w.attn_flops * 100 * 2 / 2.25 / 1e12)
