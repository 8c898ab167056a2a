"""Multi-rank host logic on CPU: two gloo ranks run what the benchmark's
N-GPU path does around the kernels (per-rank batches, barrier, maximum of
the per-rank times, job throughput)."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunked_linear_attention_bounded_gb300 import replicas
from chunked_linear_attention_bounded_gb300.inputs import WORKLOADS, make_inputs, small_variant


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = replicas.rank_env()
        assert (env.rank, env.world, env.local) == (rank, world, rank)
        w = replicas.rank_workload(small_variant(WORKLOADS["varlen64k"], T=300, H=2, n_docs=3), rank)
        inp = make_inputs(w, with_grad=True)
        replicas.barrier(world)
        # per-rank "step times": the job is as slow as its slowest rank
        ms = 1.5 + 2.0 * rank
        ms_max = replicas.max_over_ranks(ms, world)
        value = replicas.job_throughput(w.tokens, world, ms_max)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"seed": w.seed, "ms_max": ms_max, "value": value,
                       "q_sum": float(inp["q"].float().sum()), "tokens": w.tokens}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_and_shard(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    # each rank processed its own batch
    assert r[0]["seed"] != r[1]["seed"]
    assert r[0]["q_sum"] != r[1]["q_sum"]
    # every rank sees the slowest rank's time and the same job throughput
    assert r[0]["ms_max"] == r[1]["ms_max"] == pytest.approx(3.5)
    assert r[0]["value"] == r[1]["value"] == pytest.approx(world * r[0]["tokens"] / 3.5e-3)


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert replicas.max_over_ranks(2.5, 1) == 2.5
    replicas.barrier(1)
    w = WORKLOADS["c8k"]
    assert replicas.rank_workload(w, 0) is w
    assert replicas.rank_workload(w, 3).seed == w.seed + 3 * replicas.RANK_SEED_STRIDE
    assert replicas.job_throughput(1000, 1, 2.0) == pytest.approx(5e5)
