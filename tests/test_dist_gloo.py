"""The multi-GPU path of the benchmark on CPU: two gloo ranks, each with its own
seeded instance, the slowest rank's time deciding the step, and the reference
arm doing its work on rank 0 only."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from quantized_kv_decode_partial_gb300.dist import max_over_ranks, rank_seed, weak_scaling_rate
from quantized_kv_decode_partial_gb300.workloads import DecodeSpec, make_case


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        spec = DecodeSpec(name="dist", num_seqs=2, num_q_heads=4, num_kv_heads=2, head_dim=64, n_query=1,
                          block_size=16, bits=16, length_range=(10, 50), seed=5)
        case = make_case(spec, seed=rank_seed(spec.seed, rank))
        # every rank reports its own elapsed time; the slowest one decides
        slowest = max_over_ranks(1.5 + rank, torch.device("cpu"))
        gathered = [None] * world
        dist.all_gather_object(gathered, (case.lens_host, float(case.q.float().sum())))
        results[rank] = (slowest, gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_draw_distinct_instances_and_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn", join=True)
    assert sorted(results.keys()) == [0, 1]
    for rank in range(world):
        slowest, gathered = results[rank]
        assert slowest == 2.5  # max of 1.5 and 2.5, on every rank
        assert gathered[0][1] != gathered[1][1]  # different queries on different ranks
    assert weak_scaling_rate(10 ** 9, world, 1.0) == pytest.approx(2000.0)


def test_single_process_needs_no_group():
    assert max_over_ranks(3.25, torch.device("cpu")) == 3.25
    assert rank_seed(100, 0) == 100 and rank_seed(100, 1) != rank_seed(100, 2)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "cpu_oracle_baseline", lambda *a, **k: called.append(1))
    bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert not called and capsys.readouterr().out == ""
