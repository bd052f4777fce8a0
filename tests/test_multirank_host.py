"""The replicated multi-GPU bench's host logic on CPU ranks (gloo, world size 2): seeds
differ per rank, the job time is the slowest rank's, the job rate counts every replica,
and the reference arm runs on rank 0 only.  No GPU is used."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        seconds = 1.0 + rank  # rank 1 is slower
        job = bench.max_over_ranks(dist, seconds, torch.device("cpu"))
        out[rank] = (w, r, local, job, bench.job_rate(100, 10, w, job), bench.rank_seed(2, r))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_cpu_ranks_share_the_slowest_time():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert sorted(out.keys()) == [0, 1]
    for rank in range(world):
        w, r, local, job, rate, seed = out[rank]
        assert (w, r, local) == (world, rank, rank)
        assert job == 2.0                       # the slowest rank's time, on every rank
        assert rate == pytest.approx(100 * 10 * 2 / 2.0)
    assert out[0][5] != out[1][5]               # each replica draws its own inputs


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, 3.5, torch.device("cpu")) == 3.5
    assert bench.job_rate(640, 5, 1, 2.0) == 1600.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "1", "--config", "0"])
    assert bench.run_reference(args, world=2, rank=1) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line_on_rank_zero(capsys):
    import json
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "1", "--config", "0"])
    assert bench.run_reference(args, world=1, rank=0) == 0
    lines = capsys.readouterr().out.strip().splitlines()
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
