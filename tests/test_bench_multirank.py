"""The benchmark's multi-rank logic on CPU with the gloo backend (world size 2):
replicas get distinct seeds, the job time is the slowest rank's, and the
reported rate counts every rank's steps."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 50.0 * rank  # rank 1 is the slower replica
        worst = bench.max_over_ranks(ms, torch.device("cpu"))
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.replica_seed(0, rank))
        out[rank] = (worst, bench.job_rate(world, 20, worst), tuple(seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_on_gloo():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    for rank in range(world):
        worst, rate, seeds = res[rank]
        assert worst == 150.0                      # max over ranks
        assert rate == pytest.approx(2 * 20 / 0.150)  # all ranks' steps over the slowest time
        assert len(set(seeds)) == world            # independent replicas


def test_single_process_helpers():
    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_rate(1, 1000, 500.0) == pytest.approx(2000.0)


def test_vocab_kernel_count_follows_the_launch_form(monkeypatch):
    """The benchmark's kernel count per vocabulary step (its gpu_launches claim): the paired form
    launches a flag reset kernel, the paired kernel and the combine; DG_VOCAB_COOP=1 replaces the
    reset kernel by a memset; fp32 runs a kernel and the re-noise (plans are host-only queries)."""
    from canvas_denoising_gb300 import binding as B
    from canvas_denoising_gb300.configs import WORKLOADS
    from canvas_denoising_gb300 import build as build_mod
    build_mod.build()  # the host-side plan query needs the built library, not a GPU
    B.load()
    w = WORKLOADS["v262k_d2816_p4k"]
    monkeypatch.delenv("DG_VOCAB_COOP", raising=False)
    assert bench.vocab_kernels_per_call(B, w, torch.bfloat16) == 3
    monkeypatch.setenv("DG_VOCAB_COOP", "1")
    assert bench.vocab_kernels_per_call(B, w, torch.bfloat16) == 2
    assert bench.vocab_kernels_per_call(B, WORKLOADS["tiny_f32"], torch.float32) == 2
