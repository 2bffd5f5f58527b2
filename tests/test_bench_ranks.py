"""The multi-process side of bench.py on CPU (gloo, world size 2): the timed
region's time is the maximum over ranks, and the oracle arm runs on rank 0
alone (the other ranks return at once, before touching a GPU)."""

import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        got = bench.max_over_ranks(1.25 + rank, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    port = 29500 + os.getpid() % 1000
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 2.25, 1: 2.25}


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    # a GPU call would raise here (no CUDA in this process): returning first is the check
    monkeypatch.setattr(torch.cuda, "set_device", lambda *_: pytest.fail("touched the GPU"))
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) is None
    assert capsys.readouterr().out == ""
