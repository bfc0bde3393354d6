"""The multi-process path of bench.py, on CPU with the gloo backend.

Under torchrun every rank runs its own replica of the batch (the attention
path partitions by batch and needs no collective); the step time of the job
is the slowest rank's, and the reported value counts the tokens of all
ranks. These tests run two gloo ranks on 127.0.0.1 and check the rank
environment, the max-over-ranks reduction and the whole-job throughput.
"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = bench.dist_env()
    torch.distributed.init_process_group("gloo", rank=r, world_size=w)
    try:
        # rank 1 is the slow one in the first value, rank 0 in the second
        mine = [1.0 + r, 5.0 - r, 3.0]
        got = bench.max_over_ranks(mine, torch.device("cpu"))
        torch.distributed.barrier()
        out[r] = (r, w, local, got)
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        rank, w, local, got = out[r]
        assert (rank, w, local) == (r, world, r)
        assert got == [2.0, 5.0, 3.0]


def test_max_over_ranks_without_a_process_group_is_the_identity():
    assert not torch.distributed.is_initialized()
    assert bench.max_over_ranks([1.5, 2.0]) == [1.5, 2.0]


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_job_throughput_counts_every_rank_against_the_slowest_step(world):
    # 256 query tokens per rank, 0.1 ms slowest step -> 2.56 M tokens/s per rank
    assert bench.job_throughput(world, 256, 0.1) == pytest.approx(world * 2.56e6)


def test_dist_env_defaults_to_one_process(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
