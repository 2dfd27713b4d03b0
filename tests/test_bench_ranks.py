"""The replicas path of bench.py (--gpus N under torchrun: one independent
replica per rank, no data-path collective): the cross-rank combination of the
timed region -- slowest rank's time, all ranks' tokens -- run as two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, toks = 100.0 + 50.0 * rank, 200 + 10 * rank   # rank 1 is the slower one
        out[rank] = bench.combine_ranks(ms, toks, world, "cpu")
    finally:
        dist.destroy_process_group()


def test_combine_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    # every rank sees the slowest time and the tokens of both ranks
    assert out[0] == out[1] == (150.0, 410.0)
    # whole-job value = all tokens / slowest time
    ms_max, toks = out[0]
    assert toks / (ms_max / 1000.0) == pytest.approx(410.0 / 0.15)


def test_combine_ranks_single_process():
    assert bench.combine_ranks(12.5, 30, 1, "cpu") == (12.5, 30.0)
