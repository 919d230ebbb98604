"""The multi-replica host logic of bench.py on the CPU with two gloo ranks:
every rank gets the slowest rank's times, and the whole-job rates count the
tokens and FLOPs of all replicas over that time.  (The path shards by token
with no collective on the data path; the only collective is this reduction.)"""
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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step time 1 + r ms, kernel time 5 - r ms, e2e 2 ms
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 2.0], dist, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [2.0, 5.0, 2.0]


def test_job_rates_count_every_replica():
    tok, tflops = bench.job_rates(2048, 5.5e11, 1, 0.5)
    assert tok == pytest.approx(2048 / 0.5e-3) and tflops == pytest.approx(5.5e11 / 0.5e-3 / 1e12)
    tok8, tflops8 = bench.job_rates(2048, 5.5e11, 8, 0.5)
    assert tok8 == pytest.approx(8 * tok) and tflops8 == pytest.approx(8 * tflops)
