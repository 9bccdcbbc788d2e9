"""Host logic of a multi-GPU bench run, exercised with world_size-2 gloo ranks
on CPU: the job time is the slowest rank's, and the job throughput counts the
replicas of every rank."""
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


def _rank(rank, ws, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = bench.max_over_ranks(times[rank], ws, "cpu")
        out[rank] = (ms, bench.job_tflops(2.0e12, ws, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ws = 2
    times = [3.0, 5.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(ws, _free_port(), times, out), nprocs=ws, join=True)
        res = dict(out)
    for r in range(ws):
        ms, tf = res[r]
        assert ms == pytest.approx(5.0)            # every rank reports the slowest rank's time
        assert tf == pytest.approx(2.0e12 * 2 / 5e-3 / 1e12)  # both replicas' flops over that time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(4.5, 1) == 4.5
    assert bench.job_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
