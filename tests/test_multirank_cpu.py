"""Host logic of the multi-GPU (replicas) path, run as two gloo ranks on the
CPU: every rank gets its own batch, the whole-job figures are the summed
useful FLOPs over the slowest rank's time, and only rank 0 runs the
reference arm."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        # each rank its own batch, as the bench's GEM setup draws it
        L = bench._gem_lengths(rank)
        flops = 3.5 * 4.0 * 4 * 128 * float(np.sum(np.asarray(L, dtype=np.float64) ** 2))
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        job_flops, t_max = bench.aggregate_over_ranks(flops, ms, ws, torch.device("cpu"))
        out[rank] = (flops, job_flops, t_max, int(np.sum(L)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_sum_flops_and_take_max_time():
    ws, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
    (f0, j0, t0, T0), (f1, j1, t1, T1) = out[0], out[1]
    assert T0 != T1  # distinct batches per rank
    assert j0 == pytest.approx(f0 + f1) and j1 == pytest.approx(f0 + f1)
    assert t0 == t1 == 15.0


def test_single_rank_is_identity():
    assert bench.aggregate_over_ranks(3.0, 2.0, 1, torch.device("cpu")) == (3.0, 2.0)


def test_reference_arm_silent_on_other_ranks(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus = 1, 3, 2

    bench.run_reference(Args())
    assert capsys.readouterr().out == ""
