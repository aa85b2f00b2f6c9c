"""Host logic of bench.py that needs no GPU: the multi-replica time aggregation (two gloo
ranks on CPU) and the JSON contract of the reference arm's helpers."""
from __future__ import annotations

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = 1e-3 * (rank + 1)
    t_max = bench.max_over_ranks(t, dist, "cpu")
    out[rank] = (t_max, bench.job_busbw(world, t_max))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(2e-3) and res[1][0] == pytest.approx(2e-3)
    want = 2 * bench.BYTES_PER_RANK / 2e-3 * (2 * 7 / 8) / 1e9
    assert res[0][1] == pytest.approx(want) and res[1][1] == pytest.approx(want)


def test_single_process_time_is_unchanged():
    assert bench.max_over_ranks(0.5) == 0.5
    assert bench.job_busbw(1, 1.0) == pytest.approx(bench.BYTES_PER_RANK * 1.75 / 1e9)


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["1965, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "2070, 2070, 1000.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
