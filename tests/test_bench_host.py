"""Host logic of bench.py that needs no GPU: the multi-replica time aggregation (two gloo
ranks on CPU), the clock summary, and the JSON line of the reference arm (the oracle on
the host cores)."""
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


def test_reference_arm_prints_the_contract_line(capsys):
    import argparse
    import json

    import oracle
    oracle.build()
    args = argparse.Namespace(gpus=1, steps=1, warmup=3, impl="reference")
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["value"] > 0
    assert line["config"]["workload"] == bench.WORKLOAD
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def _fake_headline():
    plan = {"gridCtas": 16384, "threadsPerCta": 256, "vecBytes": 32, "minBytes": float(2 * 8 * bench.BYTES_PER_RANK)}
    e2e = {"value": 33.9, "unit": "GB/s", "h2d_bytes_per_step": 8 * bench.BYTES_PER_RANK,
           "d2h_bytes_per_step": 8 * bench.BYTES_PER_RANK, "ms_per_step": 3.46, "steps": 10,
           "mode": "zero-copy: vAllReduce on pinned host buffers over NVLink-C2C",
           "explicit_copies": {"value": 21.3, "ms_per_step": 5.51}, "results_match_device_path": True}
    cpu = {"value": 2.7, "unit": "GB/s", "cores": 16, "kind": "oracle",
           "sample": "whole workload (8 x 64 MiB fp32 sum), 200 runs on 16 threads, 20 on 1",
           "single_thread": {"value": 0.4, "cores": 1}, "cpu_model": "Neoverse-V2"}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 8}
    return bench.make_headline(value=762.75, t_max=1.54e-4, steps=20, warmup=5, world=1, plan=plan,
                               achieved=6973.7, hbm=6774.2, peak_kind="measured", traffic=1.0227e9,
                               clocks=clocks, e2e=e2e, cpu_baseline=cpu, sample_ok=True, async_error=0)


def test_headline_is_short_and_carries_the_contract_keys():
    import json
    line = _fake_headline()
    text = json.dumps(line)
    assert len(text) < bench.HEADLINE_MAX_CHARS
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "e2e",
              "cpu_baseline", "gpu_launches"):
        assert k in line, k
    assert line["config"]["workload"] == bench.WORKLOAD
    rf = line["roofline"]
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"]) and rf["bound"] == "hbm"
    assert rf["algorithmic_bytes_per_launch"] == 2 * 8 * bench.BYTES_PER_RANK
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert line["cpu_baseline"]["single_thread"]["cores"] == 1 and line["cpu_baseline"]["cpu_model"]


def test_headline_is_printed_last_after_the_side_lines():
    import io
    import json
    big = [{"bytes_per_rank": 1024 * 4 ** k, "us": 1.0, "graph_us": 1.0} for k in range(11)]
    extras = [("sweep_allreduce_onepass", big), ("ring_sweep", {"rows": [[1, 2, 3]] * 400}),
              ("other_workloads", {"a": {"us": 1.0}})]
    buf = io.StringIO()
    bench.emit(extras, _fake_headline(), out=buf)
    lines = buf.getvalue().strip().splitlines()
    assert len(lines) == 4
    assert [json.loads(x)["extra"] for x in lines[:3]] == [e[0] for e in extras]
    last = json.loads(lines[-1])
    assert last["metric"] == bench.METRIC and "extra" not in last
    assert len(lines[-1]) < bench.HEADLINE_MAX_CHARS


def test_emit_refuses_an_overlong_headline():
    line = _fake_headline()
    line["config"]["padding"] = "x" * bench.HEADLINE_MAX_CHARS
    with pytest.raises(RuntimeError):
        bench.emit([], line, out=__import__("io").StringIO())


def test_cpu_model_names_something():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
