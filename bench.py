"""Benchmark: ring all-reduce among 8 virtual ranks on one GB300.

Workload (one "step"): all-reduce, sum, fp32, N = 8 virtual ranks, 64 MiB per rank,
seeded uniform[-1,1) inputs resident in HBM, through the C ABI (vAllReduce).  The
reported metric is bus bandwidth, busBW = algBW * 2(N-1)/N with algBW = bytes per rank /
time (NCCL book chapter 5, ring.cc), plus the fraction of measured HBM bandwidth that
the kernel's minimum traffic (read N*S + write N*S) reaches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]

--impl reference times the CPU oracle (the plain order-matched C implementation) on the
host cores for the same workload.  With --gpus N > 1 (under torchrun) every GPU runs an
independent replica of the workload (the virtual ranks never span GPUs); the value is
the sum over GPUs of bytes moved divided by the slowest GPU's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
N_RANKS = 8
BYTES_PER_RANK = 64 << 20
COUNT = BYTES_PER_RANK // 4
METRIC = "allreduce busBW GB/s & % of HBM peak vs bytes/rank, N=8 virtual ranks, 1×GB300"
WORKLOAD = "ring all-reduce, sum, fp32, N=8 virtual ranks, 64 MiB per rank"
PROFILE = os.path.join(ROOT, "profiles", "allreduce_onepass_fp32_8x64MiB.md")
KERNEL_SOURCES = ["collective_communication_virtual_gb300/csrc/k_onepass.cu",
                  "collective_communication_virtual_gb300/csrc/device.cuh"]


def bus_factor(n):
    return 2.0 * (n - 1) / n


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches these sources."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m or not t or m.group(1) != kernel_hash():
        return None
    return float(t.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(t, dist=None, device=None):
    """The slowest replica's time (the job's time); t itself on a single process."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt)


def job_busbw(world, t_max):
    """Whole-job busBW: every replica moves BYTES_PER_RANK per virtual rank per step."""
    return world * BYTES_PER_RANK / t_max * bus_factor(N_RANKS) / 1e9


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ---------------------------------------------------------------------------------------
# Reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch

    import oracle
    from collective_communication_virtual_gb300 import inputs
    cores = len(os.sched_getaffinity(0))
    xs = inputs.uniform_ranks(N_RANKS, COUNT, torch.float32, 1)
    for _ in range(args.warmup):
        oracle.allreduce(xs, "sum", nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.allreduce(xs, "sum", nthreads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    busbw = BYTES_PER_RANK / dt * bus_factor(N_RANKS) / 1e9
    line = {"metric": METRIC, "value": busbw, "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD, "n_ranks": N_RANKS, "bytes_per_rank": BYTES_PER_RANK},
            "cpu_baseline": {"value": busbw, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "the whole workload per step (8 x 64 MiB fp32)"},
            "e2e": {"value": busbw, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------------------

def time_allreduce(V, torch, comm, send, recv, count, steps, warmup, stream):
    for _ in range(warmup):
        V.vAllReduce(send, recv, count, torch.float32, "sum", comm, stream)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        V.vAllReduce(send, recv, count, torch.float32, "sum", comm, stream)
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / 1e3 / steps


def load(V, torch, comm, send, recv, stream, seconds):
    """Untimed all-reduces for about `seconds` (keeps clocks at their loaded value)."""
    t0 = time.time()
    while time.time() - t0 < seconds:
        for _ in range(50):
            V.vAllReduce(send, recv, COUNT, torch.float32, "sum", comm, stream)
        torch.cuda.synchronize()


def cpu_baseline_sample(torch):
    import oracle
    from collective_communication_virtual_gb300 import inputs
    cores = len(os.sched_getaffinity(0))
    xs = inputs.uniform_ranks(N_RANKS, COUNT, torch.float32, 1)
    oracle.allreduce(xs, "sum", nthreads=cores)
    reps, t0 = 0, time.perf_counter()
    while reps < 3 or (time.perf_counter() - t0 < 10.0 and reps < 50):
        oracle.allreduce(xs, "sum", nthreads=cores)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return {"value": BYTES_PER_RANK / dt * bus_factor(N_RANKS) / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": f"the whole workload (8 x 64 MiB fp32 sum), {reps} runs"}


def run_ours(args):
    import torch

    from collective_communication_virtual_gb300 import build, inputs, vcomm as V

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm, peak_kind = peaks()

    xs = inputs.uniform_ranks(N_RANKS, COUNT, torch.float32, 1)
    send = [x.to(dev) for x in xs]
    recv = [torch.empty_like(s) for s in send]
    comm = V.vcommInit(N_RANKS, 1, V.vProtoSimple)
    V.vcommSetAlgo(comm, "onepass")
    plan = V.vcommQueryPlan(comm, V.vCollAllReduce, COUNT, torch.float32, True)

    # correctness of the timed configuration: sampled elements against the oracle
    V.vAllReduce(send, recv, COUNT, torch.float32, "sum", comm, stream)
    torch.cuda.synchronize()
    sample_ok = check_sample(torch, V, xs, recv)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # The timed region is milliseconds long, far shorter than nvidia-smi's 200 ms
        # sampling period, so the GPU is kept under the same load (untimed all-reduces)
        # for about a second on either side of it; the samples bracket the timed steps.
        clocks.wait_first()
        load(V, torch, comm, send, recv, stream, seconds=1.0)
        t = time_allreduce(V, torch, comm, send, recv, COUNT, args.steps, args.warmup, stream)
        load(V, torch, comm, send, recv, stream, seconds=0.5)
        t_max = max_over_ranks(t, dist if world > 1 else None, dev)
    err = V.vcommGetAsyncError(comm)
    busbw_one = BYTES_PER_RANK / t * bus_factor(N_RANKS) / 1e9
    value = job_busbw(world, t_max)
    achieved = plan["minBytes"] / t / 1e9

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_ranks": N_RANKS, "bytes_per_rank": BYTES_PER_RANK,
                       "algo": "onepass", "channels": plan["nChannels"], "grid_ctas": plan["gridCtas"],
                       "threads_per_cta": plan["threadsPerCta"],
                       "l2": "inputs larger than L2 (8 x 64 MiB read + 8 x 64 MiB written per step)",
                       "parallelism": f"{world} independent replica(s) of 8 virtual ranks"},
            "hbm_frac": achieved / hbm,
            "alg_bw_gbs": BYTES_PER_RANK / t / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_kind": peak_kind,
                         "traffic": profiled_traffic(),
                         "algorithmic_bytes_per_launch": plan["minBytes"]},
            "gpu_launches": args.steps,
            "clocks": clocks.summary(),
            "parity_sample_ok": sample_ok,
            "async_error": err}

    if rank == 0 and not args.no_extras:
        line["e2e"] = e2e_allreduce(torch, V, comm, xs, dev, stream, steps=max(3, min(args.steps, 10)))
        line["sweep"] = sweep(torch, V, dev, stream, hbm)
        line["channel_sweep"] = channel_sweep(torch, V, send, recv, stream)
        line["cpu_baseline"] = cpu_baseline_sample(torch)
    elif not args.no_extras:
        line["e2e"] = None
    V.vcommDestroy(comm)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


def check_sample(torch, V, xs, recv, n_samples=4096):
    """Compare sampled outputs with the oracle: the elements of each sample are placed in a
    tiny all-reduce whose block layout reproduces their ring order."""
    import oracle
    g = torch.Generator().manual_seed(123)
    idx = torch.randint(0, COUNT, (n_samples,), generator=g)
    B = oracle.block_elems(COUNT, N_RANKS, 4)
    blocks = (idx // B).tolist()
    ve = 4                                   # one 16-byte vector per block in the tiny case
    tiny = [torch.zeros(N_RANKS * ve, dtype=torch.float32) for _ in range(N_RANKS)]
    got = [r.cpu() for r in recv[:2]]
    for k, (e, b) in enumerate(zip(idx.tolist(), blocks)):
        for r in range(N_RANKS):
            tiny[r][b * ve] = xs[r][e]
        want = oracle.allreduce(tiny, "sum")[0][b * ve]
        for g_ in got:
            if g_[e].view(torch.int32) != want.view(torch.int32):
                return False
        if k >= 512:                         # the oracle call per sample is slow; 512 is plenty
            break
    return True


def e2e_allreduce(torch, V, comm, xs, dev, stream, steps):
    """Host buffers in, host buffers out: H2D of every rank's input, the all-reduce, and
    D2H of every rank's result, all inside the timed region."""
    host_in = [x.pin_memory() for x in xs]
    host_out = [torch.empty_like(x).pin_memory() for x in xs]
    d_in = [torch.empty_like(x, device=dev) for x in xs]
    d_out = [torch.empty_like(x, device=dev) for x in xs]

    def step():
        for d, h in zip(d_in, host_in):
            d.copy_(h, non_blocking=True)
        V.vAllReduce(d_in, d_out, COUNT, torch.float32, "sum", comm, stream)
        for h, d in zip(host_out, d_out):
            h.copy_(d, non_blocking=True)

    step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    t = start.elapsed_time(stop) / 1e3 / steps
    nbytes = N_RANKS * BYTES_PER_RANK
    return {"value": BYTES_PER_RANK / t * bus_factor(N_RANKS) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "ms_per_step": t * 1e3,
            "steps": steps}


def sweep(torch, V, dev, stream, hbm):
    """busBW and HBM fraction against bytes per rank (1 KiB .. 1 GiB, powers of 4)."""
    out = []
    comm = V.vcommInit(N_RANKS, 1, V.vProtoSimple)
    V.vcommSetAlgo(comm, "onepass")
    for k in range(11):
        nbytes = 1024 * 4 ** k
        count = nbytes // 4
        send = [torch.rand(count, device=dev) for _ in range(N_RANKS)]
        recv = [torch.empty_like(s) for s in send]
        steps = 200 if nbytes <= (1 << 20) else (50 if nbytes <= (64 << 20) else 10)
        t = time_allreduce(V, torch, comm, send, recv, count, steps, 5, stream)
        out.append({"bytes_per_rank": nbytes, "busbw_gbs": nbytes / t * bus_factor(N_RANKS) / 1e9,
                    "hbm_frac": 2 * N_RANKS * nbytes / t / 1e9 / hbm, "us": t * 1e6})
        del send, recv
        torch.cuda.empty_cache()
    V.vcommDestroy(comm)
    return out


def channel_sweep(torch, V, send, recv, stream):
    out = []
    for algo, proto in (("onepass", V.vProtoSimple), ("ring", V.vProtoSimple)):
        for ch in (1, 8, 16, 32):
            comm = V.vcommInit(N_RANKS, ch, proto)
            V.vcommSetAlgo(comm, algo)
            try:
                t = time_allreduce(V, torch, comm, send, recv, COUNT, 5, 2, stream)
                out.append({"algo": algo, "proto": "simple", "channels": ch,
                            "busbw_gbs": BYTES_PER_RANK / t * bus_factor(N_RANKS) / 1e9})
            except V.VcommError as e:
                out.append({"algo": algo, "channels": ch, "error": str(e)})
            V.vcommDestroy(comm)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip e2e, sweeps and the CPU baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    sys.path.insert(0, ROOT)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
