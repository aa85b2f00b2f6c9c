"""Benchmark: ring all-reduce among 8 virtual ranks on one GB300.

Workload (one "step"): all-reduce, sum, fp32, N = 8 virtual ranks, 64 MiB per rank,
seeded uniform[-1,1) inputs resident in HBM, through the C ABI (vAllReduce).  The
reported metric is bus bandwidth, busBW = algBW * 2(N-1)/N with algBW = bytes per rank /
time (NCCL book chapter 5, ring.cc), plus the fraction of measured HBM bandwidth that
the kernel's minimum traffic (read N*S + write N*S) reaches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]
  python bench.py --workloads [--only NAME]      # the other collectives' workloads only

Output: one JSON line per side measurement (size sweeps, the staged ring's protocol and
channel grids, the other collectives' workloads, the oracle's per-workload timings), each
{"extra": name, ...}, then the headline as the LAST line: the contract keys, the
roofline of the all-reduce kernel, the clocks, e2e and cpu_baseline, under 2,000
characters.

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
                  "collective_communication_virtual_gb300/csrc/onepass.cuh",
                  "collective_communication_virtual_gb300/csrc/reduce_ring.cuh",
                  "collective_communication_virtual_gb300/csrc/device.cuh"]


def bus_factor(n):
    return 2.0 * (n - 1) / n


# GB300 HBM3e bandwidth as NVIDIA states it (context only; the roofline uses the measured
# copy bandwidth).
NOMINAL_HBM_GBS = 7900.0


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


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), e.g. "Neoverse-V2"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                name = line.split(":", 1)[1].strip()
                if name and name != "-":
                    return name
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


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
                             "sample": "the whole workload per step (8 x 64 MiB fp32)",
                             "cpu_model": cpu_model()},
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


def oracle_rate(torch, xs, nthreads, seconds):
    """busBW of the oracle's all-reduce over `xs` on `nthreads` host threads, repeated for
    about `seconds` (at least twice): (GB/s, runs)."""
    import oracle
    oracle.allreduce(xs, "sum", nthreads=nthreads)
    reps, t0 = 0, time.perf_counter()
    while reps < 2 or (time.perf_counter() - t0 < seconds and reps < 1000):
        oracle.allreduce(xs, "sum", nthreads=nthreads)
        reps += 1
    dt = (time.perf_counter() - t0) / reps
    return BYTES_PER_RANK / dt * bus_factor(N_RANKS) / 1e9, reps


def cpu_baseline_sample(torch):
    """The oracle on the whole workload (8 x 64 MiB fp32 sum): on every host core the
    process may use, and on one core; about 8 s of CPU work each."""
    from collective_communication_virtual_gb300 import inputs
    cores = len(os.sched_getaffinity(0))
    xs = inputs.uniform_ranks(N_RANKS, COUNT, torch.float32, 1)
    value, reps = oracle_rate(torch, xs, cores, 8.0)
    one, reps1 = oracle_rate(torch, xs, 1, 8.0)
    return {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"whole workload (8 x 64 MiB fp32 sum), {reps} runs on {cores} threads, {reps1} on 1",
            "single_thread": {"value": one, "cores": 1}, "cpu_model": cpu_model()}


def cpu_baseline_workloads(torch):
    """The oracle as it stands on the other collectives' workloads, once each, on all host
    cores where it takes a thread count: minimum bytes per second, the GPU rows' basis."""
    import oracle
    from collective_communication_virtual_gb300 import inputs
    cores = len(os.sched_getaffinity(0))
    n, out = N_RANKS, {}

    def row(name, fn, nbytes):
        t0 = time.perf_counter()
        fn()
        t = time.perf_counter() - t0
        out[name] = {"us": t * 1e6, "min_bytes": nbytes, "gbs": nbytes / t / 1e9}

    cnt, rc = 13_107_200, 13_107_200 // n
    g = inputs.normal_ranks(n, cnt, 1e-3, torch.bfloat16, 2)
    row("fsdp_reduce_scatter_scale_cast_bf16_25MiB",
        lambda: oracle.reduce_scatter_scale(g, "sum", 1.0 / n, nthreads=cores), n * cnt * 2 + n * rc * 4)
    sh = [x[:rc].clone() for x in g]
    row("fsdp_allgather_bf16_25MiB", lambda: oracle.allgather(sh), n * rc * 2 + n * cnt * 2)
    del g, sh
    send, counts, sd, rd, recv_elems = inputs.moe_dispatch()
    moved = int(counts.sum()) * 2
    row("moe_alltoallv_bf16_8x4096x4096_top2", lambda: oracle.alltoallv(send, counts, sd, rd, recv_elems), 2 * moved)
    del send
    S = BYTES_PER_RANK
    xs = inputs.uniform_ranks(n, COUNT, torch.float32, 1)
    parts = [x[:COUNT // n].clone() for x in xs]
    row("reduce_scatter_fp32_64MiB", lambda: oracle.reduce_scatter(xs, "sum", nthreads=cores), n * S + S)
    row("allgather_fp32_64MiB", lambda: oracle.allgather(parts), S + n * S)
    row("broadcast_fp32_64MiB", lambda: oracle.broadcast(xs, 0), S + n * S)
    row("alltoall_fp32_64MiB", lambda: oracle.alltoall(xs), 2 * n * S)
    row("reduce_fp32_64MiB", lambda: oracle.reduce(xs, "sum", 0, nthreads=cores), n * S + S)
    row("gather_fp32_8x64MiB", lambda: oracle.gather(xs, 0), 2 * n * S)
    big = torch.cat(xs)
    row("scatter_fp32_8x64MiB", lambda: oracle.scatter(big, n, 0), 2 * n * S)
    row("allreduce_double_binary_tree_fp32_64MiB", lambda: oracle.allreduce_tree(xs, "sum", nthreads=cores),
        2 * n * S)
    return {"cores": cores, "kind": "oracle", "runs": 1, "workloads": out}


HEADLINE_MAX_CHARS = 2000


def make_headline(*, value, t_max, steps, warmup, world, plan, achieved, hbm, peak_kind, traffic, clocks,
                  e2e, cpu_baseline, sample_ok, async_error):
    """The contract line: the keys the driver reads, the roofline of the all-reduce kernel,
    clocks, e2e and cpu_baseline -- nothing of the side measurements, which go on lines
    of their own, so that it stays short."""
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": t_max * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_ranks": N_RANKS, "bytes_per_rank": BYTES_PER_RANK,
                       "algo": "onepass", "grid_ctas": plan["gridCtas"],
                       "threads_per_cta": plan["threadsPerCta"], "vector_bytes": plan["vecBytes"],
                       "l2": "inputs larger than L2 (8 x 64 MiB read + 8 x 64 MiB written per step)",
                       "parallelism": f"{world} independent replica(s) of 8 virtual ranks"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_kind": peak_kind, "traffic": traffic,
                         "algorithmic_bytes_per_launch": plan["minBytes"],
                         "kernel": "k_allreduce_onepass<f32,sum,32B,8 ranks>"},
            "gpu_launches": steps,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu_baseline,
            "parity_sample_ok": sample_ok,
            "async_error": async_error}
    return line


def emit(extras, headline, out=None):
    """Print every side measurement as its own JSON line, then the headline last."""
    out = out or sys.stdout
    for name, data in extras:
        print(json.dumps({"extra": name, "data": data}), file=out)
    text = json.dumps(headline)
    if len(text) > HEADLINE_MAX_CHARS:
        raise RuntimeError(f"headline is {len(text)} characters, over {HEADLINE_MAX_CHARS}")
    print(text, file=out)
    out.flush()


def run_ours(args):
    import torch

    from collective_communication_virtual_gb300 import build, inputs, vcomm as V

    rank, world, local = dist_env()
    dist = None
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
    plan = V.vcommQueryPlan(comm, V.vCollAllReduce, COUNT, torch.float32, 32)

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
        t_max = max_over_ranks(t, dist, dev)
    err = V.vcommGetAsyncError(comm)
    value = job_busbw(world, t_max)
    achieved = plan["minBytes"] / t / 1e9

    # end to end through the public API with host buffers, every replica, slowest one
    e2e = e2e_allreduce(torch, V, comm, xs, dev, stream, steps=max(3, min(args.steps, 10)), dist=dist,
                        world=world)
    extras = []
    cpu = None
    if rank == 0 and not args.no_extras:
        extras.append(("sweep_allreduce_onepass", sweep(torch, V, dev, stream, hbm)))
        extras.append(("sweep_collectives_onepass", sweep_collectives(torch, V, dev, hbm)))
        extras.append(("ring_sweep", ring_sweep(torch, V, dev)))
        extras.append(("ring_allreduce_chunk_channel_grid", ring_grid(torch, V, send, recv, stream)))
        extras.append(("other_workloads", other_workloads(torch, V, dev, stream, hbm)))
    if rank == 0 and world == 1:
        cpu = cpu_baseline_sample(torch)
        if not args.no_extras:
            extras.append(("cpu_baseline_other_workloads", cpu_baseline_workloads(torch)))
    V.vcommDestroy(comm)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        line = make_headline(value=value, t_max=t_max, steps=args.steps, warmup=args.warmup, world=world,
                             plan=plan, achieved=achieved, hbm=hbm, peak_kind=peak_kind,
                             traffic=profiled_traffic(), clocks=clocks.summary(), e2e=e2e,
                             cpu_baseline=cpu, sample_ok=sample_ok, async_error=err)
        emit(extras, line)
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


def e2e_allreduce(torch, V, comm, xs, dev, stream, steps, dist=None, world=1):
    """The headline metric end to end: host buffers in, host buffers out, through
    vAllReduce, on every replica; the slowest replica's time.

    value (mode "zero-copy"): the caller hands vAllReduce pinned host buffers, which the
    library accepts as they are; every step the kernel reads all 8 ranks' inputs from host
    memory and writes all 8 results back to host memory over NVLink-C2C, inside the timed
    region.  explicit_copies: per step, cudaMemcpyAsync of the 8 inputs to device buffers,
    vAllReduce on them, and cudaMemcpyAsync of the 8 results back, serialised on one
    stream.  Both move 8 x 64 MiB each way per step."""
    host_in = [x.pin_memory() for x in xs]
    host_out = [torch.empty_like(x).pin_memory() for x in xs]
    d_in = [torch.empty_like(x, device=dev) for x in xs]
    d_out = [torch.empty_like(x, device=dev) for x in xs]

    def zero_copy():
        V.vAllReduce(host_in, host_out, COUNT, torch.float32, "sum", comm, stream)

    def explicit():
        for d, h in zip(d_in, host_in):
            d.copy_(h, non_blocking=True)
        V.vAllReduce(d_in, d_out, COUNT, torch.float32, "sum", comm, stream)
        for h, d in zip(host_out, d_out):
            h.copy_(d, non_blocking=True)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            fn()
        stop.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(start.elapsed_time(stop) / 1e3 / steps, dist, dev)

    # the host link's own ceiling for this traffic: the copy engines moving the same bytes
    # both ways at once (8 inputs in, 8 results out, on two streams)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def copies_both_ways():
        up.wait_stream(stream)
        down.wait_stream(stream)
        with torch.cuda.stream(up):
            for d, h in zip(d_in, host_in):
                d.copy_(h, non_blocking=True)
        with torch.cuda.stream(down):
            for h, d in zip(host_out, d_out):
                h.copy_(d, non_blocking=True)
        stream.wait_stream(up)
        stream.wait_stream(down)

    t = timed(zero_copy)
    t_copy = timed(explicit)
    consistent = all(torch.equal(host_out[r], d_out[r].cpu()) for r in range(N_RANKS))
    t_link = timed(copies_both_ways)
    nbytes = N_RANKS * BYTES_PER_RANK
    return {"value": job_busbw(world, t), "unit": "GB/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes, "ms_per_step": t * 1e3,
            "steps": steps, "mode": "zero-copy: vAllReduce on pinned host buffers over NVLink-C2C",
            "explicit_copies": {"value": job_busbw(world, t_copy), "ms_per_step": t_copy * 1e3},
            "host_link": {"copy_engines_gbs": 2 * nbytes / t_link / 1e9, "frac": t_link / t},
            "results_match_device_path": consistent}


def other_workloads(torch, V, dev, stream, hbm, only=None):
    """Kernel time and HBM fraction of the other collectives on their workloads.  `only`:
    a comma-separated list of workload names to run alone (a profiler then sees few
    launches and little memory)."""
    from collective_communication_virtual_gb300 import inputs
    comm = V.vcommInit(N_RANKS, 1, V.vProtoSimple)
    V.vcommSetAlgo(comm, "onepass")
    out = {}

    chosen = None if only is None else set(only.split(","))

    def want(*names):
        return chosen is None or any(nm in chosen for nm in names)

    def tm(fn, steps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / steps

    def rec(name, t, nbytes, bytes_per_rank, factor):
        out[name] = {"us": t * 1e6, "min_bytes": nbytes, "hbm_frac": nbytes / t / 1e9 / hbm,
                     "busbw_gbs": bytes_per_rank / t * factor / 1e9}

    def literal(row, nbytes, t):
        # The staged ring's own traffic: every block of input read once and of output
        # written once, plus a FIFO slot written and read at every hop -- (6N-4)·S for an
        # all-reduce, (3N-1)·S for reduce-scatter and all-gather (S = bytes per rank).
        row["literal_bytes"] = nbytes
        row["literal_frac"] = nbytes / t / 1e9 / hbm

    n = N_RANKS
    f1 = (n - 1) / n
    # FSDP bucket: bf16 25 MiB per rank, reduce-scatter * 1/8 -> fp32, then all-gather
    if want("fsdp_reduce_scatter_scale_cast_bf16_25MiB", "fsdp_allgather_bf16_25MiB"):
        cnt, rc = 13_107_200, 13_107_200 // n
        g = [x.to(dev) for x in inputs.normal_ranks(n, cnt, 1e-3, torch.bfloat16, 2)]
        sh = [torch.empty(rc, device=dev) for _ in range(n)]
        t = tm(lambda: V.vReduceScatterScaleCast(g, sh, rc, torch.bfloat16, "sum", torch.float32, 1.0 / n,
                                                 comm, stream))
        rec("fsdp_reduce_scatter_scale_cast_bf16_25MiB", t, n * cnt * 2 + n * rc * 4, cnt * 2, f1)
        shb = [s.to(torch.bfloat16) for s in sh]
        if want("fsdp_allgather_bf16_25MiB"):
            t = tm(lambda: V.vAllGather(shb, g, rc, torch.bfloat16, "sum", comm, stream))
            rec("fsdp_allgather_bf16_25MiB", t, n * rc * 2 + n * cnt * 2, cnt * 2, f1)
        del g, sh, shb
    # MoE dispatch: variable all-to-all, bf16, 8 x 4096 tokens x 4096, top-2 Zipf(1.2)
    if want("moe_alltoallv_bf16_8x4096x4096_top2"):
        send, counts, sd, rd, recv_elems = inputs.moe_dispatch()
        s_d = [x.to(dev) for x in send]
        r_d = [torch.empty(e, dtype=torch.bfloat16, device=dev) for e in recv_elems]
        tabs = [x.to(dev) for x in (counts, sd, rd)]
        t = tm(lambda: V.vAllToAllv(s_d, r_d, *tabs, torch.bfloat16, comm, stream))
        moved = int(counts.sum()) * 2
        rec("moe_alltoallv_bf16_8x4096x4096_top2", t, 2 * moved, moved // n, f1)
        out["moe_alltoallv_bf16_8x4096x4096_top2"]["max_recv_mib"] = max(recv_elems) * 2 / 2**20
        del s_d, r_d
        torch.cuda.empty_cache()
    # a ragged reduce-scatter: 3 ranks of 64 MiB bf16, blocks of 11,184,810 elements
    # (22,369,620 bytes, 4 past a 16-byte boundary)
    if want("reduce_scatter_bf16_3x64MiB_ragged"):
        n3, rc3 = 3, (32 << 20) // 3
        c3 = V.vcommInit(n3, 1, V.vProtoSimple)
        V.vcommSetAlgo(c3, "onepass")
        xs = [x.to(dev) for x in inputs.uniform_ranks(n3, n3 * rc3, torch.bfloat16, 9)]
        ys = [torch.empty(rc3, dtype=torch.bfloat16, device=dev) for _ in range(n3)]
        t = tm(lambda: V.vReduceScatter(xs, ys, rc3, torch.bfloat16, "sum", c3, stream))
        rec("reduce_scatter_bf16_3x64MiB_ragged", t, (n3 + 1) * n3 * rc3 * 2, n3 * rc3 * 2, (n3 - 1) / n3)
        V.vcommDestroy(c3)
        del xs, ys
        torch.cuda.empty_cache()
    # a ragged all-to-all: 3 ranks of 64 MiB bf16, blocks of 11,184,810 elements
    if want("alltoall_bf16_3x64MiB_ragged"):
        n3, rc3 = 3, (32 << 20) // 3
        c3 = V.vcommInit(n3, 1, V.vProtoSimple)
        V.vcommSetAlgo(c3, "onepass")
        xs = [x.to(dev) for x in inputs.uniform_ranks(n3, n3 * rc3, torch.bfloat16, 10)]
        ys = [torch.empty(n3 * rc3, dtype=torch.bfloat16, device=dev) for _ in range(n3)]
        t = tm(lambda: V.vAllToAll(xs, ys, rc3, torch.bfloat16, "sum", c3, stream))
        rec("alltoall_bf16_3x64MiB_ragged", t, 2 * n3 * n3 * rc3 * 2, n3 * rc3 * 2, (n3 - 1) / n3)
        V.vcommDestroy(c3)
        del xs, ys
        torch.cuda.empty_cache()
    # uniform all-to-all at 1 GiB per rank
    if want("alltoall_fp32_1GiB", "ring_allreduce_fp32_1GiB_simple_32ch"):
        cnt = 1 << 28
        a = [torch.empty(cnt, device=dev) for _ in range(n)]
        b = [torch.empty(cnt, device=dev) for _ in range(n)]
        if want("alltoall_fp32_1GiB"):
            t = tm(lambda: V.vAllToAll(a, b, cnt // n, torch.float32, "sum", comm, stream), 10)
            rec("alltoall_fp32_1GiB", t, 2 * n * cnt * 4, cnt * 4, f1)
        # the staged ring all-reduce at 1 GiB per rank (Simple, 32 channels, 1 MiB chunks)
        if want("ring_allreduce_fp32_1GiB_simple_32ch"):
            for t_ in a:
                t_.uniform_(-1, 1)
            ring = V.vcommInit(n, 32, V.vProtoSimple)
            V.vcommSetAlgo(ring, "ring")
            V.vcommSetChunkBytes(ring, 1 << 20)
            t = tm(lambda: V.vAllReduce(a, b, cnt, torch.float32, "sum", ring, stream), 3)
            rec("ring_allreduce_fp32_1GiB_simple_32ch", t, 2 * n * cnt * 4, cnt * 4, 2 * f1)
            literal(out["ring_allreduce_fp32_1GiB_simple_32ch"], (6 * n - 4) * cnt * 4, t)
            V.vcommDestroy(ring)
        del a, b
        torch.cuda.empty_cache()
    def row(name, fn, nbytes, bytes_per_rank, factor, steps=20):
        if want(name):
            rec(name, tm(fn, steps), nbytes, bytes_per_rank, factor)

    # reduce-scatter, all-gather, broadcast, all-to-all at 64 MiB per rank (fp32)
    S = BYTES_PER_RANK
    x = [torch.rand(COUNT, device=dev) for _ in range(n)]
    y = [torch.empty(COUNT, device=dev) for _ in range(n)]
    part = [torch.empty(COUNT // n, device=dev) for _ in range(n)]
    row("reduce_scatter_fp32_64MiB", lambda: V.vReduceScatter(x, part, COUNT // n, torch.float32, "sum", comm, stream),
        n * S + S, S, f1)
    row("allgather_fp32_64MiB", lambda: V.vAllGather(part, y, COUNT // n, torch.float32, "sum", comm, stream),
        S + n * S, S, f1)
    row("broadcast_fp32_64MiB", lambda: V.vBroadcast(x, y, COUNT, torch.float32, "sum", 0, comm, stream),
        S + n * S, S, f1)
    row("alltoall_fp32_64MiB", lambda: V.vAllToAll(x, y, COUNT // n, torch.float32, "sum", comm, stream),
        2 * n * S, S, f1)
    # rooted collectives: reduce to rank 0; gather to and scatter from rank 0 with 64 MiB
    # per rank (512 MiB at the root, so the working set is far larger than L2)
    out0 = [y[0]] + [None] * (n - 1)
    row("reduce_fp32_64MiB", lambda: V.vReduce(x, out0, COUNT, torch.float32, "sum", 0, comm, stream),
        n * S + S, S, f1)
    if want("gather_fp32_8x64MiB", "scatter_fp32_8x64MiB"):
        root = [torch.empty(n * COUNT, device=dev)] + [None] * (n - 1)
        row("gather_fp32_8x64MiB", lambda: V.vGather(x, root, COUNT, torch.float32, 0, comm, stream),
            2 * n * S, S, f1)
        row("scatter_fp32_8x64MiB", lambda: V.vScatter(root, y, COUNT, torch.float32, 0, comm, stream),
            2 * n * S, S, f1)
        del root
    # the 16-bit and integer all-reduce paths on the same 64 MiB per rank
    for dt, op, name in ((torch.bfloat16, "sum", "bf16_sum"), (torch.float16, "max", "fp16_max"),
                         (torch.int32, "prod", "int32_prod")):
        xs16 = [t_.view(dt) for t_ in x]
        ys16 = [t_.view(dt) for t_ in y]
        cnt16 = xs16[0].numel()
        row(f"allreduce_{name}_64MiB", lambda: V.vAllReduce(xs16, ys16, cnt16, dt, op, comm, stream),
            2 * n * S, S, 2 * f1)
    # the staged ring's own reduce-scatter and all-gather (Simple, 32 channels, 1 MiB chunks)
    ring = V.vcommInit(n, 32, V.vProtoSimple)
    V.vcommSetAlgo(ring, "ring")
    V.vcommSetChunkBytes(ring, 1 << 20)
    for name, fn, nbytes, factor, lit in (
            ("ring_reduce_scatter_fp32_64MiB_simple_32ch",
             lambda: V.vReduceScatter(x, part, COUNT // n, torch.float32, "sum", ring, stream), n * S + S, f1, 3 * n - 1),
            ("ring_allgather_fp32_64MiB_simple_32ch",
             lambda: V.vAllGather(part, y, COUNT // n, torch.float32, "sum", ring, stream), S + n * S, f1, 3 * n - 1),
            ("ring_allreduce_fp32_64MiB_simple_32ch",
             lambda: V.vAllReduce(x, y, COUNT, torch.float32, "sum", ring, stream), 2 * n * S, 2 * f1, 6 * n - 4)):
        row(name, fn, nbytes, S, factor, 10)
        if name in out:
            literal(out[name], lit * S, out[name]["us"] / 1e6)
    # the flag protocols on the same three collectives (32 channels, 1 MiB chunks)
    for proto, pname in ((V.vProtoLL, "ll"), (V.vProtoLL128, "ll128")):
        V.vcommSetProtocol(ring, proto)
        for name, fn, nbytes, factor, lit in (
                (f"ring_reduce_scatter_fp32_64MiB_{pname}_32ch",
                 lambda: V.vReduceScatter(x, part, COUNT // n, torch.float32, "sum", ring, stream), n * S + S, f1,
                 3 * n - 1),
                (f"ring_allgather_fp32_64MiB_{pname}_32ch",
                 lambda: V.vAllGather(part, y, COUNT // n, torch.float32, "sum", ring, stream), S + n * S, f1,
                 3 * n - 1),
                (f"ring_allreduce_fp32_64MiB_{pname}_32ch",
                 lambda: V.vAllReduce(x, y, COUNT, torch.float32, "sum", ring, stream), 2 * n * S, 2 * f1,
                 6 * n - 4)):
            row(name, fn, nbytes, S, factor, 10)
            if name in out:
                literal(out[name], lit * S, out[name]["us"] / 1e6)
    V.vcommSetProtocol(ring, V.vProtoSimple)
    # the same all-reduce with 128 KiB chunks: FIFOs small enough to stay in L2
    V.vcommSetChunkBytes(ring, 128 << 10)
    row("ring_allreduce_fp32_64MiB_simple_32ch_128KiB_chunks",
        lambda: V.vAllReduce(x, y, COUNT, torch.float32, "sum", ring, stream), 2 * n * S, S, 2 * f1, 10)
    if "ring_allreduce_fp32_64MiB_simple_32ch_128KiB_chunks" in out:
        row_ = out["ring_allreduce_fp32_64MiB_simple_32ch_128KiB_chunks"]
        literal(row_, (6 * n - 4) * S, row_["us"] / 1e6)
    V.vcommDestroy(ring)
    tree = V.vcommInit(n, 1, V.vProtoSimple)
    V.vcommSetAlgo(tree, "tree")
    row("allreduce_double_binary_tree_fp32_64MiB", lambda: V.vAllReduce(x, y, COUNT, torch.float32, "sum", tree, stream),
        2 * n * S, S, 2 * f1)
    V.vcommDestroy(tree)
    del x, y, part
    if not want("ddp_64_buckets_64KiB_fp32"):
        V.vcommDestroy(comm)
        return out
    # group batching: 64 gradient buckets of 64 KiB fp32, separate calls vs one group
    nb, bc = 64, 16384
    bx = [[torch.rand(bc, device=dev) for _ in range(n)] for _ in range(nb)]
    by = [[torch.empty(bc, device=dev) for _ in range(n)] for _ in range(nb)]

    def separate(s=stream):
        for i in range(nb):
            V.vAllReduce(bx[i], by[i], bc, torch.float32, "sum", comm, s)

    t_eager = tm(separate, 10)
    # device time of the 64 separate launches: replayed from a CUDA graph (no host gaps)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        separate(torch.cuda.current_stream())
    t_graph = tm(g.replay, 10)
    # device time of the group: the recording happens on the host before the timed region,
    # vcommGroupEnd then uploads the work table and launches one fused kernel
    ts = []
    for rep in range(13):
        V.vcommGroupStart(comm)
        separate()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        V.vcommGroupEnd(comm)
        b.record(stream)
        torch.cuda.synchronize()
        if rep >= 3:
            ts.append(a.elapsed_time(b) / 1e3)
    t_grp = sum(ts) / len(ts)
    out["ddp_64_buckets_64KiB_fp32"] = {"separate_eager_us": t_eager * 1e6,
                                        "separate_graph_replay_us": t_graph * 1e6,
                                        "grouped_us": t_grp * 1e6, "launches_separate": nb,
                                        "launches_grouped": 1,
                                        "min_bytes": 2 * n * nb * bc * 4}
    V.vcommDestroy(comm)
    return out


def time_graph_allreduce(V, torch, comm, send, recv, count, launches, reps):
    """Device time per all-reduce with no host gaps: `launches` calls captured into one CUDA
    graph, replayed `reps` times."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(launches):
            V.vAllReduce(send, recv, count, torch.float32, "sum", comm)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / (reps * launches)


def sweep(torch, V, dev, stream, hbm):
    """busBW and HBM fraction against bytes per rank (1 KiB .. 1 GiB, powers of 4): eager
    calls (host launch cost included) and the same calls replayed from a CUDA graph (device
    time only)."""
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
        tg = time_graph_allreduce(V, torch, comm, send, recv, count, 20 if nbytes <= (64 << 20) else 4, 5)
        out.append({"bytes_per_rank": nbytes, "busbw_gbs": nbytes / t * bus_factor(N_RANKS) / 1e9,
                    "hbm_frac": 2 * N_RANKS * nbytes / t / 1e9 / hbm, "us": t * 1e6,
                    "graph_us": tg * 1e6, "graph_busbw_gbs": nbytes / tg * bus_factor(N_RANKS) / 1e9,
                    "graph_hbm_frac": 2 * N_RANKS * nbytes / tg / 1e9 / hbm})
        del send, recv
        torch.cuda.empty_cache()
    V.vcommDestroy(comm)
    return out


def sweep_collectives(torch, V, dev, hbm):
    """Reduce-scatter, all-gather, broadcast and all-to-all (fp32) against bytes per rank,
    1 KiB .. 1 GiB in powers of 4: eager and replayed from a CUDA graph.  Bytes per rank
    is the send size (RS, BC, A2A) or the receive size (AG); minimum bytes and bus factor
    as the planner reports them."""
    n = N_RANKS
    comm = V.vcommInit(n, 1, V.vProtoSimple)
    V.vcommSetAlgo(comm, "onepass")
    out = {}

    def calls(coll, send, recv, elems):
        if coll == "reduce_scatter":
            return lambda: V.vReduceScatter(send, recv, elems // n, torch.float32, "sum", comm)
        if coll == "allgather":
            return lambda: V.vAllGather(send, recv, elems // n, torch.float32, "sum", comm)
        if coll == "broadcast":
            return lambda: V.vBroadcast(send, recv, elems, torch.float32, "sum", 0, comm)
        return lambda: V.vAllToAll(send, recv, elems // n, torch.float32, "sum", comm)

    codes = {"reduce_scatter": V.vCollReduceScatter, "allgather": V.vCollAllGather,
             "broadcast": V.vCollBroadcast, "alltoall": V.vCollAllToAll}
    for coll in ("reduce_scatter", "allgather", "broadcast", "alltoall"):
        rows = []
        for k in range(11):
            nbytes = 1024 * 4 ** k
            elems = nbytes // 4                          # elements per rank of the big side
            small = elems // n
            send_elems = small if coll == "allgather" else elems
            recv_elems = small if coll == "reduce_scatter" else elems
            send = [torch.rand(send_elems, device=dev) for _ in range(n)]
            recv = [torch.empty(recv_elems, device=dev) for _ in range(n)]
            fn = calls(coll, send, recv, elems)
            count = small if coll in ("reduce_scatter", "allgather", "alltoall") else elems
            plan = V.vcommQueryPlan(comm, codes[coll], count, torch.float32, 32)
            steps = 200 if nbytes <= (1 << 20) else (50 if nbytes <= (64 << 20) else 10)
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                fn()
            b.record()
            torch.cuda.synchronize()
            t = a.elapsed_time(b) / 1e3 / steps
            g = torch.cuda.CUDAGraph()
            launches = 20 if nbytes <= (64 << 20) else 4
            with torch.cuda.graph(g):
                for _ in range(launches):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(5):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            tg = a.elapsed_time(b) / 1e3 / (5 * launches)
            rows.append({"bytes_per_rank": nbytes, "us": t * 1e6, "graph_us": tg * 1e6,
                         "busbw_gbs": nbytes / tg * plan["busFactor"] / 1e9,
                         "graph_hbm_frac": plan["minBytes"] / tg / 1e9 / hbm})
            del send, recv, g
            torch.cuda.empty_cache()
        out[coll] = rows
    V.vcommDestroy(comm)
    return out


RING_COLLS = ("allreduce", "reduce_scatter", "allgather", "broadcast")


def ring_call(V, torch, coll, comm, send, recv, nbytes, n):
    """(enqueue function, count argument, vColl_t) of one staged-ring collective whose
    bytes per rank are `nbytes` (the send size; the receive size for all-gather)."""
    elems = nbytes // 4
    if coll == "allreduce":
        s_, r_ = [x[:elems] for x in send], [x[:elems] for x in recv]
        return (lambda st=None: V.vAllReduce(s_, r_, elems, torch.float32, "sum", comm, st)), elems, V.vCollAllReduce
    if coll == "reduce_scatter":
        s_, r_ = [x[:elems] for x in send], [x[:elems // n] for x in recv]
        return (lambda st=None: V.vReduceScatter(s_, r_, elems // n, torch.float32, "sum", comm, st)), elems // n, \
            V.vCollReduceScatter
    if coll == "allgather":
        s_, r_ = [x[:elems // n] for x in send], [x[:elems] for x in recv]
        return (lambda st=None: V.vAllGather(s_, r_, elems // n, torch.float32, "sum", comm, st)), elems // n, \
            V.vCollAllGather
    s_, r_ = [x[:elems] for x in send], [x[:elems] for x in recv]
    return (lambda st=None: V.vBroadcast(s_, r_, elems, torch.float32, "sum", 0, comm, st)), elems, V.vCollBroadcast


def graph_us(torch, fn, launches, reps):
    """Device time of one call: `launches` calls captured into a CUDA graph, replayed
    `reps` times after one untimed replay (no host gaps between the kernels)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(launches):
            fn(torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) * 1e3 / (reps * launches)


def eager_us(torch, fn, warm, reps):
    """Time of one call from CUDA events around `reps` back-to-back calls after `warm`."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    st = torch.cuda.current_stream()
    a.record(st)
    for _ in range(reps):
        fn(st)
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps


def ring_sweep(torch, V, dev, channels=(1, 8, 32), max_bytes=1 << 30):
    """The staged ring (fp32 sum, 8 virtual ranks, the planner's default chunk) for
    all-reduce, reduce-scatter, all-gather and broadcast x Simple/LL/LL128 x channel counts
    x bytes per rank 1 KiB .. 1 GiB in powers of 4: device time (CUDA-graph replays up to
    4 MiB per rank, back-to-back eager calls above) beside the planner's predictedUs.  The
    data behind the planner's ring cost model."""
    n = N_RANKS
    top = max_bytes // 4
    send = [torch.rand(top, device=dev) for _ in range(n)]
    recv = [torch.empty(top, device=dev) for _ in range(n)]
    rows = []
    for proto, pname in ((V.vProtoSimple, "simple"), (V.vProtoLL, "ll"), (V.vProtoLL128, "ll128")):
        for ch in channels:
            comm = V.vcommInit(n, ch, proto)
            V.vcommSetAlgo(comm, "ring")
            for coll in RING_COLLS:
                nbytes = 1024
                while nbytes <= max_bytes:
                    fn, count, code = ring_call(V, torch, coll, comm, send, recv, nbytes, n)
                    try:
                        if nbytes <= (4 << 20):
                            t = graph_us(torch, fn, 20, 5)
                        else:
                            # Milliseconds per call: launch gaps do not matter, and an eager
                            # call skips the FIFO clearing a captured LL/LL128 transfer does
                            # before every replay.
                            t = eager_us(torch, fn, 2 if nbytes <= (64 << 20) else 1, 3 if nbytes <= (64 << 20) else 2)
                        pred = V.vcommQueryPlan(comm, code, count, torch.float32, 32)["predictedUs"]
                        rows.append([coll, pname, ch, nbytes, round(t, 2), round(pred, 2)])
                    except V.VcommError as e:
                        rows.append([coll, pname, ch, nbytes, None, str(e)])
                    nbytes *= 4
            V.vcommDestroy(comm)
    del send, recv
    torch.cuda.empty_cache()
    return {"columns": ["coll", "proto", "channels", "bytes_per_rank", "device_us", "model_us"],
            "n_ranks": n, "dtype": "f32", "op": "sum", "chunk": "planner default", "rows": rows}


def ring_grid(torch, V, send, recv, stream):
    """The staged ring all-reduce at 8 x 64 MiB fp32 for every protocol x channels
    {1, 8, 16, 32} x chunk bytes {128K .. 2M}: measured time (CUDA events, 3 calls after
    one) beside the planner's predictedUs.  Every cell gives the same bits."""
    rows = []
    for proto, pname in ((V.vProtoSimple, "simple"), (V.vProtoLL, "ll"), (V.vProtoLL128, "ll128")):
        for ch in (1, 8, 16, 32):
            comm = V.vcommInit(N_RANKS, ch, proto)
            V.vcommSetAlgo(comm, "ring")
            for chunk in (128 << 10, 256 << 10, 512 << 10, 1 << 20, 2 << 20):
                V.vcommSetChunkBytes(comm, chunk)
                try:
                    t = time_allreduce(V, torch, comm, send, recv, COUNT, 3, 1, stream)
                    pred = V.vcommQueryPlan(comm, V.vCollAllReduce, COUNT, torch.float32, 32)["predictedUs"]
                    rows.append([pname, ch, chunk, round(t * 1e6, 1), round(pred, 1),
                                 round(BYTES_PER_RANK / t * bus_factor(N_RANKS) / 1e9, 1)])
                except V.VcommError as e:
                    rows.append([pname, ch, chunk, None, str(e), None])
            V.vcommDestroy(comm)
    return {"columns": ["proto", "channels", "chunk_bytes", "measured_us", "model_us", "busbw_gbs"],
            "rows": rows}


def run_workloads(only=None):
    import torch

    from collective_communication_virtual_gb300 import build, vcomm as V
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    hbm, _ = peaks()
    print(json.dumps({"other_workloads": other_workloads(torch, V, dev, torch.cuda.current_stream(), hbm, only)}))
    return 0


def run_ring_sweep():
    """The staged ring's side measurements alone (the planner's calibration data)."""
    import torch

    from collective_communication_virtual_gb300 import build, vcomm as V
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    send = [torch.rand(COUNT, device=dev) for _ in range(N_RANKS)]
    recv = [torch.empty(COUNT, device=dev) for _ in range(N_RANKS)]
    grid = ring_grid(torch, V, send, recv, torch.cuda.current_stream())
    del send, recv
    torch.cuda.empty_cache()
    for name, data in (("ring_allreduce_chunk_channel_grid", grid), ("ring_sweep", ring_sweep(torch, V, dev))):
        print(json.dumps({"extra": name, "data": data}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side measurements (sweeps, grids, other workloads)")
    ap.add_argument("--workloads", action="store_true",
                    help="only time the other collectives (FSDP bucket, MoE dispatch, all-to-all, "
                         "reduce-scatter, all-gather, broadcast) and print them as one JSON line")
    ap.add_argument("--ring-sweep", action="store_true",
                    help="only time the staged ring's protocol x channel x size sweep and chunk grid")
    ap.add_argument("--only", default=None,
                    help="with --workloads: a comma-separated list of the workload names to run")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    sys.path.insert(0, ROOT)
    if args.impl == "reference":
        return run_reference(args)
    if args.workloads:
        return run_workloads(args.only)
    if args.ring_sweep:
        return run_ring_sweep()
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
