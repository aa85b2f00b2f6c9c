"""Refit the planner's cost-model constants on the GPU at hand.

The planner models a ring all-reduce as latency + bus bytes / bus rate per protocol and
channel count (the ring.cc form of the NCCL book, chapter 5), and the one-pass kernels as
latency + minimum HBM bytes / rate.  This script measures the anchor points through the
library -- an fp32 sum all-reduce over 8 virtual ranks, replayed from a CUDA graph, at
1 KiB per rank (latency) and 256 MiB per rank (rate), for 1, 8 and 32 channels -- and
prints the constants in the form `csrc/planner.cpp` declares them.

    python -m collective_communication_virtual_gb300.calibrate
"""
from __future__ import annotations

N_RANKS = 8
SMALL, LARGE = 1024, 256 << 20


def graph_time_us(torch, V, comm, send, recv, count, launches, reps):
    for _ in range(2):
        V.vAllReduce(send, recv, count, torch.float32, "sum", comm)
    torch.cuda.synchronize()
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
    return a.elapsed_time(b) * 1e3 / (reps * launches)


def main() -> None:
    import torch

    from collective_communication_virtual_gb300 import build, vcomm as V

    build.build()
    dev = torch.device("cuda:0")
    bufs = {}
    for nbytes in (SMALL, LARGE):
        count = nbytes // 4
        bufs[nbytes] = ([torch.rand(count, device=dev) for _ in range(N_RANKS)],
                        [torch.empty(count, device=dev) for _ in range(N_RANKS)], count)
    steps = 2 * (N_RANKS - 1)
    rows = []
    for proto, name in ((V.vProtoSimple, "Simple"), (V.vProtoLL, "LL"), (V.vProtoLL128, "LL128")):
        lat, rate = [], []
        for ch in (1, 8, 32):
            comm = V.vcommInit(N_RANKS, ch, proto)
            V.vcommSetAlgo(comm, "ring")
            send, recv, count = bufs[SMALL]
            t0 = graph_time_us(torch, V, comm, send, recv, count, 20, 5)
            send, recv, count = bufs[LARGE]
            t1 = graph_time_us(torch, V, comm, send, recv, count, 1, 2)
            V.vcommDestroy(comm)
            lat.append(t0)
            rate.append(LARGE * steps / N_RANKS / (t1 - t0))
        rows.append(f"    {{{{{lat[0]:.1f}, {lat[1]:.1f}, {lat[2]:.1f}}}, "
                    f"{{{rate[0]:.1f}, {rate[1]:.1f}, {rate[2]:.1f}}}}},   // {name}")
    comm = V.vcommInit(N_RANKS, 1, V.vProtoSimple)
    V.vcommSetAlgo(comm, "onepass")
    send, recv, count = bufs[SMALL]
    t0 = graph_time_us(torch, V, comm, send, recv, count, 20, 5)
    send, recv, count = bufs[LARGE]
    t1 = graph_time_us(torch, V, comm, send, recv, count, 4, 3)
    V.vcommDestroy(comm)
    print("const RingFit kRingFit[3] = {")
    print("\n".join(rows))
    print("};")
    print(f"const double kOnePassLatUs = {t0:.1f};")
    print(f"const double kOnePassBytesPerUs = {2 * N_RANKS * LARGE / (t1 - t0):.3e};")


if __name__ == "__main__":
    main()
