"""Refit the planner's ring cost model from measured staged-ring times.

The planner predicts a staged-ring collective of x bytes per rank over N ranks as
  ring steps (all-reduce, reduce-scatter, all-gather):  lat + f * min(x, knee) + max(0, x - knee) / rate
  broadcast chain:                                       lat + c * sqrt(x) + x / rate
for each (collective, protocol) at 1, 8 and 32 channels (interpolated in log2 of the
channel count, held flat beyond), with lat and the byte terms scaled from N = 8 by the
step count (the ring.cc form of the NCCL book, chapter 5: time = latency + bus bytes /
bus bandwidth, with LL and LL128 trading bandwidth for latency).  Below the knee a
transfer is one slot per step and every step pays for its bytes in turn (f, microseconds
per byte); above it the slots pipeline and the bytes cost 1 / rate; the broadcast's
square-root term is the pipeline fill of a chain whose slot count grows as sqrt(bytes)
(the planner's broadcast slot rule).

Input: the `ring_sweep` rows that `bench.py --ring-sweep` prints (device time of fp32 sum
over 8 ranks, default chunks, 1 KiB .. 1 GiB per rank in powers of 4), committed as
ring_timings_gb300.json.  Output: the table planner.cpp declares.

    python -m collective_communication_virtual_gb300.calibrate [timings.json]
"""
from __future__ import annotations

import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
DATA = os.path.join(HERE, "ring_timings_gb300.json")
COLLS = ("allreduce", "reduce_scatter", "allgather", "broadcast")
PROTOS = ("simple", "ll", "ll128")
CHANNELS = (1, 8, 32)


def load(path=DATA):
    with open(path) as f:
        d = json.load(f)
    cols = d["columns"]
    return [dict(zip(cols, r)) for r in d["rows"] if r[cols.index("device_us")] is not None]


def _lsq(cols, m):
    """Least squares on the relative error: minimise sum((cols . p) / m - 1)^2."""
    A = np.stack([c / m for c in cols], 1)
    p, *_ = np.linalg.lstsq(A, np.ones_like(m), rcond=None)
    return p


def fit_curve(coll, x, m):
    """(lat_us, bytes_per_us, third, us_per_mib_below_knee) for one (collective, protocol,
    channels) curve; third is the knee in bytes (ring steps) or the square-root coefficient
    (broadcast, whose last value is 0)."""
    x, m = np.asarray(x, float), np.asarray(m, float)
    one = np.ones_like(x)
    if coll == "broadcast":
        lat, c, inv = _lsq([one, np.sqrt(x), x], m)
        if c < 0 or inv <= 0:
            (lat, inv), c = _lsq([one, x], m), 0.0
        return float(lat), float(1.0 / inv), float(c), 0.0
    best = None
    for knee in [0.0] + [float(2 ** k) for k in range(10, 27)]:
        below, above = np.minimum(x, knee), np.maximum(0.0, x - knee)
        f = -1.0
        if knee > 0:
            lat, f, inv = _lsq([one, below, above], m)
        if f < 0:                      # no knee, or a negative slope below it: none
            (lat, inv), f = _lsq([one, above], m), 0.0
        if lat < 0 or inv <= 0:
            continue
        score = float(np.sum(((lat + f * below + inv * above) / m - 1.0) ** 2))
        if best is None or score < best[0]:
            best = (score, float(lat), float(1.0 / inv), knee, float(f) * (1 << 20))
    return best[1], best[2], best[3], best[4]


def fit(rows):
    table = {}
    for coll in COLLS:
        for proto in PROTOS:
            table[(coll, proto)] = []
            for ch in CHANNELS:
                pts = sorted((r["bytes_per_rank"], r["device_us"]) for r in rows
                             if r["coll"] == coll and r["proto"] == proto and r["channels"] == ch)
                table[(coll, proto)].append(fit_curve(coll, [p[0] for p in pts], [p[1] for p in pts]))
    return table


def cpp(table):
    out = ["const RingFit kRingFit[4][3] = {                         // calibrate.py prints these"]
    for coll in COLLS:
        out.append(f"    {{  // {coll}")
        for proto in PROTOS:
            f = table[(coll, proto)]
            lat = ", ".join(f"{v[0]:.2f}" for v in f)
            rate = ", ".join(f"{v[1]:.1f}" for v in f)
            third = ", ".join((f"{v[2]:.0f}" if coll != "broadcast" else f"{v[2]:.5f}") for v in f)
            below = ", ".join(f"{v[3]:.2f}" for v in f)
            out.append(f"        {{{{{lat}}}, {{{rate}}}, {{{third}}}, {{{below}}}}},   // {proto}")
        out.append("    },")
    out.append("};")
    return "\n".join(out)


def main() -> None:
    rows = load(sys.argv[1] if len(sys.argv) > 1 else DATA)
    table = fit(rows)
    print(cpp(table))
    errs = []
    for r in rows:
        lat, rate, third, below = table[(r["coll"], r["proto"])][CHANNELS.index(r["channels"])]
        x = r["bytes_per_rank"]
        if r["coll"] == "broadcast":
            pred = lat + third * math.sqrt(x) + x / rate
        else:
            pred = lat + below / (1 << 20) * min(x, third) + max(0.0, x - third) / rate
        errs.append(abs(pred / r["device_us"] - 1.0))
    print(f"// median relative error {float(np.median(errs)):.3f}, max {max(errs):.3f} over {len(errs)} points")


if __name__ == "__main__":
    main()
