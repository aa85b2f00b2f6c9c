"""The planner's ring cost model against the staged-ring times measured on GB300
(collective_communication_virtual_gb300/ring_timings_gb300.json: fp32 sum over 8 ranks,
default chunks, all-reduce / reduce-scatter / all-gather / broadcast x Simple / LL / LL128
x 1, 8, 32 channels x 1 KiB .. 1 GiB per rank).  The model has the ring.cc form of the
NCCL book, chapter 5 (latency + bytes / bandwidth per protocol and channel count), and
vProtoAuto picks the protocol it predicts fastest (ncclTuningCompute's minimum)."""
from __future__ import annotations

import json
import os
import statistics

import pytest

from collective_communication_virtual_gb300 import vcomm as V

DATA = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "collective_communication_virtual_gb300", "ring_timings_gb300.json")
COLL = {"allreduce": V.vCollAllReduce, "reduce_scatter": V.vCollReduceScatter,
        "allgather": V.vCollAllGather, "broadcast": V.vCollBroadcast}
PROTO = {"simple": V.vProtoSimple, "ll": V.vProtoLL, "ll128": V.vProtoLL128}
N = 8


def _rows():
    with open(DATA) as f:
        d = json.load(f)
    cols = d["columns"]
    return [dict(zip(cols, r)) for r in d["rows"] if r[cols.index("device_us")] is not None]


def _count(coll, nbytes):
    # the count argument of the call whose bytes per rank are nbytes (send size, or the
    # receive size for all-gather)
    elems = nbytes // 4
    return elems // N if coll in ("reduce_scatter", "allgather") else elems


def _plan(coll, proto, ch, nbytes):
    return V.vPlanCompute(nRanks=N, nChannels=ch, proto=proto, algo=V.vAlgoRing, coll=COLL[coll],
                          datatype=V.vFloat32, count=_count(coll, nbytes), aligned16=1, aligned32=1,
                          smCount=152)


def test_the_measured_table_covers_the_sweep():
    rows = _rows()
    assert len(rows) == 4 * 3 * 3 * 11
    assert {r["coll"] for r in rows} == set(COLL) and {r["proto"] for r in rows} == set(PROTO)
    assert sorted({r["bytes_per_rank"] for r in rows}) == [1024 * 4 ** k for k in range(11)]


def test_model_error_against_the_measurements():
    rows = _rows()
    errs = {}
    for r in rows:
        p = _plan(r["coll"], PROTO[r["proto"]], r["channels"], r["bytes_per_rank"])
        assert p.algo == V.vAlgoRing
        errs.setdefault((r["coll"], r["proto"]), []).append(abs(p.predictedUs / r["device_us"] - 1.0))
    every = [e for v in errs.values() for e in v]
    assert statistics.median(every) <= 0.05, statistics.median(every)
    for key, v in errs.items():
        assert statistics.median(v) <= 0.15, (key, statistics.median(v))
        assert max(v) <= 0.50, (key, max(v))


def test_auto_protocol_is_within_15_percent_of_the_best_measured():
    rows = _rows()
    meas = {}
    for r in rows:
        meas.setdefault((r["coll"], r["channels"], r["bytes_per_rank"]), {})[r["proto"]] = r["device_us"]
    names = {v: k for k, v in PROTO.items()}
    worst = 0.0
    for (coll, ch, nbytes), t in meas.items():
        p = _plan(coll, V.vProtoAuto, ch, nbytes)
        ratio = t[names[p.proto]] / min(t.values())
        worst = max(worst, ratio)
        assert ratio <= 1.15, (coll, ch, nbytes, names[p.proto], t)
    assert worst >= 1.0


@pytest.mark.parametrize("coll", list(COLL))
def test_model_scales_with_rank_and_channel_counts(coll):
    # latency grows with the step count, bandwidth terms with the bytes; more channels never
    # predict a slower large transfer
    small8 = _plan(coll, V.vProtoSimple, 8, 1024).predictedUs
    p16 = V.vPlanCompute(nRanks=16, nChannels=8, proto=V.vProtoSimple, algo=V.vAlgoRing, coll=COLL[coll],
                         datatype=V.vFloat32, count=_count(coll, 1024) if coll not in ("reduce_scatter", "allgather")
                         else 1024 // 4 // 16, aligned16=1, smCount=152).predictedUs
    assert p16 > small8
    big = [_plan(coll, V.vProtoSimple, ch, 1 << 30).predictedUs for ch in (1, 4, 8, 16, 32, 64)]
    assert all(b >= c for b, c in zip(big, big[1:])), big


def test_calibration_recovers_known_curves():
    # the fit on curves drawn from the model's own forms, at the sweep's sizes, gives their
    # parameters back: ring steps (two slopes around a knee) and the broadcast chain
    from collective_communication_virtual_gb300 import calibrate
    xs = [1024 * 4 ** k for k in range(11)]
    lat, f_mib, knee, rate = 30.0, 40.0, float(1 << 20), 150_000.0
    m = [lat + f_mib / (1 << 20) * min(x, knee) + max(0.0, x - knee) / rate for x in xs]
    got = calibrate.fit_curve("allreduce", xs, m)
    assert got[0] == pytest.approx(lat, rel=1e-6) and got[1] == pytest.approx(rate, rel=1e-6)
    assert got[2] == knee and got[3] == pytest.approx(f_mib, rel=1e-6)
    c = 0.02
    m = [lat + c * x ** 0.5 + x / rate for x in xs]
    got = calibrate.fit_curve("broadcast", xs, m)
    assert got[0] == pytest.approx(lat, rel=1e-6) and got[1] == pytest.approx(rate, rel=1e-6)
    assert got[2] == pytest.approx(c, rel=1e-6) and got[3] == 0.0
