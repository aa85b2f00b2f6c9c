"""Seeded random sweep of GPU parity against the oracle, bit for bit.

Each case draws a collective, rank count, element count, data type, op, root, pointer
misalignment, algorithm, protocol and channel count from a fixed-seed generator, runs it
through the C ABI and compares every output with the oracle.  The cases are small (the
oracle finishes each in milliseconds) but they reach combinations the hand-written tests
do not: odd rank counts with rings and trees, one-element blocks, more channels than
elements, every protocol on misaligned buffers."""
from __future__ import annotations

import random

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import Comms, assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.float16, torch.bfloat16, torch.int32]
OPS = ["sum", "prod", "min", "max"]
PROTOS = [V.vProtoSimple, V.vProtoLL, V.vProtoLL128]
COLLS = ["allreduce", "allreduce", "allreduce", "reduce_scatter", "rs_scale_cast", "allgather", "broadcast",
         "alltoall", "alltoallv", "reduce", "gather", "scatter"]
N_CASES = 240


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def draw(case: int) -> dict:
    rng = random.Random(0x5EED0000 + case)
    coll = rng.choice(COLLS)
    staged = coll in ("allreduce", "reduce_scatter", "rs_scale_cast", "allgather", "broadcast")
    algo = "onepass"
    if coll == "allreduce":
        algo = rng.choice(["onepass", "ring", "tree", "auto"])
    elif staged:
        algo = rng.choice(["onepass", "ring", "auto"])
    n = rng.choice([1, 2, 3, 4, 5, 6, 7, 8, 8, 8, 11, 16] + ([] if algo == "ring" else [24, 64]))
    big = rng.random() < 0.2
    count = rng.randint(0, 70_000 if big else 3_000)
    dtype = rng.choice(DTYPES)
    if coll == "rs_scale_cast":
        dtype = rng.choice([torch.float32, torch.float16, torch.bfloat16])
    return {
        "coll": coll, "algo": algo, "n": n, "count": count, "dtype": dtype,
        "op": "sum" if coll == "rs_scale_cast" else rng.choice(OPS),
        "root": rng.randrange(n), "pad": rng.choice([0, 0, 0, 1, 3]),
        "proto": rng.choice(PROTOS), "channels": rng.choice([1, 1, 2, 3, 4, 8]),
        "chunk": rng.choice([None, 4096, 65536]), "seed": case,
    }


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_case_matches_oracle(comms, case):
    run_case(comms, case)


# The engines that are not the default stay selectable; the first cases run again under
# each (the switches are read when a communicator is created).
@pytest.mark.parametrize("env", [{"VCOMM_GRID": "persistent"}, {"VCOMM_COPY_TMA": "1"}, {"VCOMM_PDL": "0"}],
                         ids=["persistent_grid", "tma_fanout", "no_pdl"])
@pytest.mark.parametrize("case", range(0, N_CASES, 4))
def test_random_case_with_other_engines(monkeypatch, env, case):
    for name, value in env.items():
        monkeypatch.setenv(name, value)
    local = Comms()
    try:
        run_case(local, case)
    finally:
        local.close()


def run_case(comms, case):
    k = draw(case)
    n, count, dt, op, root, pad = k["n"], k["count"], k["dtype"], k["op"], k["root"], k["pad"]
    c = comms.get(n, k["channels"], k["proto"], k["algo"], chunk=k["chunk"])
    what = f"case {case}: {k}"
    coll = k["coll"]
    if coll == "allreduce":
        xs = inputs.uniform_ranks(n, count, dt, k["seed"])
        recv = empty_dev(n, count, dt, pad)
        V.vAllReduce(to_dev(xs, pad), recv, count, dt, op, c)
        want = oracle.allreduce_tree(xs, op) if k["algo"] == "tree" else oracle.allreduce(xs, op)
    elif coll in ("reduce_scatter", "rs_scale_cast"):
        rc = count // max(n, 1) // 4 + (count % 5)
        xs = inputs.uniform_ranks(n, n * rc, dt, k["seed"])
        if coll == "reduce_scatter":
            recv = empty_dev(n, rc, dt, pad)
            V.vReduceScatter(to_dev(xs, pad), recv, rc, dt, op, c)
            want = oracle.reduce_scatter(xs, op)
        else:
            scale = 1.0 / n
            recv = empty_dev(n, rc, torch.float32, pad)
            V.vReduceScatterScaleCast(to_dev(xs, pad), recv, rc, dt, "sum", torch.float32, scale, c)
            want = oracle.reduce_scatter_scale(xs, "sum", scale)
    elif coll == "allgather":
        sc = count // max(n, 1) + 1
        xs = inputs.uniform_ranks(n, sc, dt, k["seed"])
        recv = empty_dev(n, n * sc, dt, pad)
        V.vAllGather(to_dev(xs, pad), recv, sc, dt, "sum", c)
        want = oracle.allgather(xs)
    elif coll == "broadcast":
        xs = inputs.uniform_ranks(n, count, dt, k["seed"])
        send = to_dev(xs, pad)
        send = [s if r == root else None for r, s in enumerate(send)]
        recv = empty_dev(n, count, dt, pad)
        V.vBroadcast(send, recv, count, dt, "sum", root, c)
        want = oracle.broadcast(xs, root)
    elif coll == "alltoall":
        blk = count // max(n * n, 1) + 1
        xs = inputs.uniform_ranks(n, n * blk, dt, k["seed"])
        recv = empty_dev(n, n * blk, dt, pad)
        V.vAllToAll(to_dev(xs, pad), recv, blk, dt, "sum", c)
        want = oracle.alltoall(xs)
    elif coll == "alltoallv":
        g = torch.Generator().manual_seed(k["seed"])
        counts = torch.randint(0, 1 + count // max(n, 1) // 2, (n, n), generator=g, dtype=torch.int32)
        counts[torch.rand((n, n), generator=g) < 0.25] = 0
        sd = (torch.cumsum(counts, 1) - counts).to(torch.int32)
        rd = (torch.cumsum(counts, 0) - counts).t().contiguous().to(torch.int32)
        recv_elems = [int(v) for v in counts.sum(0)]
        xs = [inputs.uniform_ranks(1, int(counts[i].sum()), dt, k["seed"] * 64 + i)[0] for i in range(n)]
        recv = [empty_dev(1, e, dt, pad)[0] for e in recv_elems]
        for t in recv:
            t.zero_()
        V.vAllToAllv(to_dev(xs, pad), recv, *[t.cuda() for t in (counts, sd, rd)], dt, c)
        want = oracle.alltoallv(xs, counts, sd, rd, recv_elems)
    elif coll == "reduce":
        xs = inputs.uniform_ranks(n, count, dt, k["seed"])
        out = empty_dev(1, count, dt, pad)[0]
        recv = [out if r == root else None for r in range(n)]
        V.vReduce(to_dev(xs, pad), recv, count, dt, op, root, c)
        recv, want = [out], [oracle.reduce(xs, op, root)]
    elif coll == "gather":
        sc = count // max(n, 1) + 1
        xs = inputs.uniform_ranks(n, sc, dt, k["seed"])
        out = empty_dev(1, n * sc, dt, pad)[0]
        recv = [out if r == root else None for r in range(n)]
        V.vGather(to_dev(xs, pad), recv, sc, dt, root, c)
        recv, want = [out], [oracle.gather(xs, root)]
    else:  # scatter
        rc = count // max(n, 1) + 1
        src = inputs.uniform_ranks(1, n * rc, dt, k["seed"])[0]
        send = [to_dev([src], pad)[0] if r == root else None for r in range(n)]
        recv = empty_dev(n, rc, dt, pad)
        V.vScatter(send, recv, rc, dt, root, c)
        want = oracle.scatter(src, n, root)
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(c) == V.vSuccess, what
    assert_bits_equal(recv, want, what)
