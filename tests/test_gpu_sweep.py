"""The collective sweep on 8 ranks: all-reduce, reduce-scatter, all-gather and broadcast
(root 0), bytes per rank 1 KiB .. 1 GiB in powers of 4, fp32/fp16/bf16/int32, sum/prod/
min/max, one-pass and the staged ring with Simple, LL and LL128.

Up to 4 MiB per rank every (collective, type, op) cell is compared bit for bit with the
oracle, once per cell for all four variants.  At 16 and 64 MiB one type/op per
collective is compared in full.  At 256 MiB and 1 GiB the outputs are checked on the GPU
for properties that hold at any size (every rank's result identical; the copies equal
their sources) and sampled elements of the reductions are compared with the oracle."""
from __future__ import annotations

import os

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, Comms, assert_bits_equal, bits

pytestmark = pytest.mark.gpu

N = 8
NTHREADS = max(1, min(16, os.cpu_count() or 1))
DTYPES = [torch.float32, torch.float16, torch.bfloat16, torch.int32]
OPS = ["sum", "prod", "min", "max"]
VARIANTS = [("onepass", V.vProtoSimple), ("ring", V.vProtoSimple), ("ring", V.vProtoLL),
            ("ring", V.vProtoLL128)]
SIZES = [1024 * 4 ** k for k in range(11)]


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def esize(dt):
    return torch.tensor([], dtype=dt).element_size()


def ibits(t):
    """Raw bits of a device tensor, for exact comparison on the GPU."""
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


def run(comms, coll, algo, proto, send, recv, count, dt, op, channels=8):
    c = comms.get(N, channels, proto, algo, None)
    if coll == "ar":
        V.vAllReduce(send, recv, count, dt, op, c)
    elif coll == "rs":
        V.vReduceScatter(send, recv, count, dt, op, c)
    elif coll == "ag":
        V.vAllGather(send, recv, count, dt, op, c)
    else:
        V.vBroadcast(send, recv, count, dt, op, 0, c)
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(c) == V.vSuccess


def shapes(coll, nbytes, dt):
    """(send elements, recv elements, count argument) for `nbytes` per rank."""
    e = nbytes // esize(dt)
    if coll == "ar" or coll == "bc":
        return e, e, e
    if coll == "rs":
        return e, e // N, e // N
    return e // N, e, e // N             # all-gather: bytes per rank = receive size


def oracle_out(coll, xs, op):
    if coll == "ar":
        return oracle.allreduce(xs, op, nthreads=NTHREADS)
    if coll == "rs":
        return oracle.reduce_scatter(xs, op, nthreads=NTHREADS)
    if coll == "ag":
        return oracle.allgather(xs)
    return oracle.broadcast(xs, 0)


def sampled_expectation(xs, op, samples):
    """Expected reductions of sampled elements.  Sample s reads flat index e_s of every
    rank and is reduced in the ring order of block b_s (ranks b_s+1, ..., b_s).  One tiny
    reduce-scatter with S elements per block computes all of them: its block b, column s
    holds the sampled values, and output rank b's column s is then the reduction in that
    order."""
    S = len(samples)
    tiny = [torch.zeros(N * S, dtype=xs[0].dtype) for _ in range(N)]
    for s, (e, b) in enumerate(samples):
        for j in range(N):
            tiny[j][b * S + s] = xs[j][e]
    out = oracle.reduce_scatter(tiny, op)
    return torch.stack([out[b][s] for s, (e, b) in enumerate(samples)])


@pytest.mark.parametrize("coll", ["ar", "rs", "ag", "bc"])
def test_sweep_up_to_4MiB_every_cell(comms, coll):
    for nbytes in SIZES[:7]:
        for dt in DTYPES:
            ops = OPS if coll in ("ar", "rs") else ["sum"]
            ns, nr, cnt = shapes(coll, nbytes, dt)
            xs = inputs.uniform_ranks(N, ns, dt, seed=nbytes % 9973 + esize(dt))
            send = [x.to(DEV) for x in xs]
            for op in ops:
                want = oracle_out(coll, xs, op)
                for algo, proto in VARIANTS:
                    recv = [torch.empty(nr, dtype=dt, device=DEV) for _ in range(N)]
                    run(comms, coll, algo, proto, send, recv, cnt, dt, op)
                    assert_bits_equal(recv, want, f"{coll} {nbytes}B {dt} {op} {algo}/{proto}")


LARGE_CASES = {"ar": (torch.float32, "sum"), "rs": (torch.bfloat16, "max"),
               "ag": (torch.float16, "sum"), "bc": (torch.int32, "sum")}


@pytest.mark.parametrize("coll", ["ar", "rs", "ag", "bc"])
def test_sweep_16_and_64MiB_full_compare(comms, coll):
    dt, op = LARGE_CASES[coll]
    for nbytes in SIZES[7:9]:
        ns, nr, cnt = shapes(coll, nbytes, dt)
        xs = inputs.uniform_ranks(N, ns, dt, seed=7)
        want = oracle_out(coll, xs, op)
        send = [x.to(DEV) for x in xs]
        for algo, proto in VARIANTS:
            recv = [torch.empty(nr, dtype=dt, device=DEV) for _ in range(N)]
            run(comms, coll, algo, proto, send, recv, cnt, dt, op, channels=16)
            assert_bits_equal(recv, want, f"{coll} {nbytes}B {algo}/{proto}")
            del recv


@pytest.mark.parametrize("coll", ["ar", "rs", "ag", "bc"])
def test_sweep_256MiB_and_1GiB_properties_and_samples(comms, coll):
    dt, op = LARGE_CASES[coll]
    g = torch.Generator().manual_seed(99)
    for nbytes in SIZES[9:]:
        ns, nr, cnt = shapes(coll, nbytes, dt)
        xs = inputs.uniform_ranks(N, ns, dt, seed=11)
        send = [x.to(DEV) for x in xs]
        recv = [torch.empty(nr, dtype=dt, device=DEV) for _ in range(N)]
        for algo, proto in VARIANTS[:2] if nbytes > SIZES[9] else VARIANTS:
            for r_ in recv:
                r_.zero_()
            run(comms, coll, algo, proto, send, recv, cnt, dt, op, channels=32)
            if coll in ("ar", "bc"):
                for r in range(1, N):                      # every rank holds the same result
                    assert torch.equal(ibits(recv[r]), ibits(recv[0])), (coll, r)
            if coll == "bc":
                assert torch.equal(ibits(recv[0]), ibits(send[0]))
            if coll == "ag":
                for r in range(N):
                    for s in range(N):
                        assert torch.equal(ibits(recv[r][s * cnt:(s + 1) * cnt]), ibits(send[s])), (r, s)
            if coll in ("ar", "rs"):
                idx = torch.randint(0, ns, (256,), generator=g).tolist()
                if coll == "ar":
                    B = oracle.block_elems(ns, N, esize(dt))
                    samples = [(e, e // B) for e in idx]
                    got = torch.stack([recv[0][e].cpu() for e in idx])
                else:
                    samples = [(e, e // cnt) for e in idx]
                    got = torch.stack([recv[e // cnt][e % cnt].cpu() for e in idx])
                want = sampled_expectation(xs, op, samples)
                assert torch.equal(bits(got), bits(want)), (coll, nbytes, algo, proto)
        del send, recv, xs
        torch.cuda.empty_cache()
