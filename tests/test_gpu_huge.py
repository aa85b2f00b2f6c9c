"""Buffers of more than 2^31 elements per rank, so that every element index, block offset
and tile number past 32 bits is exercised: all-reduce, reduce-scatter (vector and
element paths), all-gather (vector and element paths) and all-to-all, two ranks.

The inputs come from ``inputs.index_pattern``, a function of (rank, index) alone, so the
device fills multi-GiB buffers and the host rebuilds exactly the sampled elements.  The
expected values of the sampled elements come from the oracle: the reductions through a
tiny reduce-scatter whose block b holds the samples reduced in block b's ring order, the
copies by rebuilding the source element.  Peak device memory per test is at most 32 GiB."""
from __future__ import annotations

import random

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, bits

pytestmark = pytest.mark.gpu

N = 2
BIG = 1 << 31


def fill(rank, count, dt):
    t = torch.empty(count, dtype=dt, device=DEV)
    step = 1 << 27
    for s in range(0, count, step):
        m = min(step, count - s)
        t[s:s + m] = inputs.index_pattern(rank, s, m, dt, DEV)
    return t


def host(rank, e, dt):
    return inputs.index_pattern(rank, e, 1, dt)[0]


def picks(count, edges, k=48, seed=0):
    rng = random.Random(seed)
    out = {e for e in edges if 0 <= e < count}
    out |= {rng.randrange(count) for _ in range(k)}
    return sorted(out)


def ring_expect(samples, dt, op):
    """Sample (e, b): element e of every rank reduced in the ring order of block b."""
    S = len(samples)
    tiny = [torch.zeros(N * S, dtype=dt) for _ in range(N)]
    for s, (e, b) in enumerate(samples):
        for j in range(N):
            tiny[j][b * S + s] = host(j, e, dt)
    out = oracle.reduce_scatter(tiny, op)
    return torch.stack([out[b][s] for s, (e, b) in enumerate(samples)])


def gather_at(t, idx):
    return t[torch.tensor(idx, dtype=torch.int64, device=DEV)].cpu()


@pytest.fixture
def comm():
    c = V.vcommInit(N, 1, V.vProtoSimple)
    V.vcommSetAlgo(c, "onepass")
    yield c
    V.vcommDestroy(c)
    torch.cuda.empty_cache()


def ok(c):
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(c) == V.vSuccess


def test_allreduce_past_2_31_elements(comm):
    dt, count = torch.float32, BIG + (1 << 20) + 3
    send = [fill(r, count, dt) for r in range(N)]
    recv = [torch.empty(count, dtype=dt, device=DEV) for _ in range(N)]
    V.vAllReduce(send, recv, count, dt, "sum", comm)
    ok(comm)
    B = oracle.block_elems(count, N, 4)
    idx = picks(count, [0, 1, B - 1, B, BIG - 1, BIG, BIG + 1, count - 1])
    want = ring_expect([(e, e // B) for e in idx], dt, "sum")
    for r in range(N):
        assert torch.equal(bits(gather_at(recv[r], idx)), bits(want)), r


@pytest.mark.parametrize("rc", [BIG + 16, BIG + 5], ids=["vector", "element"])
def test_reduce_scatter_past_2_31_elements(comm, rc):
    dt = torch.bfloat16
    send = [fill(r, N * rc, dt) for r in range(N)]
    recv = [torch.empty(rc, dtype=dt, device=DEV) for _ in range(N)]
    V.vReduceScatter(send, recv, rc, dt, "max", comm)
    ok(comm)
    for r in range(N):
        idx = picks(rc, [0, 1, BIG - 1, BIG, rc - 1], seed=r)
        want = ring_expect([(r * rc + t, r) for t in idx], dt, "max")
        assert torch.equal(bits(gather_at(recv[r], idx)), bits(want)), r


@pytest.mark.parametrize("sc", [BIG + 8, BIG + 3], ids=["vector", "element"])
def test_allgather_past_2_31_elements(comm, sc):
    dt = torch.bfloat16
    send = [fill(r, sc, dt) for r in range(N)]
    recv = [torch.empty(N * sc, dtype=dt, device=DEV) for _ in range(N)]
    V.vAllGather(send, recv, sc, dt, "sum", comm)
    ok(comm)
    for r in range(N):
        idx = picks(N * sc, [0, sc - 1, sc, sc + 1, BIG, sc + BIG, N * sc - 1], seed=r)
        want = torch.stack([host(e // sc, e % sc, dt) for e in idx])
        assert torch.equal(bits(gather_at(recv[r], idx)), bits(want)), r


def test_alltoall_past_2_31_elements(comm):
    dt, c = torch.bfloat16, BIG + 1
    send = [fill(r, N * c, dt) for r in range(N)]
    recv = [torch.empty(N * c, dtype=dt, device=DEV) for _ in range(N)]
    V.vAllToAll(send, recv, c, dt, "sum", comm)
    ok(comm)
    for j in range(N):
        idx = picks(N * c, [0, c - 1, c, BIG, c + BIG, N * c - 1], seed=10 + j)
        # recv[j][i*c + t] = send[i][j*c + t]
        want = torch.stack([host(e // c, j * c + e % c, dt) for e in idx])
        assert torch.equal(bits(gather_at(recv[j], idx)), bits(want)), j
