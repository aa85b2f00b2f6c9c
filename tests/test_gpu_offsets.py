"""Every rank's buffer at its own offset from a 16-byte boundary, bit for bit against the
oracle.  Equal offsets let the element paths build 16-byte vectors (aligned to the
outputs, cut from the inputs); unequal ones must fall back to element copies and
element reductions.  Covers all-reduce, reduce-scatter, all-gather, broadcast, all-to-all,
gather and scatter for 2- and 4-byte types, ragged counts."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, Comms, assert_bits_equal

pytestmark = pytest.mark.gpu

N = 4
PADS = {"same": [1, 1, 1, 1], "mixed": [0, 1, 2, 3], "mixed2": [3, 0, 5, 2]}
DTYPES = [torch.bfloat16, torch.float32]


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def place(xs, pads):
    """Device copies, buffer r starting pads[r] elements into its own allocation."""
    out = []
    for x, p in zip(xs, pads):
        big = torch.empty(x.numel() + p + 8, dtype=x.dtype, device=DEV)
        v = big[p:p + x.numel()]
        v.copy_(x)
        out.append(v)
    return out


def blank(counts, dt, pads):
    return [torch.full((c + p + 8,), -7, dtype=dt, device=DEV)[p:p + c] for c, p in zip(counts, pads)]


def ok(c):
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(c) == V.vSuccess


@pytest.mark.parametrize("dt", DTYPES, ids=["bf16", "fp32"])
@pytest.mark.parametrize("send_pads", list(PADS), ids=lambda k: "send_" + k)
@pytest.mark.parametrize("recv_pads", list(PADS), ids=lambda k: "recv_" + k)
def test_allreduce_and_reduce_scatter(comms, dt, send_pads, recv_pads):
    c = comms.get(N, 2, V.vProtoSimple, "onepass")
    sp, rp = PADS[send_pads], PADS[recv_pads]
    count = 50_003
    xs = inputs.uniform_ranks(N, count, dt, seed=sum(sp) * 7 + sum(rp))
    recv = blank([count] * N, dt, rp)
    V.vAllReduce(place(xs, sp), recv, count, dt, "sum", c)
    ok(c)
    assert_bits_equal(recv, oracle.allreduce(xs, "sum"), f"all-reduce {send_pads}/{recv_pads}")
    rc = 12_345
    ys = inputs.uniform_ranks(N, N * rc, dt, seed=sum(sp) * 11 + sum(rp))
    recv = blank([rc] * N, dt, rp)
    V.vReduceScatter(place(ys, sp), recv, rc, dt, "max", c)
    ok(c)
    assert_bits_equal(recv, oracle.reduce_scatter(ys, "max"), f"reduce-scatter {send_pads}/{recv_pads}")


@pytest.mark.parametrize("dt", DTYPES, ids=["bf16", "fp32"])
@pytest.mark.parametrize("send_pads", list(PADS), ids=lambda k: "send_" + k)
@pytest.mark.parametrize("recv_pads", list(PADS), ids=lambda k: "recv_" + k)
def test_copies(comms, dt, send_pads, recv_pads):
    c = comms.get(N, 1, V.vProtoSimple, "onepass")
    sp, rp = PADS[send_pads], PADS[recv_pads]
    sc = 20_001
    xs = inputs.uniform_ranks(N, sc, dt, seed=3 + sum(sp) + 5 * sum(rp))
    recv = blank([N * sc] * N, dt, rp)
    V.vAllGather(place(xs, sp), recv, sc, dt, "sum", c)
    ok(c)
    assert_bits_equal(recv, oracle.allgather(xs), f"all-gather {send_pads}/{recv_pads}")
    recv = blank([sc] * N, dt, rp)
    V.vBroadcast(place(xs, sp), recv, sc, dt, "sum", 2, c)
    ok(c)
    assert_bits_equal(recv, oracle.broadcast(xs, 2), f"broadcast {send_pads}/{recv_pads}")
    blk = 3_001
    ys = inputs.uniform_ranks(N, N * blk, dt, seed=4 + sum(sp) + 5 * sum(rp))
    recv = blank([N * blk] * N, dt, rp)
    V.vAllToAll(place(ys, sp), recv, blk, dt, "sum", c)
    ok(c)
    assert_bits_equal(recv, oracle.alltoall(ys), f"all-to-all {send_pads}/{recv_pads}")
    root = 1
    out = blank([N * sc], dt, [rp[root]])[0]
    V.vGather(place(xs, sp), [out if r == root else None for r in range(N)], sc, dt, root, c)
    ok(c)
    assert_bits_equal([out], [oracle.gather(xs, root)], f"gather {send_pads}/{recv_pads}")
    src = inputs.uniform_ranks(1, N * blk, dt, seed=9)[0]
    send = [place([src], [sp[root]])[0] if r == root else None for r in range(N)]
    recv = blank([blk] * N, dt, rp)
    V.vScatter(send, recv, blk, dt, root, c)
    ok(c)
    assert_bits_equal(recv, oracle.scatter(src, N, root), f"scatter {send_pads}/{recv_pads}")
