"""GPU parity of the rooted collectives (reduce to root, gather, scatter) against the
oracle, bit for bit: every type and op, several roots, ragged sizes, 32-byte, 16-byte
and element paths, in place."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, Comms, assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu

DTYPES = [torch.float32, torch.float16, torch.bfloat16, torch.int32]
OPS = ["sum", "prod", "min", "max"]


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def dname(d):
    return str(d).split(".")[1]


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_reduce_parity(comms, dtype, op):
    for n, count, root, pad in [(2, 1, 1, 0), (8, 100_003, 0, 0), (8, 1 << 20, 5, 0), (5, 33_333, 4, 0),
                                (8, 50_001, 3, 1), (8, 65_536, 7, 16 // torch.tensor([], dtype=dtype).element_size())]:
        xs = inputs.uniform_ranks(n, count, dtype, seed=count + root)
        send = to_dev(xs, pad)
        recv = [None] * n
        recv[root] = empty_dev(1, count, dtype, pad)[0]
        c = comms.get(n, 4)
        V.vReduce(send, recv, count, dtype, op, root, c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vSuccess
        assert_bits_equal([recv[root]], [oracle.reduce(xs, op, root)], f"reduce n={n} count={count} root={root}")


def test_reduce_in_place(comms):
    n, count, root = 8, 77_777, 6
    xs = inputs.uniform_ranks(n, count, torch.bfloat16, 2)
    send = to_dev(xs)
    recv = [None] * n
    recv[root] = send[root]
    c = comms.get(n, 2)
    V.vReduce(send, recv, count, torch.bfloat16, "sum", root, c)
    torch.cuda.synchronize()
    assert_bits_equal([send[root]], [oracle.reduce(xs, "sum", root)], "reduce in place")


@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_gather_parity(comms, dtype):
    for n, sc, root, pad in [(2, 1, 0, 0), (8, 4096, 3, 0), (8, 1 << 18, 7, 0), (5, 3001, 2, 0), (8, 10_000, 1, 1)]:
        xs = inputs.uniform_ranks(n, sc, dtype, seed=sc + n)
        send = to_dev(xs, pad)
        recv = [None] * n
        recv[root] = empty_dev(1, n * sc, dtype, pad)[0]
        c = comms.get(n, 3)
        V.vGather(send, recv, sc, dtype, root, c)
        torch.cuda.synchronize()
        assert_bits_equal([recv[root]], [oracle.gather(xs, root)], f"gather n={n} sc={sc} root={root}")


@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_scatter_parity(comms, dtype):
    for n, rc, root, pad in [(2, 1, 1, 0), (8, 4096, 0, 0), (8, 1 << 18, 4, 0), (7, 2999, 6, 0), (8, 10_000, 2, 1)]:
        src = inputs.uniform_ranks(1, n * rc, dtype, seed=rc)[0]
        send = [None] * n
        send[root] = to_dev([src], pad)[0]
        recv = empty_dev(n, rc, dtype, pad)
        c = comms.get(n, 3)
        V.vScatter(send, recv, rc, dtype, root, c)
        torch.cuda.synchronize()
        assert_bits_equal(recv, oracle.scatter(src, n, root), f"scatter n={n} rc={rc} root={root}")


def test_gather_then_scatter_in_place_round_trip(comms):
    n, sc, root = 8, 12_288, 3
    xs = inputs.uniform_ranks(n, sc, torch.float32, 4)
    big = torch.empty(n * sc, device=DEV)
    send = to_dev(xs)
    send[root] = big[root * sc:(root + 1) * sc]              # gather in place at the root
    send[root].copy_(xs[root].to(DEV))
    recv = [None] * n
    recv[root] = big
    c = comms.get(n, 1)
    V.vGather(send, recv, sc, torch.float32, root, c)
    torch.cuda.synchronize()
    assert_bits_equal([big], [torch.cat(xs)], "gather in place")
    out = empty_dev(n, sc, torch.float32)
    out[root] = big[root * sc:(root + 1) * sc]               # scatter in place at the root
    V.vScatter([None] * root + [big] + [None] * (n - root - 1), out, sc, torch.float32, root, c)
    torch.cuda.synchronize()
    assert_bits_equal(out, xs, "scatter in place")


def test_rooted_arguments_are_checked(comms):
    c = comms.get(4, 1)
    x = [torch.zeros(16, device=DEV) for _ in range(4)]
    for fn in (lambda: V.vReduce(x, x, 16, torch.float32, "sum", 4, c),
               lambda: V.vGather(x, x, 4, torch.float32, -1, c),
               lambda: V.vScatter(x, x, 4, torch.float32, 9, c),
               lambda: V.vReduce(x, [None] * 4, 16, torch.float32, "sum", 0, c),
               lambda: V.vScatter([None] * 4, x, 4, torch.float32, 0, c)):
        with pytest.raises(V.VcommError) as e:
            fn()
        assert e.value.code == V.vInvalidArgument
