"""GPU parity of the double-binary-tree all-reduce (vAlgoTree) against the oracle's tree
order, bit for bit: every type and op, rank counts with mirrored (even) and shifted (odd)
second trees, ragged sizes, 32-byte / 16-byte / element paths, in place, full size."""
from __future__ import annotations

import os

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import Comms, assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu
NTHREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def run_tree(comms, xs, op, pad=0, inplace=False):
    n, count, dt = len(xs), xs[0].numel(), xs[0].dtype
    send = to_dev(xs, pad)
    recv = send if inplace else empty_dev(n, count, dt, pad)
    c = comms.get(n, 1, V.vProtoSimple, "tree")
    V.vAllReduce(send, recv, count, dt, op, c)
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(c) == V.vSuccess
    return recv


@pytest.mark.parametrize("op", ["sum", "prod", "min", "max"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16, torch.int32],
                         ids=lambda d: str(d).split(".")[1])
def test_tree_allreduce_parity(comms, dtype, op):
    for n, count in [(2, 1), (3, 7), (8, 4099), (5, 33_333), (8, 100_003), (7, 65_536), (16, 20_000),
                     (2, 50_000), (4, 40_000), (4, 4_097), (16, 70_001)]:
        xs = inputs.uniform_ranks(n, count, dtype, seed=n * 31 + count)
        got = run_tree(comms, xs, op)
        assert_bits_equal(got, oracle.allreduce_tree(xs, op), f"tree n={n} count={count}")


def test_tree_paths_and_in_place(comms):
    xs = inputs.uniform_ranks(8, 50_001, torch.float32, 3)
    want = oracle.allreduce_tree(xs, "sum")
    assert_bits_equal(run_tree(comms, xs, "sum", pad=1), want, "element path")
    assert_bits_equal(run_tree(comms, xs, "sum", pad=4), want, "16-byte path")
    assert_bits_equal(run_tree(comms, xs, "sum", inplace=True), want, "in place")


def test_tree_allreduce_64MiB(comms):
    xs = inputs.uniform_ranks(8, 16 << 20, torch.float32, 1)
    want = oracle.allreduce_tree(xs, "sum", nthreads=NTHREADS)
    assert_bits_equal(run_tree(comms, xs, "sum"), want, "tree 64 MiB")
    # a different reduction order than the ring: some bits differ from vAllReduce's default
    ring = oracle.allreduce(xs, "sum", nthreads=NTHREADS)
    assert not torch.equal(want[0].view(torch.int32), ring[0].view(torch.int32))
