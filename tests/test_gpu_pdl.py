"""Programmatic dependent launch keeps stream order: a chain of collectives whose every
step reads the previous step's output, launched back to back without synchronizing,
equals the oracle's chain bit for bit, with and without the launch attribute; a torch
kernel between two collectives is waited for as usual."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu


def _chain(comm, xs, n, count):
    """AR x -> y, AR y -> z (reads y), RS z -> w (reads z), AG w -> v (reads w), AR in place
    on v: each launch depends on the one before it."""
    send = to_dev(xs)
    y = empty_dev(n, count, torch.float32)
    z = empty_dev(n, count, torch.float32)
    w = empty_dev(n, count // n, torch.float32)
    v = empty_dev(n, count, torch.float32)
    V.vAllReduce(send, y, count, torch.float32, "sum", comm)
    V.vAllReduce(y, z, count, torch.float32, "max", comm)
    V.vReduceScatter(z, w, count // n, torch.float32, "sum", comm)
    V.vAllGather(w, v, count // n, torch.float32, "sum", comm)
    V.vAllReduce(v, v, count, torch.float32, "min", comm)
    torch.cuda.synchronize()
    return y, z, w, v


@pytest.mark.parametrize("pdl", ["1", "0"])
def test_dependent_chain_matches_the_oracle(monkeypatch, pdl):
    monkeypatch.setenv("VCOMM_PDL", pdl)
    n, count = 8, 8 * 300_000
    comm = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        xs = inputs.uniform_ranks(n, count, torch.float32, 77)
        y, z, w, v = _chain(comm, xs, n, count)
        oy = oracle.allreduce(xs, "sum")
        oz = oracle.allreduce(oy, "max")
        ow = oracle.reduce_scatter(oz, "sum")
        ov = oracle.allreduce(oracle.allgather(ow), "min")
        assert_bits_equal(y, oy, "AR")
        assert_bits_equal(z, oz, "AR of AR")
        assert_bits_equal(w, ow, "RS")
        assert_bits_equal(v, ov, "AR in place of AG")
        assert V.vcommGetAsyncError(comm) == V.vSuccess
    finally:
        V.vcommDestroy(comm)


def test_torch_kernel_between_collectives_is_waited_for():
    n, count = 8, 1 << 20
    comm = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        xs = inputs.uniform_ranks(n, count, torch.float32, 5)
        send = to_dev(xs)
        y = empty_dev(n, count, torch.float32)
        V.vAllReduce(send, y, count, torch.float32, "sum", comm)
        for t in y:
            t.mul_(0.5)                     # torch kernels writing the next call's input
        z = empty_dev(n, count, torch.float32)
        V.vAllReduce(y, z, count, torch.float32, "sum", comm)
        torch.cuda.synchronize()
        half = [t * 0.5 for t in oracle.allreduce(xs, "sum")]
        assert_bits_equal(z, oracle.allreduce(half, "sum"), "AR after torch kernel")
    finally:
        V.vcommDestroy(comm)
