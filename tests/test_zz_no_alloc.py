"""vAllReduceNoAlloc: the ring all-reduce for callers that cannot allocate device memory
(allocator or memory-pool callbacks that must not re-enter the allocator, runtimes that
hand out all device memory themselves).  It must give the same bits as vAllReduce, and
as the CPU oracle, call after call, with its fixed scratch array reused.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process, where its
first call does the per-device set-up."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import build, inputs, vcomm as V

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


def _check(n, channels, count, proto, calls):
    """Each call: vAllReduceNoAlloc against vAllReduce on the same communicator settings
    and against the oracle, bit for bit."""
    dev = torch.device("cuda:0")
    comm = V.vcommInit(n, channels, proto)
    try:
        V.vcommSetAlgo(comm, "ring")
        for call, (dtype, op, seed) in enumerate(calls):
            host = inputs.uniform_ranks(n, count, dtype, seed)
            xs = [x.to(dev) for x in host]
            want = [torch.empty_like(x) for x in xs]
            V.vAllReduce(xs, want, count, dtype, op, comm)
            got = [torch.full_like(x, 7) for x in xs]
            V.vAllReduceNoAlloc(xs, got, count, dtype, op, n, channels, proto)
            torch.cuda.synchronize()
            assert V.vcommGetAsyncError(comm) == V.vSuccess
            ref = oracle.allreduce(host, op)
            for r in range(n):
                g = got[r].cpu()
                assert torch.equal(_bits(g), _bits(want[r].cpu())), ("vAllReduce", call, r)
                assert torch.equal(_bits(g), _bits(ref[r])), ("oracle", call, r)
    finally:
        V.vcommDestroy(comm)


@pytest.mark.parametrize("proto", [V.vProtoSimple, V.vProtoLL, V.vProtoLL128], ids=["simple", "ll", "ll128"])
def test_no_alloc_matches_vAllReduce_and_the_oracle_twice(proto):
    build.build()
    _check(8, 4, 300_007, proto, [(torch.float32, "sum", 1 + 10 * proto), (torch.bfloat16, "max", 2 + 10 * proto)])


def test_no_alloc_at_its_largest_ring():
    # 8 ranks x 8 channels = 64 (channel, rank) FIFOs, the most the array holds, with an
    # odd count; two calls in a row
    build.build()
    _check(8, 8, 1_000_003, V.vProtoLL128, [(torch.float32, "sum", 41), (torch.float16, "prod", 42)])


def test_no_alloc_refuses_rings_beyond_its_array():
    build.build()
    x = [torch.zeros(64, device="cuda:0") for _ in range(16)]
    with pytest.raises(V.VcommError) as e:
        V.vAllReduceNoAlloc(x, x, 64, torch.float32, "sum", 16, 8, V.vProtoSimple)   # 128 FIFOs > 64
    assert e.value.code == V.vInvalidArgument
    with pytest.raises(V.VcommError) as e:
        V.vAllReduceNoAlloc(x[:1], x[:1], 64, torch.float32, "sum", 1, 1, V.vProtoSimple)
    assert e.value.code == V.vInvalidArgument
