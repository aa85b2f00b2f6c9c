"""vAllReduceNoAlloc: the ring all-reduce for callers that cannot allocate device memory
(graph capture, allocator callbacks, runtimes that own all memory).  It must give the
same bits as vAllReduce, call after call, with its fixed scratch array reused.

This file is collected last on purpose, so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process, where its
first call does the per-device set-up."""
from __future__ import annotations

import pytest
import torch

from collective_communication_virtual_gb300 import build, inputs, vcomm as V

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("proto", [V.vProtoSimple, V.vProtoLL, V.vProtoLL128], ids=["simple", "ll", "ll128"])
def test_no_alloc_matches_vAllReduce_twice(proto):
    build.build()
    dev = torch.device("cuda:0")
    n, channels, count = 8, 4, 300_007
    comm = V.vcommInit(n, channels, proto)
    try:
        V.vcommSetAlgo(comm, "ring")
        for call, (dtype, op, seed) in enumerate([(torch.float32, "sum", 1), (torch.bfloat16, "max", 2)]):
            xs = [x.to(dev) for x in inputs.uniform_ranks(n, count, dtype, seed + 10 * proto)]
            want = [torch.empty_like(x) for x in xs]
            V.vAllReduce(xs, want, count, dtype, op, comm)
            got = [torch.full_like(x, 7) for x in xs]
            V.vAllReduceNoAlloc(xs, got, count, dtype, op, n, channels, proto)
            torch.cuda.synchronize()
            assert V.vcommGetAsyncError(comm) == V.vSuccess
            for r in range(n):
                assert torch.equal(got[r].view(torch.int16 if dtype != torch.float32 else torch.int32),
                                   want[r].view(torch.int16 if dtype != torch.float32 else torch.int32)), \
                    (call, r)
    finally:
        V.vcommDestroy(comm)


def test_no_alloc_refuses_rings_beyond_its_array():
    build.build()
    x = [torch.zeros(64, device="cuda:0") for _ in range(16)]
    with pytest.raises(V.VcommError) as e:
        V.vAllReduceNoAlloc(x, x, 64, torch.float32, "sum", 16, 8, V.vProtoSimple)   # 128 FIFOs > 64
    assert e.value.code == V.vInvalidArgument
    with pytest.raises(V.VcommError) as e:
        V.vAllReduceNoAlloc(x[:1], x[:1], 64, torch.float32, "sum", 1, 1, V.vProtoSimple)
    assert e.value.code == V.vInvalidArgument
