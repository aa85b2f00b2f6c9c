"""The staged ring's protocols under skewed timing: with the jitter test hook every thread
sleeps for pseudo-random times where a producer publishes a slot (Simple: before its
counter; LL: between 16-byte units; LL128: between lines and before the release flag) and where
a consumer starts one.  Consumers then see slots half written, flags ahead of or behind
their neighbours, and FIFOs full or empty at other moments than usual.  Every result must
still equal the oracle bit for bit."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu

PROTOS = [V.vProtoSimple, V.vProtoLL, V.vProtoLL128]


@pytest.mark.parametrize("proto", PROTOS, ids=["simple", "ll", "ll128"])
@pytest.mark.parametrize("n,channels", [(4, 1), (8, 2)])
def test_ring_results_do_not_depend_on_timing(proto, n, channels):
    c = V.vcommInit(n, channels, proto)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommSetChunkBytes(c, 16384)              # 4 KiB slots: many slots per transfer
        V.vcommSetTimeoutMs(c, 20000)
        V.vcommTestSetJitterNs(c, 3000)
        for dt, op, count in ((torch.float32, "sum", 100_003), (torch.bfloat16, "max", 65_536),
                              (torch.int32, "prod", 7_777)):
            xs = inputs.uniform_ranks(n, count, dt, seed=n * 100 + count)
            recv = empty_dev(n, count, dt)
            V.vAllReduce(to_dev(xs), recv, count, dt, op, c)
            torch.cuda.synchronize()
            assert V.vcommGetAsyncError(c) == V.vSuccess
            assert_bits_equal(recv, oracle.allreduce(xs, op), f"jittered ring all-reduce {dt} {op}")
        rc = 9_001
        xs = inputs.uniform_ranks(n, n * rc, torch.float16, seed=5)
        recv = empty_dev(n, rc, torch.float16)
        V.vReduceScatter(to_dev(xs), recv, rc, torch.float16, "sum", c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vSuccess
        assert_bits_equal(recv, oracle.reduce_scatter(xs, "sum"), "jittered ring reduce-scatter")
        xs = inputs.uniform_ranks(n, rc, torch.float32, seed=6)
        recv = empty_dev(n, n * rc, torch.float32)
        V.vAllGather(to_dev(xs), recv, rc, torch.float32, "sum", c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vSuccess
        assert_bits_equal(recv, oracle.allgather(xs), "jittered ring all-gather")
        # the hook off again: the same communicator keeps its results
        V.vcommTestSetJitterNs(c, 0)
        xs = inputs.uniform_ranks(n, 4_099, torch.float32, seed=7)
        recv = empty_dev(n, 4_099, torch.float32)
        V.vAllReduce(to_dev(xs), recv, 4_099, torch.float32, "sum", c)
        torch.cuda.synchronize()
        assert_bits_equal(recv, oracle.allreduce(xs, "sum"), "ring all-reduce after jitter")
    finally:
        V.vcommDestroy(c)


@pytest.mark.parametrize("proto", PROTOS, ids=["simple", "ll", "ll128"])
def test_ring_large_slots_do_not_depend_on_timing(proto):
    # 1 MiB chunks: 256 KiB slots, so LL128 runs its whole-line steps (four lines per lane
    # group) and Simple its full rounds under the same random sleeps
    n = 4
    c = V.vcommInit(n, 1, proto)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommSetChunkBytes(c, 1 << 20)
        V.vcommSetTimeoutMs(c, 20000)
        V.vcommTestSetJitterNs(c, 2000)
        for dt, op, count in ((torch.float32, "sum", 1_200_000), (torch.bfloat16, "min", 2_400_016)):
            xs = inputs.uniform_ranks(n, count, dt, seed=11 + count)
            recv = empty_dev(n, count, dt)
            V.vAllReduce(to_dev(xs), recv, count, dt, op, c)
            torch.cuda.synchronize()
            assert V.vcommGetAsyncError(c) == V.vSuccess
            assert_bits_equal(recv, oracle.allreduce(xs, op), f"jittered ring all-reduce, large slots, {dt}")
    finally:
        V.vcommDestroy(c)


def test_jitter_hook_reaches_the_kernels():
    # sleeps of up to 200 us at every slot make the ring measurably slower (a sleep lasts
    # anywhere from 0 to about twice its request, so the check leaves wide room); the
    # limits hold
    n, count = 8, 65_536
    c = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        with pytest.raises(V.VcommError):
            V.vcommTestSetJitterNs(c, 2_000_000)
        V.vcommSetAlgo(c, "ring")
        V.vcommSetChunkBytes(c, 16384)
        send = to_dev(inputs.uniform_ranks(n, count, torch.float32, seed=8))
        recv = empty_dev(n, count, torch.float32)

        def timed():
            V.vAllReduce(send, recv, count, torch.float32, "sum", c)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            V.vAllReduce(send, recv, count, torch.float32, "sum", c)
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b)

        plain = timed()
        V.vcommTestSetJitterNs(c, 200_000)
        jittered = timed()
        V.vcommTestSetJitterNs(c, 0)
        assert jittered > 1.5 * plain, (plain, jittered)
        assert V.vcommGetAsyncError(c) == V.vSuccess
    finally:
        V.vcommDestroy(c)
