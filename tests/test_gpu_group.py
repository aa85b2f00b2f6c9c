"""Group batching: calls between vcommGroupStart and vcommGroupEnd run at the end, with
one-pass all-reduces of one type/op/stream fused into one launch.  Results must equal
the oracle (and so separate calls) bit for bit."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture()
def comm():
    c = V.vcommInit(8, 2, V.vProtoSimple)
    yield c
    V.vcommDestroy(c)


def test_group_of_mixed_all_reduces_matches_oracle(comm):
    n = 8
    cases = []
    V.vcommGroupStart(comm)
    for i, (count, dtype, op) in enumerate([(1, torch.float32, "sum"), (4099, torch.float32, "sum"),
                                            (100_003, torch.float32, "sum"), (65_536, torch.bfloat16, "max"),
                                            (7, torch.bfloat16, "max"), (33_333, torch.int32, "prod"),
                                            (12_345, torch.float32, "sum"), (1 << 20, torch.float16, "sum")]):
        xs = inputs.uniform_ranks(n, count, dtype, seed=i)
        send = to_dev(xs)
        recv = empty_dev(n, count, dtype)
        V.vAllReduce(send, recv, count, dtype, op, comm)
        cases.append((xs, op, send, recv))
    V.vcommGroupEnd(comm)
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(comm) == V.vSuccess
    for xs, op, _, recv in cases:
        assert_bits_equal(recv, oracle.allreduce(xs, op), f"group allreduce {xs[0].dtype} {op}")


def test_group_of_all_reduces_off_16_bytes(comm):
    # pointers one or three elements off a 16-byte boundary: the batched element path
    n = 8
    cases = []
    V.vcommGroupStart(comm)
    # items of one type and op fuse into one launch: fp32 sum, bf16 sum and int32 max pairs
    for i, (count, dtype, op, pad) in enumerate([(5, torch.float32, "sum", 1), (40_001, torch.float32, "sum", 1),
                                                 (33_333, torch.bfloat16, "sum", 3), (70_000, torch.bfloat16, "sum", 1),
                                                 (9_999, torch.int32, "max", 3), (257, torch.int32, "max", 1)]):
        xs = inputs.uniform_ranks(n, count, dtype, seed=40 + i)
        send = to_dev(xs, pad)
        recv = empty_dev(n, count, dtype, pad)
        V.vAllReduce(send, recv, count, dtype, op, comm)
        cases.append((xs, op, send, recv))           # the inputs must live until the group ends
    V.vcommGroupEnd(comm)
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(comm) == V.vSuccess
    for xs, op, _, recv in cases:
        assert_bits_equal(recv, oracle.allreduce(xs, op), f"group element path {xs[0].dtype} {op}")


def test_group_runs_nothing_before_end(comm):
    n, count = 8, 4096
    xs = inputs.uniform_ranks(n, count, torch.float32, 3)
    send = to_dev(xs)
    recv = empty_dev(n, count, torch.float32, fill=-1.0)
    V.vcommGroupStart(comm)
    V.vAllReduce(send, recv, count, torch.float32, "sum", comm)
    torch.cuda.synchronize()
    assert bool((recv[0] == -1.0).all())
    V.vcommGroupEnd(comm)
    torch.cuda.synchronize()
    assert_bits_equal(recv, oracle.allreduce(xs, "sum"), "after end")


def test_group_beyond_one_launch_and_with_other_collectives(comm):
    n = 8
    many = []
    V.vcommGroupStart(comm)
    V.vcommGroupStart(comm)                      # nested: only the outer end enqueues
    for i in range(1100):                        # more than one fused launch holds
        count = 1 + (i * 37) % 300
        xs = inputs.uniform_ranks(n, count, torch.float32, seed=1000 + i)
        send = to_dev(xs)
        recv = empty_dev(n, count, torch.float32)
        V.vAllReduce(send, recv, count, torch.float32, "sum", comm)
        many.append((xs, send, recv))      # the buffers must live until the group has run
    ag_in = inputs.uniform_ranks(n, 5000, torch.bfloat16, 9)
    ag_send = to_dev(ag_in)
    ag_recv = empty_dev(n, n * 5000, torch.bfloat16)
    V.vAllGather(ag_send, ag_recv, 5000, torch.bfloat16, "sum", comm)
    rs_in = inputs.uniform_ranks(n, n * 3000, torch.float32, 10)
    rs_send = to_dev(rs_in)
    rs_recv = empty_dev(n, 3000, torch.float32)
    V.vReduceScatter(rs_send, rs_recv, 3000, torch.float32, "min", comm)
    V.vcommGroupEnd(comm)                        # inner end: still recorded
    V.vcommGroupEnd(comm)
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(comm) == V.vSuccess
    for xs, _, recv in many:
        assert_bits_equal(recv, oracle.allreduce(xs, "sum"), "many")
    assert_bits_equal(ag_recv, oracle.allgather(ag_in), "group allgather")
    assert_bits_equal(rs_recv, oracle.reduce_scatter(rs_in, "min"), "group reduce-scatter")


def test_group_end_without_start_and_errors(comm):
    with pytest.raises(V.VcommError) as e:
        V.vcommGroupEnd(comm)
    assert e.value.code == V.vInvalidUsage
    x = [torch.zeros(16, device=DEV) for _ in range(8)]
    V.vcommGroupStart(comm)
    with pytest.raises(V.VcommError) as e:          # argument errors are reported at the call
        V.vAllReduce(x[:7] + [None], x, 16, torch.float32, "sum", comm)
    assert e.value.code == V.vInvalidArgument
    V.vcommGroupEnd(comm)


def test_ring_all_reduce_in_a_group_runs_unfused(comm):
    n, count = 8, 50_000
    V.vcommSetAlgo(comm, "ring")
    xs = inputs.uniform_ranks(n, count, torch.float16, 5)
    send = to_dev(xs)
    recv = empty_dev(n, count, torch.float16)
    V.vcommGroupStart(comm)
    V.vAllReduce(send, recv, count, torch.float16, "sum", comm)
    V.vcommGroupEnd(comm)
    torch.cuda.synchronize()
    V.vcommSetAlgo(comm, "auto")
    assert_bits_equal(recv, oracle.allreduce(xs, "sum"), "ring in group")


def test_group_captured_in_a_graph_replays_the_fused_launch(comm):
    # The work table rides in the launch's parameters, so a captured group replays with
    # its own table; new data written into the same buffers gives new, exact results.
    n, counts = 8, [4096, 1000, 77, 65_536, 3]
    bufs = [(empty_dev(n, c, torch.float32), empty_dev(n, c, torch.float32)) for c in counts]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        V.vcommGroupStart(comm)
        for (send, recv), c in zip(bufs, counts):
            V.vAllReduce(send, recv, c, torch.float32, "sum", comm)
        V.vcommGroupEnd(comm)
    for rep in range(2):
        xss = [inputs.uniform_ranks(n, c, torch.float32, seed=50 + 10 * rep + i) for i, c in enumerate(counts)]
        for (send, _), xs in zip(bufs, xss):
            for r in range(n):
                send[r].copy_(xs[r])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(comm) == V.vSuccess
        for (_, recv), xs in zip(bufs, xss):
            assert_bits_equal(recv, oracle.allreduce(xs, "sum"), f"captured group, replay {rep}")
