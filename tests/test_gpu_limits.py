"""The interface at its limits, bit for bit against the oracle: the largest rank count (64)
on the staged ring with every protocol, the largest channel count (64), ragged counts;
and a staged ring too large to be co-resident, which is refused with vInvalidUsage before
anything is launched or allocated (the error table of the NCCL-style interface: a
protocol forced where the staged kernel cannot run).  The communicator stays usable."""
from __future__ import annotations

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, Comms, assert_bits_equal, empty_dev, to_dev

pytestmark = pytest.mark.gpu

PROTOS = [V.vProtoSimple, V.vProtoLL, V.vProtoLL128]
PROTO_IDS = ["simple", "ll", "ll128"]


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def _ok(c):
    torch.cuda.synchronize()
    assert V.vcommGetAsyncError(c) == V.vSuccess


@pytest.mark.parametrize("proto", PROTOS, ids=PROTO_IDS)
@pytest.mark.parametrize("channels", [1, 2])
def test_ring_with_64_ranks(comms, proto, channels):
    n = 64
    c = comms.get(n, channels, proto, "ring")
    for dt, op, count in ((torch.float32, "sum", 100_003), (torch.bfloat16, "max", 4_099),
                          (torch.int32, "prod", 64)):
        xs = inputs.uniform_ranks(n, count, dt, seed=640 + count)
        recv = empty_dev(n, count, dt)
        V.vAllReduce(to_dev(xs), recv, count, dt, op, c)
        _ok(c)
        assert_bits_equal(recv, oracle.allreduce(xs, op), f"ring all-reduce N=64 {dt} {op} {count}")
    rc = 1_001
    xs = inputs.uniform_ranks(n, n * rc, torch.float16, seed=641)
    recv = empty_dev(n, rc, torch.float16)
    V.vReduceScatter(to_dev(xs), recv, rc, torch.float16, "min", c)
    _ok(c)
    assert_bits_equal(recv, oracle.reduce_scatter(xs, "min"), "ring reduce-scatter N=64")
    xs = inputs.uniform_ranks(n, rc, torch.float32, seed=642)
    recv = empty_dev(n, n * rc, torch.float32)
    V.vAllGather(to_dev(xs), recv, rc, torch.float32, "sum", c)
    _ok(c)
    assert_bits_equal(recv, oracle.allgather(xs), "ring all-gather N=64")
    xs = inputs.uniform_ranks(n, 777, torch.float32, seed=643)
    recv = empty_dev(n, 777, torch.float32)
    V.vBroadcast(to_dev(xs), recv, 777, torch.float32, "sum", 63, c)
    _ok(c)
    assert_bits_equal(recv, oracle.broadcast(xs, 63), "ring broadcast N=64 root 63")


@pytest.mark.parametrize("proto", PROTOS, ids=PROTO_IDS)
def test_ring_with_64_channels(comms, proto):
    # 8 ranks x 64 channels = 512 co-resident CTAs; a ragged count leaves the last
    # channels of every block short or empty
    n = 8
    c = comms.get(n, 64, proto, "ring")
    for dt, count in ((torch.float32, 70_001), (torch.float16, 1_000_003)):
        xs = inputs.uniform_ranks(n, count, dt, seed=650 + count)
        recv = empty_dev(n, count, dt)
        V.vAllReduce(to_dev(xs), recv, count, dt, "sum", c)
        _ok(c)
        assert_bits_equal(recv, oracle.allreduce(xs, "sum"), f"ring 64 channels {dt} {count}")


@pytest.mark.parametrize("proto", [V.vProtoLL, V.vProtoLL128], ids=["ll", "ll128"])
def test_ring_too_large_to_be_coresident_is_refused(proto):
    # 64 ranks x 64 channels with 1M fp32 elements per rank: 4096 CTAs of 128 threads,
    # more threads than the device holds at once, so the cooperative ring cannot run
    n, count = 64, 1 << 20
    c = V.vcommInit(n, 64, proto)
    try:
        V.vcommSetAlgo(c, "ring")
        p = V.vcommQueryPlan(c, V.vCollAllReduce, count, torch.float32, 32)
        props = torch.cuda.get_device_properties(0)
        per_sm = getattr(props, "max_threads_per_multi_processor", 2048)
        assert p["algo"] == V.vAlgoRing
        assert p["gridCtas"] * p["threadsPerCta"] > props.multi_processor_count * per_sm
        # real buffers of the full size (in place), so the call is valid in every other way
        bufs = [torch.full((count,), float(r), device=DEV) for r in range(n)]
        with pytest.raises(V.VcommError) as e:
            V.vAllReduce(bufs, bufs, count, torch.float32, "sum", c)
        assert e.value.code == V.vInvalidUsage
        _ok(c)
        for r in range(n):                          # nothing ran
            assert torch.equal(bufs[r], torch.full((count,), float(r), device=DEV))
        # the same communicator runs the one-pass kernel
        V.vcommSetAlgo(c, "onepass")
        xs = inputs.uniform_ranks(n, 5_003, torch.float32, seed=660)
        recv = empty_dev(n, 5_003, torch.float32)
        V.vAllReduce(to_dev(xs), recv, 5_003, torch.float32, "sum", c)
        _ok(c)
        assert_bits_equal(recv, oracle.allreduce(xs, "sum"), "one-pass after a refused ring")
    finally:
        V.vcommDestroy(c)


@pytest.mark.parametrize("coll", ["allreduce", "reduce_scatter", "allgather", "alltoall"])
def test_onepass_with_64_ranks_ragged(comms, coll):
    n = 64
    c = comms.get(n, 3, V.vProtoSimple, "onepass")
    dt = torch.bfloat16
    if coll == "allreduce":
        xs = inputs.uniform_ranks(n, 123_457, dt, seed=670)
        recv = empty_dev(n, 123_457, dt, 1)
        V.vAllReduce(to_dev(xs, 1), recv, 123_457, dt, "sum", c)
        want = oracle.allreduce(xs, "sum")
    elif coll == "reduce_scatter":
        xs = inputs.uniform_ranks(n, n * 997, dt, seed=671)
        recv = empty_dev(n, 997, dt)
        V.vReduceScatter(to_dev(xs), recv, 997, dt, "prod", c)
        want = oracle.reduce_scatter(xs, "prod")
    elif coll == "allgather":
        xs = inputs.uniform_ranks(n, 1_003, dt, seed=672)
        recv = empty_dev(n, n * 1_003, dt, 3)
        V.vAllGather(to_dev(xs, 3), recv, 1_003, dt, "sum", c)
        want = oracle.allgather(xs)
    else:
        xs = inputs.uniform_ranks(n, n * 33, dt, seed=673)
        recv = empty_dev(n, n * 33, dt)
        V.vAllToAll(to_dev(xs), recv, 33, dt, "sum", c)
        want = oracle.alltoall(xs)
    _ok(c)
    assert_bits_equal(recv, want, f"one-pass {coll} N=64")
