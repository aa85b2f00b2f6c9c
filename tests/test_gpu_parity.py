"""GPU parity: every collective through the C ABI against the CPU oracle, bit for bit.

Sizes span several CTAs, channels, chunks and FIFO slots and end on ragged tails; the
full-size workloads (64 MiB fp32 all-reduce over 8 ranks, the 25 MiB bf16 FSDP bucket,
the MoE dispatch) are compared element by element as well, with the oracle on all host
cores.  Floating-point results are compared as raw bits (the order-matched oracle makes
them exact); NaN results, where a test makes them, are compared as "is NaN".
"""
from __future__ import annotations

import os
import time

import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from collective_communication_virtual_gb300 import vcomm as V
from tests.gpu_util import DEV, Comms, assert_bits_equal, bits, empty_dev, to_dev

pytestmark = pytest.mark.gpu

NTHREADS = max(1, min(16, os.cpu_count() or 1))
DTYPES = [torch.float32, torch.float16, torch.bfloat16, torch.int32]
OPS = ["sum", "prod", "min", "max"]
VARIANTS = [("onepass", V.vProtoSimple), ("ring", V.vProtoSimple), ("ring", V.vProtoLL),
            ("ring", V.vProtoLL128)]
VID = ["onepass", "ring-simple", "ring-ll", "ring-ll128"]
SMALL_CHUNK = 16 * 1024            # ring: many chunks and slots even for small buffers


def dname(d):
    return str(d).split(".")[1]


@pytest.fixture(scope="module")
def comms():
    c = Comms()
    yield c
    c.close()


def _sync_ok(c):
    torch.cuda.synchronize()
    err = V.vcommGetAsyncError(c)
    assert err == V.vSuccess, f"async error {V.RESULT_NAMES.get(err, err)}"


def _inputs(n, count, dtype, seed):
    if dtype == torch.int32:
        return inputs.uniform_ranks(n, count, dtype, seed)
    return inputs.uniform_ranks(n, count, dtype, seed)


def run_allreduce(comms, xs, op, algo, proto, channels=1, chunk=SMALL_CHUNK, pad=0, inplace=False):
    n, count, dt = len(xs), xs[0].numel(), xs[0].dtype
    send = to_dev(xs, pad)
    recv = send if inplace else empty_dev(n, count, dt, pad)
    c = comms.get(n, channels, proto, algo, chunk)
    V.vAllReduce(send, recv, count, dt, op, c)
    _sync_ok(c)
    return recv


# ---------------------------------------------------------------------------------------
# The small correctness workload: 4 ranks x 1024 fp32 (4 KiB), sum, 1 channel, Simple
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ["onepass", "ring"])
def test_allreduce_4_ranks_4KiB(comms, algo):
    xs = inputs.uniform_ranks(4, 1024, torch.float32, 0)
    got = run_allreduce(comms, xs, "sum", algo, V.vProtoSimple, chunk=None)
    assert_bits_equal(got, oracle.allreduce(xs, "sum"), f"allreduce {algo}")


# ---------------------------------------------------------------------------------------
# All-reduce: dtypes x ops x algorithms/protocols x rank counts, ragged sizes
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_allreduce_parity(comms, dtype, op, variant):
    algo, proto = variant
    for n, count in [(2, 1), (3, 7), (8, 4099), (5, 33_333), (8, 100_003)]:
        xs = _inputs(n, count, dtype, seed=n * 1000 + count)
        got = run_allreduce(comms, xs, op, algo, proto)
        assert_bits_equal(got, oracle.allreduce(xs, op), f"allreduce n={n} count={count}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
def test_allreduce_channels_and_chunks_give_same_bits(comms, variant):
    algo, proto = variant
    xs = inputs.uniform_ranks(8, 1 << 20, torch.float32, 1)        # 4 MiB per rank
    want = oracle.allreduce(xs, "sum", nthreads=NTHREADS)
    for channels in (1, 8, 16, 32):
        for chunk in ((128 << 10, 2 << 20) if algo == "ring" else (None,)):
            got = run_allreduce(comms, xs, "sum", algo, proto, channels=channels, chunk=chunk)
            assert_bits_equal(got, want, f"channels={channels} chunk={chunk}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
def test_allreduce_unaligned_and_inplace(comms, variant):
    algo, proto = variant
    for dtype in (torch.float32, torch.bfloat16):
        xs = inputs.uniform_ranks(8, 50_001, dtype, 7)
        want = oracle.allreduce(xs, "sum")
        assert_bits_equal(run_allreduce(comms, xs, "sum", algo, proto, pad=1), want, "unaligned")
        # 16-byte but not 32-byte aligned buffers take the 16-byte vector path
        assert_bits_equal(run_allreduce(comms, xs, "sum", algo, proto, pad=16 // xs[0].element_size()),
                          want, "16-byte aligned")
        assert_bits_equal(run_allreduce(comms, xs, "sum", algo, proto, inplace=True), want, "in place")


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16], ids=dname)
def test_special_values(comms, dtype):
    """NaN, +-inf, +-0, subnormals and large exponent gaps through every variant."""
    g = torch.Generator().manual_seed(5)
    n, count = 4, 4096
    fin = torch.finfo(dtype)
    pool = torch.tensor([0.0, -0.0, float("inf"), float("-inf"), float("nan"), fin.tiny, -fin.tiny,
                         fin.tiny / 4, fin.max, -fin.max, 1.0, -1.0, 2.0 ** -10, 3.0, 1e-3],
                        dtype=torch.float32).to(dtype)
    xs = [pool[torch.randint(0, pool.numel(), (count,), generator=g)] for _ in range(n)]
    for op in OPS:
        want = oracle.allreduce(xs, op)
        for algo, proto in VARIANTS:
            got = run_allreduce(comms, xs, op, algo, proto)
            for r in range(n):
                gr, wr = got[r].cpu(), want[r]
                nan = torch.isnan(wr.float())
                assert torch.equal(torch.isnan(gr.float()), nan), (op, algo, proto)
                assert torch.equal(bits(gr)[~nan], bits(wr)[~nan]), (op, algo, proto)


def test_allreduce_guard_bands(comms):
    """Writes stay inside the receive buffers: canaries around them survive."""
    n, count, pad = 8, 10_007, 64
    xs = inputs.uniform_ranks(n, count, torch.float32, 12)
    for algo, proto in VARIANTS:
        c = comms.get(n, 4, proto, algo, SMALL_CHUNK)
        send = to_dev(xs)
        bigs = [torch.full((count + 2 * pad,), -7.0, device=DEV) for _ in range(n)]
        recv = [b[pad:pad + count] for b in bigs]
        V.vAllReduce(send, recv, count, torch.float32, "sum", c)
        _sync_ok(c)
        for b in bigs:
            assert bool((b[:pad] == -7.0).all()) and bool((b[pad + count:] == -7.0).all()), (algo, proto)
        assert_bits_equal(recv, oracle.allreduce(xs, "sum"), f"{algo}/{proto}")


# ---------------------------------------------------------------------------------------
# Reduce-scatter (+ fused scale / cast epilogue)
# ---------------------------------------------------------------------------------------

def run_rs(comms, xs, op, algo, proto, rc, out_dtype=None, scale=None, pad=0, inplace=False, channels=2):
    n, dt = len(xs), xs[0].dtype
    send = to_dev(xs, pad)
    odt = out_dtype or dt
    if inplace:
        recv = [s[r * rc:(r + 1) * rc] for r, s in enumerate(send)]
    else:
        recv = empty_dev(n, rc, odt, pad)
    c = comms.get(n, channels, proto, algo, SMALL_CHUNK)
    if scale is None:
        V.vReduceScatter(send, recv, rc, dt, op, c)
    else:
        V.vReduceScatterScaleCast(send, recv, rc, dt, op, odt, scale, c)
    _sync_ok(c)
    return recv


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_reduce_scatter_parity(comms, dtype, op, variant):
    algo, proto = variant
    for n, rc in [(2, 1), (3, 5), (8, 4096), (7, 3001), (8, 12_345)]:
        xs = _inputs(n, n * rc, dtype, seed=31 * n + rc)
        got = run_rs(comms, xs, op, algo, proto, rc)
        assert_bits_equal(got, oracle.reduce_scatter(xs, op), f"rs n={n} rc={rc}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32], ids=dname)
def test_reduce_scatter_scale_cast(comms, dtype, variant):
    algo, proto = variant
    n = 8
    for rc in (4096, 3001):
        xs = inputs.normal_ranks(n, n * rc, 1e-3, dtype, 2)
        for out in {torch.float32, dtype}:
            got = run_rs(comms, xs, "sum", algo, proto, rc, out_dtype=out, scale=1.0 / n)
            want = oracle.reduce_scatter_scale(xs, "sum", 1.0 / n, out)
            assert_bits_equal(got, want, f"rs scale/cast {dtype}->{out} rc={rc}")
        got = run_rs(comms, xs, "sum", algo, proto, rc, out_dtype=torch.float32, scale=1.0 / 3)
        assert_bits_equal(got, oracle.reduce_scatter_scale(xs, "sum", 1.0 / 3, torch.float32), "scale 1/3")


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
def test_reduce_scatter_unaligned_and_inplace(comms, variant):
    algo, proto = variant
    n, rc = 8, 5000
    xs = inputs.uniform_ranks(n, n * rc, torch.bfloat16, 4)
    want = oracle.reduce_scatter(xs, "sum")
    assert_bits_equal(run_rs(comms, xs, "sum", algo, proto, rc, pad=1), want, "unaligned")
    assert_bits_equal(run_rs(comms, xs, "sum", algo, proto, rc, inplace=True), want, "in place")
    xs = inputs.uniform_ranks(n, n * 4099, torch.float32, 4)        # odd block: element path
    assert_bits_equal(run_rs(comms, xs, "max", algo, proto, 4099), oracle.reduce_scatter(xs, "max"), "odd")


@pytest.mark.parametrize("n", [2, 3, 4, 8])
@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_reduce_scatter_ragged_warp_tiles(comms, n, dtype):
    # Ragged blocks (rc * esz not a multiple of 16) of several warp tiles: the one-pass
    # path reduces 16-byte vectors that follow the inputs, tile by tile, and realigns the
    # stores to the outputs through shuffles; the head and tail elements, the tile edges
    # (lane 31, the last vector of a tile) and a channel split all land on these sizes.
    esz = torch.empty((), dtype=dtype).element_size()
    for rc, channels in ((5 * 32 * 4 * (16 // esz) + 3, 1), (3 * 32 * 4 * (16 // esz) + 1, 2)):
        assert (rc * esz) % 16 != 0
        xs = _inputs(n, n * rc, dtype, seed=97 * n + rc)
        for op in ("sum", "max"):
            got = run_rs(comms, xs, op, "onepass", V.vProtoSimple, rc, channels=channels)
            assert_bits_equal(got, oracle.reduce_scatter(xs, op), f"ragged rs n={n} rc={rc} {op}")
        if dtype in (torch.float16, torch.bfloat16):
            got = run_rs(comms, xs, "sum", "onepass", V.vProtoSimple, rc, out_dtype=torch.float32,
                         scale=1.0 / n, channels=channels)
            assert_bits_equal(got, oracle.reduce_scatter_scale(xs, "sum", 1.0 / n, torch.float32),
                              f"ragged rs scale/cast n={n} rc={rc}")
        # send and receive buffers one element off 16 bytes: other head and output offsets
        got = run_rs(comms, xs, "sum", "onepass", V.vProtoSimple, rc, pad=1, channels=channels)
        assert_bits_equal(got, oracle.reduce_scatter(xs, "sum"), f"ragged rs padded n={n} rc={rc}")


# ---------------------------------------------------------------------------------------
# All-gather, broadcast
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_allgather_parity(comms, dtype, variant):
    algo, proto = variant
    for n, sc, pad, inplace in [(2, 1, 0, False), (8, 4096, 0, False), (5, 3001, 0, False),
                                (8, 12_347, 1, False), (8, 8192, 0, True)]:
        xs = _inputs(n, sc, dtype, seed=sc + n)
        if inplace:
            recv = empty_dev(n, n * sc, dtype)
            send = [recv[r][r * sc:(r + 1) * sc] for r in range(n)]
            for r in range(n):
                send[r].copy_(xs[r].to(DEV))
        else:
            send = to_dev(xs, pad)
            recv = empty_dev(n, n * sc, dtype, pad)
        c = comms.get(n, 3, proto, algo, SMALL_CHUNK)
        V.vAllGather(send, recv, sc, dtype, "sum", c)
        _sync_ok(c)
        assert_bits_equal(recv, oracle.allgather(xs), f"allgather n={n} sc={sc} pad={pad} inplace={inplace}")


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=dname)
def test_broadcast_parity(comms, dtype, variant):
    algo, proto = variant
    for n, count, root, pad in [(2, 1, 1, 0), (8, 65_536, 0, 0), (8, 100_001, 5, 0), (3, 7777, 2, 1)]:
        xs = _inputs(n, count, dtype, seed=count + root)
        send = [None] * n
        send[root] = to_dev([xs[root]], pad)[0]
        recv = empty_dev(n, count, dtype, pad)
        c = comms.get(n, 2, proto, algo, SMALL_CHUNK)
        V.vBroadcast(send, recv, count, dtype, "sum", root, c)
        _sync_ok(c)
        assert_bits_equal(recv, oracle.broadcast(xs, root), f"broadcast n={n} count={count} root={root}")
        # in place at the root, and idempotent: broadcasting the result again changes nothing
        V.vBroadcast(recv, recv, count, dtype, "sum", root, c)
        _sync_ok(c)
        assert_bits_equal(recv, oracle.broadcast(xs, root), "broadcast again")


# ---------------------------------------------------------------------------------------
# All-to-all (uniform and variable)
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
def test_alltoall_parity(comms, dtype):
    for n, c_, pad in [(2, 1, 0), (8, 4096, 0), (5, 777, 0), (8, 5003, 1)]:
        xs = _inputs(n, n * c_, dtype, seed=c_)
        send = to_dev(xs, pad)
        recv = empty_dev(n, n * c_, dtype, pad)
        c = comms.get(n, 4)
        V.vAllToAll(send, recv, c_, dtype, "sum", c)
        _sync_ok(c)
        want = oracle.alltoall(xs)
        assert_bits_equal(recv, want, f"alltoall n={n} c={c_}")
        # applying it twice gives back the input
        back = empty_dev(n, n * c_, dtype)
        V.vAllToAll(recv, back, c_, dtype, "sum", c)
        _sync_ok(c)
        assert_bits_equal(back, xs, "alltoall twice")


def _a2av(comms, send_cpu, counts, sd, rd, recv_elems, dtype, pad=0):
    n = len(send_cpu)
    send = to_dev(send_cpu, pad)
    recv = [torch.zeros(int(e) + pad, dtype=dtype, device=DEV)[pad:] for e in recv_elems]
    tabs = [t.to(torch.int32).contiguous().to(DEV) for t in (counts, sd, rd)]
    c = comms.get(n, 1)
    V.vAllToAllv(send, recv, *tabs, dtype, c)
    _sync_ok(c)
    return recv


def test_alltoallv_small_moe(comms):
    send, counts, sd, rd, recv_elems = inputs.moe_dispatch(n_ranks=8, tokens=256, hidden=64)
    got = _a2av(comms, send, counts, sd, rd, recv_elems, torch.bfloat16)
    assert_bits_equal(got, oracle.alltoallv(send, counts, sd, rd, recv_elems), "alltoallv")
    got = _a2av(comms, send, counts, sd, rd, recv_elems, torch.bfloat16, pad=1)
    assert_bits_equal(got, oracle.alltoallv(send, counts, sd, rd, recv_elems), "alltoallv unaligned")


def test_alltoallv_odd_blocks_and_empty(comms):
    n = 5
    g = torch.Generator().manual_seed(9)
    counts = torch.randint(0, 3000, (n, n), generator=g)
    counts[1, 3] = 0
    counts[2, :] = 0
    sd = torch.zeros_like(counts)
    sd[:, 1:] = torch.cumsum(counts, 1)[:, :-1]
    rd = torch.zeros_like(counts)
    rd[:, 1:] = torch.cumsum(counts.t(), 1)[:, :-1]
    recv_elems = counts.sum(0).tolist()
    send = [torch.randint(-100, 100, (int(counts[i].sum()) + 1,), generator=g, dtype=torch.int32)
            for i in range(n)]
    got = _a2av(comms, send, counts, sd, rd, recv_elems, torch.int32)
    assert_bits_equal(got, oracle.alltoallv(send, counts, sd, rd, recv_elems), "alltoallv odd")


# ---------------------------------------------------------------------------------------
# Degenerate cases
# ---------------------------------------------------------------------------------------

def test_count_zero_and_single_rank(comms):
    c = comms.get(4, 1)
    dummy = [torch.empty(0, device=DEV) for _ in range(4)]
    V.vAllReduce(dummy, dummy, 0, torch.float32, "sum", c)
    V.vReduceScatter(dummy, dummy, 0, torch.float32, "sum", c)
    V.vAllGather(dummy, dummy, 0, torch.float32, "sum", c)
    _sync_ok(c)
    xs = inputs.uniform_ranks(1, 12_345, torch.bfloat16, 3)
    for algo in ("onepass", "ring"):
        got = run_allreduce(comms, xs, "prod", algo, V.vProtoSimple)
        assert_bits_equal(got, xs, f"single rank {algo}")


def test_invalid_arguments_launch_nothing(comms):
    c = comms.get(4, 1)
    x = [torch.zeros(16, device=DEV) for _ in range(4)]
    with pytest.raises(V.VcommError) as e:
        V.vAllReduce(x[:3] + [None], x, 16, torch.float32, "sum", c)
    assert e.value.code == V.vInvalidArgument
    with pytest.raises(V.VcommError) as e:
        V.vAllReduce(x, x, 16, 9, "sum", c)
    assert e.value.code == V.vInvalidArgument
    with pytest.raises(V.VcommError) as e:
        V.vBroadcast(x, x, 16, torch.float32, "sum", 4, c)
    assert e.value.code == V.vInvalidArgument
    with pytest.raises(V.VcommError) as e:        # one buffer short: refused by the binding
        V.vAllReduce(x[:3], x[:3], 16, torch.float32, "sum", c)
    assert e.value.code == V.vInvalidArgument
    assert V.vcommCount(c) == 4
    odd = [torch.zeros(17, device=DEV)[1:].view(torch.int16)[1:9] for _ in range(4)]
    with pytest.raises(V.VcommError) as e:        # 2-byte aligned pointer for a 4-byte type
        V.vAllReduce(odd, odd, 4, torch.float32, "sum", c)
    assert e.value.code == V.vInvalidArgument
    _sync_ok(c)


# ---------------------------------------------------------------------------------------
# Full-size workloads, element by element
# ---------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def allreduce_64mib():
    """The 8 x 64 MiB fp32 uniform[-1, 1) workload (seed 1) and its oracle result, computed
    once for every channel / chunk / protocol cell that checks against it."""
    n, count = 8, 16 << 20                                          # 64 MiB fp32 per rank
    xs = inputs.uniform_ranks(n, count, torch.float32, 1)
    return xs, oracle.allreduce(xs, "sum", nthreads=NTHREADS)


@pytest.mark.parametrize("variant", [("onepass", V.vProtoSimple), ("ring", V.vProtoSimple),
                                     ("ring", V.vProtoLL), ("ring", V.vProtoLL128)],
                         ids=["onepass", "ring-simple", "ring-ll", "ring-ll128"])
def test_allreduce_64MiB_8_ranks(comms, variant, allreduce_64mib):
    # the 8 x 64 MiB fp32 workload: channels {1, 8, 16, 32}; for the staged ring with Simple
    # every chunk size from 128 KiB to 2 MiB, with LL and LL128 chunks of 128 KiB, 1 MiB and
    # 2 MiB; all bit-identical to the oracle
    algo, proto = variant
    xs, want = allreduce_64mib
    if algo == "onepass":
        cases = [(ch, None) for ch in (1, 8, 16, 32)]
    elif proto == V.vProtoSimple:
        cases = [(ch, chunk) for ch in (1, 8, 16, 32) for chunk in (128 << 10, 256 << 10, 512 << 10, 1 << 20, 2 << 20)]
    else:
        cases = [(ch, chunk) for ch in (1, 8, 16, 32) for chunk in (128 << 10, 1 << 20, 2 << 20)]
    for channels, chunk in cases:
        got = run_allreduce(comms, xs, "sum", algo, proto, channels=channels, chunk=chunk)
        assert_bits_equal(got, want, f"64MiB channels={channels} chunk={chunk}")
        del got


def test_fsdp_bucket_reduce_scatter_then_allgather(comms):
    """25 MiB bf16 gradient bucket per rank: sum * 1/8 -> fp32 shard, then all-gather of
    the bf16-rounded shard."""
    n, count = 8, 13_107_200
    rc = count // n
    xs = inputs.normal_ranks(n, count, 1e-3, torch.bfloat16, 2)
    want_shard = oracle.reduce_scatter_scale(xs, "sum", 1.0 / n, torch.float32, nthreads=NTHREADS)
    shard_bf16 = [s.to(torch.bfloat16) for s in want_shard]
    want_full = oracle.allgather(shard_bf16)
    for algo, proto in [("onepass", V.vProtoSimple), ("ring", V.vProtoSimple), ("ring", V.vProtoLL128)]:
        got = run_rs(comms, xs, "sum", algo, proto, rc, out_dtype=torch.float32, scale=1.0 / n, channels=8)
        assert_bits_equal(got, want_shard, f"fsdp rs {algo}")
        send = [g.to(torch.bfloat16) for g in got]
        recv = empty_dev(n, count, torch.bfloat16)
        c = comms.get(n, 8, proto, algo, None)
        V.vAllGather(send, recv, rc, torch.bfloat16, "sum", c)
        _sync_ok(c)
        assert_bits_equal(recv, want_full, f"fsdp ag {algo}")


def test_moe_dispatch_full(comms):
    send, counts, sd, rd, recv_elems = inputs.moe_dispatch()
    got = _a2av(comms, send, counts, sd, rd, recv_elems, torch.bfloat16)
    assert_bits_equal(got, oracle.alltoallv(send, counts, sd, rd, recv_elems), "moe alltoallv")


# ---------------------------------------------------------------------------------------
# CUDA graph capture and replay (the ring clears its counters, and for LL and LL128 its
# FIFOs, inside the graph)
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
def test_graph_capture_replays_match_oracle(comms, variant):
    algo, proto = variant
    n, count = 8, 100_003
    c = comms.get(n, 4, proto, algo, SMALL_CHUNK)
    send = empty_dev(n, count, torch.float32, fill=0.0)
    recv = empty_dev(n, count, torch.float32)
    eager = empty_dev(n, count, torch.float32)
    V.vAllReduce(send, recv, count, torch.float32, "sum", c)       # allocates the ring FIFOs
    _sync_ok(c)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        V.vAllReduce(send, recv, count, torch.float32, "sum", c)
    for seed in (1, 2, 3):
        xs = inputs.uniform_ranks(n, count, torch.float32, seed)
        for d, x in zip(send, xs):
            d.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        want = oracle.allreduce(xs, "sum")
        assert_bits_equal(recv, want, f"replay {seed}")
        V.vAllReduce(send, eager, count, torch.float32, "sum", c)  # eager launches interleave
        _sync_ok(c)
        assert_bits_equal(eager, want, f"eager after replay {seed}")


# ---------------------------------------------------------------------------------------
# Failure detection: bounded waits, abort, sticky errors (no fault, no trap)
# ---------------------------------------------------------------------------------------

def test_stalled_rank_times_out_and_error_sticks():
    n = 4
    c = V.vcommInit(n, 2, V.vProtoSimple)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommSetTimeoutMs(c, 200)
        V.vcommTestSetStallRank(c, 1)
        x = [torch.ones(1 << 16, device=DEV) for _ in range(n)]
        t0 = time.time()
        V.vAllReduce(x, x, 1 << 16, torch.float32, "sum", c)
        torch.cuda.synchronize()
        assert time.time() - t0 < 20
        assert V.vcommGetAsyncError(c) == V.vTimeout
        with pytest.raises(V.VcommError) as e:
            V.vAllReduce(x, x, 1 << 16, torch.float32, "sum", c)
        assert e.value.code == V.vTimeout
    finally:
        V.vcommDestroy(c)
    # the context is still usable afterwards
    assert float(torch.ones(4, device=DEV).sum()) == 4.0


@pytest.mark.parametrize("proto", [V.vProtoLL, V.vProtoLL128])
def test_stalled_rank_times_out_flag_protocols(proto):
    c = V.vcommInit(3, 1, proto)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommSetTimeoutMs(c, 200)
        V.vcommTestSetStallRank(c, 2)
        x = [torch.ones(1 << 14, device=DEV) for _ in range(3)]
        V.vAllReduce(x, [torch.empty_like(t) for t in x], 1 << 14, torch.float32, "sum", c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vTimeout
    finally:
        V.vcommDestroy(c)


@pytest.mark.parametrize("count", [1 << 14, 1 << 18], ids=["64KiB", "1MiB"])
def test_ll128_line_flag_mismatch_is_reported(count):
    # An LL128 reader polls one release flag per warp, then checks every line flag it
    # reads.  A rank that expects wrong line flags must stop the transfer with
    # vInternalError, in bounded time and without a fault; with the hook off again the
    # lines pass their check.  64 KiB per rank: ragged steps (lane 7 checks lines whose
    # 8-byte place holds payload); 1 MiB: whole-line steps.
    n = 4
    x = [torch.ones(count, device=DEV) for _ in range(n)]
    c = V.vcommInit(n, 1, V.vProtoLL128)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommSetTimeoutMs(c, 200)
        V.vcommTestSetBadFlagRank(c, 2)
        t0 = time.time()
        V.vAllReduce(x, [torch.empty_like(t) for t in x], count, torch.float32, "sum", c)
        torch.cuda.synchronize()
        assert time.time() - t0 < 20
        assert V.vcommGetAsyncError(c) == V.vInternalError
    finally:
        V.vcommDestroy(c)
    c = V.vcommInit(n, 1, V.vProtoLL128)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommTestSetBadFlagRank(c, 2)
        V.vcommTestSetBadFlagRank(c, -1)
        y = [torch.empty_like(t) for t in x]
        V.vAllReduce(x, y, count, torch.float32, "sum", c)
        _sync_ok(c)
        assert all(torch.equal(t, torch.full_like(t, 4.0)) for t in y)
    finally:
        V.vcommDestroy(c)


def test_abort_stops_a_waiting_transfer():
    c = V.vcommInit(4, 1, V.vProtoSimple)
    try:
        V.vcommSetAlgo(c, "ring")
        V.vcommSetTimeoutMs(c, 10_000)
        V.vcommTestSetStallRank(c, 0)
        x = [torch.ones(1 << 16, device=DEV) for _ in range(4)]
        V.vAllReduce(x, x, 1 << 16, torch.float32, "sum", c)
        time.sleep(0.3)
        t0 = time.time()
        V.vcommAbort(c)
        torch.cuda.synchronize()
        assert time.time() - t0 < 5.0
        assert V.vcommGetAsyncError(c) == V.vAborted
    finally:
        V.vcommDestroy(c)


def test_alltoallv_rank_with_nothing_to_send_or_receive():
    # An empty tensor has a NULL data pointer; a rank that sends (or receives) nothing may
    # pass one.  Rank 2 sends nothing, rank 3 receives nothing.
    n = 4
    counts = torch.tensor([[5, 0, 7, 0], [1, 2, 3, 0], [0, 0, 0, 0], [9, 4, 0, 0]], dtype=torch.int32)
    sd = (torch.cumsum(counts, 1) - counts).to(torch.int32)
    rd = (torch.cumsum(counts, 0) - counts).t().contiguous().to(torch.int32)
    recv_elems = [int(v) for v in counts.sum(0)]
    xs = [torch.arange(int(counts[i].sum()), dtype=torch.float32) + 1000 * i for i in range(n)]
    send = [x.to(DEV) for x in xs]
    recv = [torch.full((e,), -1.0, device=DEV) for e in recv_elems]
    assert send[2].data_ptr() == 0 and recv[3].data_ptr() == 0
    c = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        V.vAllToAllv(send, recv, *[t.to(DEV) for t in (counts, sd, rd)], torch.float32, c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vSuccess
        assert_bits_equal(recv, oracle.alltoallv(xs, counts, sd, rd, recv_elems), "alltoallv empty ranks")
    finally:
        V.vcommDestroy(c)


def test_alltoallv_tile_counter_resets_across_launches_and_graph_replays():
    # The variable all-to-all hands tiles out from a per-launch counter that its last CTA
    # clears; many launches in a row (more than the rotating counter slots) and replays of
    # a captured launch must each copy every tile exactly once.
    n = 8
    g = torch.Generator().manual_seed(31)
    counts = torch.randint(0, 70_000, (n, n), generator=g, dtype=torch.int32)
    sd = (torch.cumsum(counts, 1) - counts).to(torch.int32)
    rd = (torch.cumsum(counts, 0) - counts).t().contiguous().to(torch.int32)
    recv_elems = [int(v) for v in counts.sum(0)]
    tabs = [t.to(DEV) for t in (counts, sd, rd)]
    send = [torch.empty(int(counts[i].sum()), device=DEV) for i in range(n)]
    recv = [torch.empty(e, device=DEV) for e in recv_elems]
    c = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        def fill(k):
            xs = [inputs.uniform_ranks(1, int(counts[i].sum()), torch.float32, 1000 * k + i)[0] for i in range(n)]
            for d, x in zip(send, xs):
                d.copy_(x)
            return xs
        for k in range(140):
            xs = fill(k) if k % 35 == 0 else None
            for t in recv:
                t.fill_(-7.0)
            V.vAllToAllv(send, recv, *tabs, torch.float32, c)
            if xs is not None:
                torch.cuda.synchronize()
                assert_bits_equal(recv, oracle.alltoallv(xs, counts, sd, rd, recv_elems), f"launch {k}")
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            V.vAllToAllv(send, recv, *tabs, torch.float32, c)
        for k in range(3):
            xs = fill(500 + k)
            for t in recv:
                t.fill_(-7.0)
            graph.replay()
            torch.cuda.synchronize()
            assert_bits_equal(recv, oracle.alltoallv(xs, counts, sd, rd, recv_elems), f"replay {k}")
        assert V.vcommGetAsyncError(c) == V.vSuccess
    finally:
        V.vcommDestroy(c)


def test_alltoallv_eager_calls_overlapping_graph_replays():
    # A captured variable all-to-all keeps its tile counters for every replay; eager calls
    # rotate through a separate set.  More eager calls than that set holds (70 > 64), each
    # issued on a second stream while a replay of the captured call runs on the first, so
    # every eager counter pair meets a running replay: every output must still equal the
    # oracle's.
    n = 8
    g = torch.Generator().manual_seed(33)
    counts = torch.randint(0, 40_000, (n, n), generator=g, dtype=torch.int32)
    sd = (torch.cumsum(counts, 1) - counts).to(torch.int32)
    rd = (torch.cumsum(counts, 0) - counts).t().contiguous().to(torch.int32)
    recv_elems = [int(v) for v in counts.sum(0)]
    tabs = [t.to(DEV) for t in (counts, sd, rd)]
    xa = [inputs.uniform_ranks(1, int(counts[i].sum()), torch.float32, 700 + i)[0] for i in range(n)]
    xb = [inputs.uniform_ranks(1, int(counts[i].sum()), torch.float32, 800 + i)[0] for i in range(n)]
    sa, sb = [x.to(DEV) for x in xa], [x.to(DEV) for x in xb]
    ra = [torch.full((e,), -7.0, device=DEV) for e in recv_elems]
    rb = [torch.full((e,), -7.0, device=DEV) for e in recv_elems]
    c = V.vcommInit(n, 1, V.vProtoSimple)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    try:
        V.vAllToAllv(sa, ra, *tabs, torch.float32, c)            # warm-up before capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            V.vAllToAllv(sa, ra, *tabs, torch.float32, c)
        torch.cuda.synchronize()
        want_a = oracle.alltoallv(xa, counts, sd, rd, recv_elems)
        want_b = oracle.alltoallv(xb, counts, sd, rd, recv_elems)
        for k in range(70):
            with torch.cuda.stream(s1):
                graph.replay()
            V.vAllToAllv(sb, rb, *tabs, torch.float32, c, s2)
            if k % 10 == 9:
                torch.cuda.synchronize()
                assert_bits_equal(ra, want_a, f"replay {k}")
                assert_bits_equal(rb, want_b, f"eager {k}")
                for t in ra + rb:
                    t.fill_(-7.0)
                torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vSuccess
    finally:
        torch.cuda.synchronize()
        V.vcommDestroy(c)


def test_alltoallv_positive_count_into_null_buffer_sets_async_error():
    n = 2
    c = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        counts = torch.tensor([[2, 2], [2, 2]], dtype=torch.int32, device=DEV)
        sd = torch.tensor([[0, 2], [0, 2]], dtype=torch.int32, device=DEV)
        x = [torch.zeros(4, device=DEV) for _ in range(n)]
        y = [torch.zeros(4, device=DEV), None]
        V.vAllToAllv(x, y, counts, sd, sd, torch.float32, c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vInvalidArgument
    finally:
        V.vcommDestroy(c)


def test_bad_alltoallv_table_sets_async_error():
    n = 2
    c = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        counts = torch.tensor([[4, -1], [4, 4]], dtype=torch.int32, device=DEV)
        zeros = torch.zeros(2, 2, dtype=torch.int32, device=DEV)
        x = [torch.zeros(16, device=DEV) for _ in range(n)]
        y = [torch.zeros(16, device=DEV) for _ in range(n)]
        V.vAllToAllv(x, y, counts, zeros, zeros, torch.float32, c)
        torch.cuda.synchronize()
        assert V.vcommGetAsyncError(c) == V.vInvalidArgument
    finally:
        V.vcommDestroy(c)


# ---------------------------------------------------------------------------------------
# Fan-out copies through both engines: TMA bulk copies (default) and per-thread loads/stores
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("tma", [True, False], ids=["tma", "lsu"])
def test_fanout_copies_both_engines(tma, monkeypatch):
    monkeypatch.setenv("VCOMM_COPY_TMA", "1" if tma else "0")
    n = 8
    c = V.vcommInit(n, 1, V.vProtoSimple)
    try:
        for dtype, sc in [(torch.float32, 1 << 20), (torch.bfloat16, 1_638_400), (torch.float16, 8),
                          (torch.int32, 12_348)]:
            plan = V.vcommQueryPlan(c, V.vCollAllGather, sc, dtype, 32)
            assert plan["bulkCopy"] == (1 if tma else 0)
            xs = inputs.uniform_ranks(n, sc, dtype, seed=sc)
            send = to_dev(xs)
            recv = empty_dev(n, n * sc, dtype)
            V.vAllGather(send, recv, sc, dtype, "sum", c)
            _sync_ok(c)
            assert_bits_equal(recv, oracle.allgather(xs), f"allgather {dtype} {sc} tma={tma}")
            root = 5
            g = [None] * n
            g[root] = torch.empty(n * sc, dtype=dtype, device=DEV)
            V.vGather(send, g, sc, dtype, root, c)
            _sync_ok(c)
            assert_bits_equal([g[root]], [oracle.gather(xs, root)], "gather")
            bcast = empty_dev(n, n * sc, dtype)
            big = inputs.uniform_ranks(1, n * sc, dtype, seed=sc + 1)[0]
            src = [None] * n
            src[root] = big.to(DEV)
            V.vBroadcast(src, bcast, n * sc, dtype, "sum", root, c)
            _sync_ok(c)
            assert all(torch.equal(b.cpu().view(torch.int16 if b.element_size() == 2 else torch.int32),
                                   big.view(torch.int16 if big.element_size() == 2 else torch.int32)) for b in bcast)
    finally:
        V.vcommDestroy(c)
