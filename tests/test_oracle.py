"""Pins for the CPU oracle, checked against things other than itself.

* converters: torch's and numpy's own fp16/bf16 conversions, exhaustively or on
  adversarial values (midpoints, overflow, subnormals);
* schedules: golden tables from the pages (ring AllGather slices, getNextSendAddr
  chunk ids) against the literal ring simulator in ``ring_sim``;
* order: hand-worked fixtures whose result changes with the ring order or the block
  alignment rule, and a brute-force comparison with the message-passing simulator;
* special cases that reduce to library routines (order-free min/max/int sums, exact
  small-integer sums, cat/transposes for the copies), invariants (AR = AG o RS,
  A2A o A2A = id, broadcast idempotent, N = 1 identity, count 0), and the fp64
  error bound of the benchmark spec.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from collective_communication_virtual_gb300 import inputs
from tests import ring_sim

DTYPES = [torch.float32, torch.float16, torch.bfloat16, torch.int32]
OPS = ["sum", "prod", "min", "max"]


def _bits(t: torch.Tensor) -> torch.Tensor:
    return t.view({4: torch.int32, 2: torch.int16}[t.element_size()])


def _same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.dtype == b.dtype and a.shape == b.shape and torch.equal(_bits(a), _bits(b))


def _read_rows(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return rows


# ---------------------------------------------------------------------------------
# Converters
# ---------------------------------------------------------------------------------

def test_bf16_to_f32_exhaustive():
    allb = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    ref = allb.float()
    got = oracle.to_f32(allb)
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(_bits(got)[~nan], _bits(ref)[~nan])


def test_f16_to_f32_exhaustive():
    allh = np.arange(65536, dtype=np.uint16).view(np.float16)
    ref = torch.from_numpy(allh.astype(np.float32))
    got = oracle.to_f32(torch.from_numpy(allh.copy()))
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(_bits(got)[~nan], _bits(ref)[~nan])


def _adversarial_f32(n=400_000, seed=11):
    g = np.random.default_rng(seed)
    u = g.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    # exact midpoints between bf16 neighbours and between fp16 neighbours, both parities
    mid_bf = (g.integers(0, 2**16, size=n // 8, dtype=np.uint32) << 16) | 0x8000
    base_h = g.integers(0x33000000 >> 13, 0x47800000 >> 13, size=n // 8).astype(np.uint32) << 13
    mid_h = base_h | 0x1000
    special = np.array([0, 0x80000000, 0x7F800000, 0xFF800000, 0x7F7FFFFF, 0x477FE000,
                        0x477FEFFF, 0x477FF000, 0x477FF001, 0x38800000, 0x387FFFFF, 0x33800000,
                        0x33000000, 0x33000001, 0x00000001, 0x00800000, 0x7F7F8000,
                        0x7F7F7FFF], dtype=np.uint32)
    allu = np.concatenate([u, mid_bf, mid_h, special])
    return torch.from_numpy(allu.view(np.float32).copy())


def test_f32_to_bf16_matches_torch():
    x = _adversarial_f32()
    ref = x.to(torch.bfloat16)
    got = oracle.from_f32(x, torch.bfloat16)
    nan = torch.isnan(ref.float())
    assert torch.equal(torch.isnan(got.float()), nan)
    assert torch.equal(_bits(got)[~nan], _bits(ref)[~nan])


def test_f32_to_f16_matches_numpy():
    x = _adversarial_f32()
    with np.errstate(over="ignore"):          # values past the fp16 range round to infinity
        ref = torch.from_numpy(x.numpy().astype(np.float16))
    got = oracle.from_f32(x, torch.float16)
    nan = torch.isnan(ref.float())
    assert torch.equal(torch.isnan(got.float()), nan)
    assert torch.equal(_bits(got)[~nan], _bits(ref)[~nan])


# ---------------------------------------------------------------------------------
# Schedules from the pages
# ---------------------------------------------------------------------------------

def test_allgather_schedule_golden(golden_dir):
    rows = _read_rows(os.path.join(golden_dir, "ring_allgather_rank0_n4.txt"))
    assert rows == [[i, *ring_sim.ag_slices(0, i, 4)] for i in range(3)]


def test_reduce_scatter_chunk_schedule_golden(golden_dir):
    rows = _read_rows(os.path.join(golden_dir, "ring_rs_chunk_n4.txt"))
    assert rows == [[r, s, ring_sim.rs_chunk(r, s, 4)] for r in range(4) for s in range(4)]


def test_order_golden_fp32(golden_dir):
    for row in _read_rows(os.path.join(golden_dir, "allreduce_order_fp32.txt")):
        count, expected = row[0], row[1:]
        vals = [2.0**24, 1.0, 1.0, -(2.0**24)]
        xs = [torch.full((count,), v, dtype=torch.float32) for v in vals]
        out = oracle.allreduce(xs, "sum")
        for r in range(4):
            assert out[r].tolist() == [float(v) for v in expected], (count, out[r])
        sim = ring_sim.ring_allreduce(xs, "sum", oracle.block_elems(count, 4, 4))
        assert sim[0].tolist() == [float(v) for v in expected]


def test_min_signed_zero_golden(golden_dir):
    (signs,) = _read_rows(os.path.join(golden_dir, "allreduce_min_signed_zero.txt"))
    xs = [torch.zeros(8, dtype=torch.float32), -torch.zeros(8, dtype=torch.float32)]
    out = oracle.allreduce(xs, "min")
    for r in range(2):
        assert torch.signbit(out[r]).int().tolist() == signs


# ---------------------------------------------------------------------------------
# Brute force against the message-passing ring
# ---------------------------------------------------------------------------------

BF_N = [1, 2, 3, 4, 5, 7, 8]
BF_COUNTS = [0, 1, 2, 3, 7, 15, 16, 17, 31, 33, 255, 1024]


def _inputs(n, count, dtype, seed):
    if dtype == torch.int32:
        return inputs.uniform_ranks(n, count, dtype, seed)
    # keep products finite and away from zero ties: uniform[-1,1) shifted off zero
    xs = inputs.uniform_ranks(n, count, torch.float32, seed)
    return [(x * 1.5 + torch.sign(x) * 0.25).to(dtype) for x in xs]


@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
@pytest.mark.parametrize("op", OPS)
def test_allreduce_matches_ring_simulation(dtype, op):
    esz = torch.tensor([], dtype=dtype).element_size()
    for n in BF_N:
        for count in BF_COUNTS:
            xs = _inputs(n, count, dtype, seed=1000 * n + count)
            got = oracle.allreduce(xs, op)
            # chunk size of getNextSendAddr's tail rule, bytes -> elements
            chunk = -(-count // n)
            chunk = -(-chunk // (16 // esz)) * (16 // esz)
            sim = ring_sim.ring_allreduce(xs, op, chunk)
            for r in range(n):
                assert _same_bits(got[r], sim[r]), (n, count, r)


@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
@pytest.mark.parametrize("op", OPS)
def test_reduce_scatter_matches_ring_simulation(dtype, op):
    for n in BF_N:
        for rc in [0, 1, 2, 3, 5, 8, 17, 33]:
            xs = _inputs(n, n * rc, dtype, seed=77 * n + rc)
            got = oracle.reduce_scatter(xs, op)
            sim = ring_sim.ring_reduce_scatter(xs, op)
            for r in range(n):
                assert _same_bits(got[r], sim[r]), (n, rc, r)


@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
def test_allgather_matches_ring_simulation(dtype):
    for n in BF_N:
        for sc in [0, 1, 3, 16, 33]:
            xs = _inputs(n, sc, dtype, seed=5 * n + sc)
            got = oracle.allgather(xs)
            sim = ring_sim.ring_allgather(xs)
            for r in range(n):
                assert _same_bits(got[r], sim[r])


def test_order_matters_for_random_fp32():
    """The simulator and the oracle agree, and a different start rank would not."""
    xs = inputs.uniform_ranks(8, 4096, torch.float32, 3)
    got = oracle.allreduce(xs, "sum")
    shifted = xs[1:] + xs[:1]            # relabel ranks: every block starts one rank later
    other = oracle.allreduce(shifted, "sum")
    assert not torch.equal(_bits(got[0]), _bits(other[0]))


# ---------------------------------------------------------------------------------
# Special cases that reduce to library routines
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
def test_min_max_are_library_reductions(dtype):
    xs = inputs.uniform_ranks(8, 3001, dtype, 21)
    stack = torch.stack(xs)
    for op, ref in (("min", stack.amin(0)), ("max", stack.amax(0))):
        out = oracle.allreduce(xs, op)
        assert all(_same_bits(o, ref) for o in out)
        rs = oracle.reduce_scatter([x[:3000] for x in xs], op)
        ref_rs = torch.stack([x[:3000] for x in xs]).amin(0) if op == "min" else \
            torch.stack([x[:3000] for x in xs]).amax(0)
        assert _same_bits(torch.cat(rs), ref_rs)


def test_int32_sum_prod_wrap_like_int64_mod_2_32():
    xs = inputs.uniform_ranks(8, 4099, torch.int32, 9)
    s64 = torch.stack([x.to(torch.int64) for x in xs])
    for op in ("sum", "prod"):
        ref = s64.sum(0) if op == "sum" else s64.prod(0)     # int64 prod wraps mod 2^64,
        ref = ring_sim._wrap32(ref)                           # whose low 32 bits are exact
        out = oracle.allreduce(xs, op)
        assert all(torch.equal(o, ref) for o in out)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16],
                         ids=lambda d: str(d).split(".")[1])
def test_small_integer_sums_are_exact(dtype):
    xs = inputs.small_int_ranks(8, 5000, dtype, 4)
    ref = torch.stack([x.to(torch.float64) for x in xs]).sum(0).to(dtype)
    out = oracle.allreduce(xs, "sum")
    assert all(_same_bits(o, ref) for o in out)
    out = oracle.reduce_scatter(xs, "sum")
    assert _same_bits(torch.cat(out), ref)


def test_copies_are_cat_and_transpose():
    n = 5
    xs = inputs.uniform_ranks(n, 3 * n, torch.bfloat16, 8)
    ag = oracle.allgather(xs)
    assert all(_same_bits(a, torch.cat(xs)) for a in ag)
    bc = oracle.broadcast(xs, root=3)
    assert all(_same_bits(b, xs[3]) for b in bc)
    a2a = oracle.alltoall(xs)
    blocks = torch.stack([x.view(n, 3) for x in xs])          # [sender, block, t]
    for j in range(n):
        assert _same_bits(a2a[j], blocks[:, j, :].reshape(-1))


def test_alltoallv_matches_slicing():
    send, counts, sd, rd, recv_elems = inputs.moe_dispatch(n_ranks=4, tokens=64, hidden=8,
                                                           n_experts=4)
    out = oracle.alltoallv(send, counts, sd, rd, recv_elems)
    for j in range(4):
        pieces = [send[i][int(sd[i, j]):int(sd[i, j]) + int(counts[i, j])] for i in range(4)]
        assert _same_bits(out[j], torch.cat(pieces))


# ---------------------------------------------------------------------------------
# Invariants and degenerate cases
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
@pytest.mark.parametrize("op", OPS)
def test_allreduce_is_reduce_scatter_then_allgather(dtype, op):
    n, rc = 8, 64                                  # rc a multiple of 16 bytes: same blocks
    xs = inputs.uniform_ranks(n, n * rc, dtype, 31)
    ar = oracle.allreduce(xs, op)
    ag = oracle.allgather(oracle.reduce_scatter(xs, op))
    assert all(_same_bits(a, b) for a, b in zip(ar, ag))


def test_alltoall_twice_is_identity_and_broadcast_idempotent():
    xs = inputs.uniform_ranks(8, 8 * 7, torch.float16, 2)
    back = oracle.alltoall(oracle.alltoall(xs))
    assert all(_same_bits(a, b) for a, b in zip(back, xs))
    once = oracle.broadcast(xs, 0)
    twice = oracle.broadcast(once, 0)
    assert all(_same_bits(a, b) for a, b in zip(once, twice))


@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
def test_single_rank_is_identity(dtype):
    (x,) = inputs.uniform_ranks(1, 1000, dtype, 1)
    for op in OPS:
        assert _same_bits(oracle.allreduce([x], op)[0], x)
        assert _same_bits(oracle.reduce_scatter([x], op)[0], x)


def test_zero_count_is_noop():
    xs = [torch.empty(0, dtype=torch.float32) for _ in range(4)]
    assert all(o.numel() == 0 for o in oracle.allreduce(xs))
    assert all(o.numel() == 0 for o in oracle.reduce_scatter(xs))
    assert all(o.numel() == 0 for o in oracle.allgather(xs))


def test_rejects_bad_arguments():
    lib = oracle.lib()
    assert lib.orc_allreduce(7, 0, 4, 10, None, None, 1) != 0          # bad dtype
    assert lib.orc_allreduce(0, 9, 4, 10, None, None, 1) != 0          # bad op
    assert lib.orc_allreduce(0, 0, 0, 10, None, None, 1) != 0          # N < 1
    assert lib.orc_broadcast(4, 4, 10, 4, None, None) != 0             # root out of range


# ---------------------------------------------------------------------------------
# Error bound against an fp64 reference (spec tolerances)
# ---------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,tol", [(torch.float32, None), (torch.float16, 1e-2),
                                       (torch.bfloat16, 1e-2)],
                         ids=["float32", "float16", "bfloat16"])
def test_sum_within_fp64_bound(dtype, tol):
    n = 8
    tol = 1e-5 * n if tol is None else tol
    xs = inputs.uniform_ranks(n, 1 << 15, dtype, 0)
    x64 = torch.stack([x.to(torch.float64) for x in xs])
    ref = x64.sum(0)
    mag = x64.abs().sum(0)
    out = oracle.allreduce(xs, "sum")[0].to(torch.float64)
    assert bool(((out - ref).abs() <= tol * mag).all())


def test_scale_cast_epilogue():
    n = 8
    xs = inputs.normal_ranks(n, n * 1000, 1e-3, torch.bfloat16, 2)
    rs = oracle.reduce_scatter(xs, "sum")
    out = oracle.reduce_scatter_scale(xs, "sum", 1.0 / n, torch.float32)
    # 1/8 is a power of two: scaling is exact, so out * 8 is the bf16 partial widened
    for a, b in zip(out, rs):
        assert torch.equal(a * n, b.float())
    out_bf = oracle.reduce_scatter_scale(xs, "sum", 1.0 / n, torch.bfloat16)
    for a, b in zip(out_bf, rs):
        assert torch.equal(a.float() * n, b.float())


def test_scale_cast_epilogue_rounds_once_in_fp32():
    # a scale that is not a power of two rounds: out = fp32(acc) * fp32(scale), one RNE
    # multiply, which numpy's float32 product computes independently of the oracle
    import numpy as np
    n = 3
    xs = inputs.uniform_ranks(n, n * 4000, torch.bfloat16, 13)
    rs = oracle.reduce_scatter(xs, "sum")
    scale = float(np.float32(1.0) / np.float32(3.0))
    out = oracle.reduce_scatter_scale(xs, "sum", scale, torch.float32)
    for a, b in zip(out, rs):
        want = b.float().numpy().astype(np.float32) * np.float32(scale)
        assert np.array_equal(a.numpy().view(np.int32), want.view(np.int32))
    # and the bf16 output is that fp32 value rounded to bf16 (torch's RNE converter)
    out_bf = oracle.reduce_scatter_scale(xs, "sum", scale, torch.bfloat16)
    for a, b in zip(out_bf, out):
        assert torch.equal(a.view(torch.int16), b.to(torch.bfloat16).view(torch.int16))


def test_threads_do_not_change_bits():
    xs = inputs.uniform_ranks(8, 100_003, torch.bfloat16, 6)
    a = oracle.allreduce(xs, "sum", nthreads=1)
    b = oracle.allreduce(xs, "sum", nthreads=7)
    assert all(_same_bits(x, y) for x, y in zip(a, b))


# ---------------------------------------------------------------------------------------
# Rooted collectives: reduce, gather, scatter
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
@pytest.mark.parametrize("op", OPS)
def test_reduce_matches_ring_chain(dtype, op):
    for n in (1, 2, 3, 5, 8):
        for count in (0, 1, 7, 33, 1000):
            xs = _inputs(n, count, dtype, seed=17 * n + count)
            for root in {0, n - 1, n // 2}:
                got = oracle.reduce(xs, op, root)
                assert _same_bits(got, ring_sim.ring_reduce_chain(xs, op, root)), (n, count, root)


def test_reduce_order_is_the_roots_block_order():
    """Reduce to root r reduces in the order that block r of an all-reduce uses."""
    xs = inputs.uniform_ranks(8, 4096, torch.float32, 5)
    B = oracle.block_elems(4096, 8, 4)
    ar = oracle.allreduce(xs, "sum")[0]
    for root in range(8):
        got = oracle.reduce(xs, "sum", root)
        assert _same_bits(got[root * B:(root + 1) * B], ar[root * B:(root + 1) * B])


def test_reduce_min_max_int_are_library_reductions():
    xs = inputs.uniform_ranks(6, 999, torch.int32, 8)
    s64 = torch.stack([x.to(torch.int64) for x in xs])
    assert torch.equal(oracle.reduce(xs, "max", 2), s64.amax(0).to(torch.int32))
    assert torch.equal(oracle.reduce(xs, "sum", 4), ring_sim._wrap32(s64.sum(0)))


def test_gather_and_scatter_are_cat_and_chunk():
    n = 6
    xs = inputs.uniform_ranks(n, 77, torch.float16, 3)
    for root in (0, 5):
        assert _same_bits(oracle.gather(xs, root), torch.cat(xs))
    src = inputs.uniform_ranks(1, n * 13, torch.bfloat16, 4)[0]
    for root in (0, 3):
        out = oracle.scatter(src, n, root)
        assert all(_same_bits(o, c) for o, c in zip(out, src.chunk(n)))
    # scatter of a gather gives every rank its own buffer back
    back = oracle.scatter(oracle.gather(xs, 2), n, 2)
    assert all(_same_bits(a, b) for a, b in zip(back, xs))


# ---------------------------------------------------------------------------------------
# Double binary tree
# ---------------------------------------------------------------------------------------

def test_btree_worked_example_golden(golden_dir):
    (row,) = _read_rows(os.path.join(golden_dir, "btree_rank1_n8.txt"))
    n, rank, parent, c0, c1 = row
    assert oracle.tree_links(n, rank, 0) == (parent, c0, c1)


def test_tree_links_hand_worked_table(golden_dir):
    # Both trees at 5, 6, 7 and 12 ranks, worked by hand from the ncclGetBtree rules and
    # the ncclGetDtree mirror (even n) / shift (odd n): the up >= n fallback, the shrinking
    # second-child step and the root's single child are all exercised.
    rows = _read_rows(os.path.join(golden_dir, "btree_links.txt"))
    assert sorted({r[0] for r in rows}) == [5, 6, 7, 12] and len(rows) == 2 * (5 + 6 + 7 + 12)
    for n, tree, rank, parent, c0, c1 in rows:
        assert oracle.tree_links(n, rank, tree) == (parent, c0, c1), (n, tree, rank)


@pytest.mark.parametrize("tree", [0, 1])
def test_trees_are_spanning_trees(tree):
    for n in range(1, 65):
        links = [oracle.tree_links(n, r, tree) for r in range(n)]
        roots = [r for r in range(n) if links[r][0] < 0]
        assert len(roots) == 1, (n, roots)
        for r, (up, c0, c1) in enumerate(links):
            for c in (c0, c1):
                if c >= 0:
                    assert 0 <= c < n and links[c][0] == r, (n, r, c)
            if up >= 0:
                assert r in links[up][1:], (n, r, up)
        seen, stack = set(), [roots[0]]
        while stack:
            v = stack.pop()
            assert v not in seen
            seen.add(v)
            stack += [c for c in links[v][1:] if c >= 0]
        assert seen == set(range(n)), n
    # tree 0 hangs from rank 0; tree 1 is its mirror (even n) or shift (odd n)
    assert oracle.tree_links(8, 0, 0)[0] < 0 and oracle.tree_links(8, 7, 1)[0] < 0
    assert oracle.tree_links(5, 1, 1)[0] < 0


def test_tree_order_golden_fp32(golden_dir):
    for row in _read_rows(os.path.join(golden_dir, "tree_allreduce_order_n4.txt")):
        count, expected = row[0], row[1:]
        vals = [1.0, 2.0**24, 1.0, -(2.0**24)]
        xs = [torch.full((count,), v, dtype=torch.float32) for v in vals]
        for out in oracle.allreduce_tree(xs, "sum"):
            assert out.tolist() == [float(v) for v in expected]


@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: str(d).split(".")[1])
@pytest.mark.parametrize("op", OPS)
def test_tree_allreduce_matches_message_passing(dtype, op):
    esz = torch.tensor([], dtype=dtype).element_size()
    for n in (1, 2, 3, 4, 5, 7, 8, 13):
        for count in (0, 1, 7, 16, 33, 255, 1000):
            xs = _inputs(n, count, dtype, seed=3 * n + count)
            got = oracle.allreduce_tree(xs, op)
            split = -(-count // 2)
            split = -(-split // (16 // esz)) * (16 // esz)
            sim = ring_sim.tree_allreduce(xs, op, lambda r, t: oracle.tree_links(n, r, t), min(split, count))
            for r in range(n):
                assert _same_bits(got[r], sim[r]), (n, count, r)


def test_tree_allreduce_library_special_cases():
    xs = inputs.uniform_ranks(8, 3001, torch.int32, 12)
    s64 = torch.stack([x.to(torch.int64) for x in xs])
    assert torch.equal(oracle.allreduce_tree(xs, "sum")[3], ring_sim._wrap32(s64.sum(0)))
    assert torch.equal(oracle.allreduce_tree(xs, "min")[0], s64.amin(0).to(torch.int32))
    ys = inputs.small_int_ranks(8, 4000, torch.bfloat16, 2)
    want = torch.stack([y.float() for y in ys]).sum(0).to(torch.bfloat16)
    assert _same_bits(oracle.allreduce_tree(ys, "sum")[0], want)
    # a different order than the ring: random fp32 sums differ somewhere
    zs = inputs.uniform_ranks(8, 4096, torch.float32, 1)
    assert not _same_bits(oracle.allreduce_tree(zs, "sum")[0], oracle.allreduce(zs, "sum")[0])


def test_index_pattern_is_a_function_of_rank_and_index_only():
    # slices rebuilt from any start agree with the whole; values are exact in every type
    whole = inputs.index_pattern(1, 0, 5000, torch.float32)
    for start in (0, 1, 511, 2047, 4999):
        part = inputs.index_pattern(1, start, 5000 - start, torch.float32)
        assert torch.equal(part, whole[start:])
    k = whole * 256
    assert torch.equal(k, k.round()) and k.abs().max() <= 255
    for dt in (torch.float16, torch.bfloat16):
        assert torch.equal(inputs.index_pattern(1, 0, 5000, dt).float(), whole)
    assert torch.equal(inputs.index_pattern(1, 0, 5000, torch.int32).float(), k)
    # far past 2^31 and 2^32 the pattern still differs from the one 2^31 or 2^32 earlier
    for e in (1 << 31, (1 << 32) + 7, (1 << 33) + 1):
        far = inputs.index_pattern(0, e, 64, torch.float32)
        for back in (1 << 31, 1 << 32):
            if e >= back:
                assert not torch.equal(far, inputs.index_pattern(0, e - back, 64, torch.float32)), (e, back)
    assert not torch.equal(inputs.index_pattern(0, 0, 64, torch.float32), inputs.index_pattern(1, 0, 64, torch.float32))
