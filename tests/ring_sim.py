"""A literal, message-passing simulation of the ring schedule (test code only).

This is an independent formulation used to pin the oracle: instead of the oracle's
closed-form per-element order it keeps one buffer per rank and moves whole chunks from
rank to rank, step by step, as the pages' ring does:

* reduce-scatter stage s: rank r works on chunk (r + N - 1 - s) mod N -- the chunk
  arithmetic of RingARAlgorithm::getNextSendAddr (NCCL book, section 2.3 "algorithm",
  Ring).  At stage 0 it sends its own copy of that chunk; at every later stage the chunk
  it receives from rank r-1 is combined with its own copy and the result is what it
  holds (and sends on);
* all-gather round i: rank r sends slice (r - i) mod N and receives (r - i - 1) mod N --
  the bootstrap ring AllGather ("NCCL Expert Course 17", ring AllGather).

Element arithmetic uses torch's own CPU ops on tensors of the storage type (fp32 IEEE
ops; fp16/bf16 ops widen to fp32 and round back), so every hop rounds like a stored
partial.  Integer ops are done in int64 and wrapped to 32 bits.
"""
from __future__ import annotations

import torch


def rs_chunk(rank: int, stage: int, n: int) -> int:
    return (rank + n - 1 - stage) % n


def ag_slices(rank: int, i: int, n: int) -> tuple[int, int]:
    return (rank - i) % n, (rank - i - 1) % n


def _wrap32(v: torch.Tensor) -> torch.Tensor:
    v = v & 0xFFFFFFFF
    return torch.where(v >= 2**31, v - 2**32, v).to(torch.int32)


def combine(op: str, partial: torch.Tensor, local: torch.Tensor) -> torch.Tensor:
    """One ring hop: the received partial combined with the receiver's own element."""
    if partial.dtype == torch.int32:
        a, b = partial.to(torch.int64), local.to(torch.int64)
        if op == "sum":
            return _wrap32(a + b)
        if op == "prod":
            return _wrap32(a * b)
    if op == "sum":
        return partial + local
    if op == "prod":
        return partial * local
    if op == "min":
        return torch.where(local < partial, local, partial)
    if op == "max":
        return torch.where(local > partial, local, partial)
    raise ValueError(op)


def ring_reduce_scatter_chunks(xs, op, bounds):
    """Run the N-1 reduce-scatter stages over chunks ``bounds[c] = (lo, hi)``.

    Returns per-rank buffers; rank r's chunk r then holds the finished result."""
    n = len(xs)
    bufs = [x.clone() for x in xs]
    for s in range(n - 1):
        msgs = []
        for r in range(n):
            c = rs_chunk(r, s, n)
            lo, hi = bounds[c]
            msgs.append((r, c, bufs[r][lo:hi].clone()))
        for r, c, data in msgs:
            dst = (r + 1) % n
            assert rs_chunk(dst, s + 1, n) == c     # the receiver's next stage is this chunk
            lo, hi = bounds[c]
            bufs[dst][lo:hi] = combine(op, data, bufs[dst][lo:hi])
    for r in range(n):
        assert rs_chunk(r, n - 1, n) == r
    return bufs


def ring_allgather_chunks(bufs, bounds):
    """N-1 all-gather rounds: each rank forwards the slice it holds to the next rank."""
    n = len(bufs)
    for i in range(n - 1):
        msgs = []
        for r in range(n):
            sl, _ = ag_slices(r, i, n)
            lo, hi = bounds[sl]
            msgs.append((r, sl, bufs[r][lo:hi].clone()))
        for r, sl, data in msgs:
            dst = (r + 1) % n
            assert ag_slices(dst, i, n)[1] == sl
            lo, hi = bounds[sl]
            bufs[dst][lo:hi] = data
    return bufs


def chunk_bounds(count: int, n: int, chunk: int):
    return [(min(c * chunk, count), min((c + 1) * chunk, count)) for c in range(n)]


def ring_allreduce(xs, op: str, chunk_elems: int):
    """Ring all-reduce over chunks of ``chunk_elems`` elements (the last chunks may be
    short or empty)."""
    n, count = len(xs), xs[0].numel()
    bounds = chunk_bounds(count, n, chunk_elems)
    bufs = ring_reduce_scatter_chunks(xs, op, bounds)
    return ring_allgather_chunks(bufs, bounds)


def ring_reduce_scatter(xs, op: str):
    n, count = len(xs), xs[0].numel()
    rc = count // n
    bounds = chunk_bounds(count, n, rc)
    bufs = ring_reduce_scatter_chunks(xs, op, bounds)
    return [bufs[r][r * rc:(r + 1) * rc].clone() for r in range(n)]


def ring_allgather(xs):
    n, sc = len(xs), xs[0].numel()
    bufs = [torch.zeros(n * sc, dtype=xs[0].dtype) for _ in range(n)]
    for r in range(n):
        bufs[r][r * sc:(r + 1) * sc] = xs[r]
    return ring_allgather_chunks(bufs, [(s * sc, (s + 1) * sc) for s in range(n)])


def ring_reduce_chain(xs, op: str, root: int):
    """Reduce to root as a ring chain: rank root+1 sends its whole buffer to root+2, which
    combines it with its own and passes it on, ..., until the root combines the last hop."""
    n = len(xs)
    partial = xs[(root + 1) % n].clone()
    for k in range(2, n + 1):
        partial = combine(op, partial, xs[(root + k) % n])
    return partial


def tree_allreduce(xs, op: str, links, split: int):
    """Double-binary-tree all-reduce by messages up each tree: every rank starts with its
    own element; a rank that has heard from all its children sends its partial to its
    parent, which combines it in child order (child 0, then child 1).  `links(rank, t)`
    gives (parent, child0, child1); elements [0, split) use tree 0, the rest tree 1."""
    n = len(xs)
    out = torch.empty_like(xs[0])
    for t, sl in ((0, slice(0, split)), (1, slice(split, xs[0].numel()))):
        partial = {r: xs[r][sl].clone() for r in range(n)}
        pending = {r: [c for c in links(r, t)[1:] if c >= 0] for r in range(n)}
        received = {r: {} for r in range(n)}
        sent = set()
        root = None
        while len(sent) < n - 1 or root is None:
            progress = False
            for r in range(n):
                parent = links(r, t)[0]
                if r in sent or any(c not in received[r] for c in pending[r]):
                    continue
                value = partial[r]
                for c in pending[r]:                     # child 0 first, then child 1
                    value = combine(op, value, received[r][c])
                if parent < 0:
                    root = value
                    sent.add(r)
                else:
                    received[parent][r] = value
                    sent.add(r)
                progress = True
            if not progress:
                raise RuntimeError("tree has a cycle or an unreachable rank")
        out[sl] = root
    return [out.clone() for _ in range(n)]
