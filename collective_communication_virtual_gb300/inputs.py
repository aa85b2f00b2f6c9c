"""Seeded synthetic inputs for the virtual-rank collectives.

Every buffer is drawn on the CPU from one ``torch.Generator`` per workload, rank by
rank in order 0..N-1, so that the CUDA path and the CPU oracle receive byte-identical
inputs.  This module only draws numbers and lays them out per virtual rank; it holds
none of the collectives' arithmetic (no reduction, no block partition, no schedule).

Workload shapes follow the pages' statement of the problem:

* uniform[-1, 1) fp32/fp16/bf16 buffers and int32 integers in [-2^20, 2^20] for the
  all-reduce / reduce-scatter / all-gather / broadcast sweeps;
* normal(0, 1e-3) bf16 gradient buckets of 25 MiB per rank, the DDP/FSDP default
  bucket size ("AI Systems Performance Engineering (3)", *Reducing Communication
  Frequency and Volume*);
* an MoE token dispatch for all-to-all: 4096 tokens x hidden 4096 per rank, each token
  routed to 2 distinct experts drawn from a Zipf(1.2) popularity over 8 experts, one
  expert per rank ("AI Systems Performance Engineering (3)", collective table, the
  all-to-all row: expert-parallel token dispatch).
"""
from __future__ import annotations

import torch

INT32_LO = -(1 << 20)
INT32_HI = 1 << 20


def uniform_ranks(n_ranks: int, count: int, dtype: torch.dtype, seed: int) -> list[torch.Tensor]:
    """N CPU buffers of ``count`` elements: uniform[-1,1) floats or int32 in [-2^20, 2^20].

    Floats are drawn in fp32 (``torch.rand * 2 - 1``) and rounded to ``dtype`` by torch
    (round-to-nearest-even)."""
    g = torch.Generator().manual_seed(seed)
    out = []
    for _ in range(n_ranks):
        if dtype == torch.int32:
            t = torch.randint(INT32_LO, INT32_HI + 1, (count,), generator=g, dtype=torch.int64)
            out.append(t.to(torch.int32))
        else:
            t = torch.rand(count, generator=g, dtype=torch.float32) * 2 - 1
            out.append(t.to(dtype))
    return out


def normal_ranks(n_ranks: int, count: int, std: float, dtype: torch.dtype, seed: int) -> list[torch.Tensor]:
    """N CPU buffers drawn from normal(0, std) in fp32, then rounded to ``dtype``."""
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn(count, generator=g, dtype=torch.float32) * std).to(dtype)
            for _ in range(n_ranks)]


def index_pattern(rank: int, start: int, count: int, dtype: torch.dtype, device="cpu") -> torch.Tensor:
    """Elements [start, start + count) of rank ``rank`` of a deterministic pattern for
    buffers too large to draw on the host: a hash of (rank, index) mapped to k / 256 with
    integer k in [-255, 255] (exact in fp16, bf16 and fp32), or to the integer k for
    int32.  The hash stays below 2^63 for indices below 2^40.  Any slice can be rebuilt
    anywhere from its indices alone, so a test fills a multi-GiB buffer on the device and
    recomputes sampled elements on the host."""
    e = torch.arange(start, start + count, dtype=torch.int64, device=device)
    k = (e * 40503 + (e >> 11) * 977 + (rank + 1) * 97531) % 511 - 255
    if dtype == torch.int32:
        return k.to(torch.int32)
    return (k.to(torch.float32) / 256).to(dtype)


def small_int_ranks(n_ranks: int, count: int, dtype: torch.dtype, seed: int, lo: int = -8,
                    hi: int = 8) -> list[torch.Tensor]:
    """N buffers of small integers stored in ``dtype`` (exact in every supported type).

    Sums and products of such values are exact, so their result does not depend on the
    reduction order; tests use them to compare against order-free library routines."""
    g = torch.Generator().manual_seed(seed)
    return [torch.randint(lo, hi + 1, (count,), generator=g, dtype=torch.int64).to(dtype)
            for _ in range(n_ranks)]


def zipf_popularity(n_experts: int, s: float) -> torch.Tensor:
    """Expert popularity p_e proportional to (e+1)^-s, e = 0..n_experts-1 (fp64)."""
    w = torch.arange(1, n_experts + 1, dtype=torch.float64) ** (-s)
    return w / w.sum()


def moe_routing(n_ranks: int, tokens: int, n_experts: int, topk: int, zipf_s: float,
                seed: int) -> list[torch.Tensor]:
    """Per rank, a (tokens, topk) int64 table of distinct expert ids per token.

    Each token draws ``topk`` distinct experts with ``torch.multinomial`` (no replacement)
    from the Zipf popularity, one generator for all ranks, rank order 0..N-1."""
    g = torch.Generator().manual_seed(seed)
    p = zipf_popularity(n_experts, zipf_s).to(torch.float32)
    probs = p.unsqueeze(0).expand(tokens, n_experts).contiguous()
    return [torch.multinomial(probs, topk, replacement=False, generator=g) for _ in range(n_ranks)]


def moe_dispatch(n_ranks: int = 8, tokens: int = 4096, hidden: int = 4096, n_experts: int = 8,
                 topk: int = 2, zipf_s: float = 1.2, seed_tokens: int = 3, seed_route: int = 4,
                 dtype: torch.dtype = torch.bfloat16):
    """An MoE dispatch workload for variable-size all-to-all.

    Returns ``(send, counts, sdispls, rdispls, recv_elems)``:

    * ``send[r]``: rank r's send buffer, rows grouped by destination rank ascending and by
      token index ascending within a group (a token routed to two ranks appears twice);
    * ``counts[i, j]``: elements rank i sends to rank j (rows x hidden), int32 (N, N);
    * ``sdispls[i, j]``: element offset of that block in ``send[i]`` (exclusive prefix over j);
    * ``rdispls[j, i]``: element offset in ``recv[j]`` where rank i's block lands, blocks
      ordered by source rank (exclusive prefix over i of ``counts[:, j]``);
    * ``recv_elems[j]``: total elements rank j receives.

    Expert e lives on rank ``e % n_ranks``.
    """
    g = torch.Generator().manual_seed(seed_tokens)
    tok = [torch.randn(tokens, hidden, generator=g, dtype=torch.float32).to(dtype)
           for _ in range(n_ranks)]
    route = moe_routing(n_ranks, tokens, n_experts, topk, zipf_s, seed_route)
    counts = torch.zeros(n_ranks, n_ranks, dtype=torch.int64)
    send = []
    for r in range(n_ranks):
        dest = route[r] % n_ranks                     # (tokens, topk) destination ranks
        rows = []
        for d in range(n_ranks):
            sel = (dest == d).any(dim=1).nonzero().flatten()
            rows.append(tok[r][sel])
            counts[r, d] = sel.numel() * hidden
        send.append(torch.cat(rows, dim=0).reshape(-1).contiguous())
    sdispls = torch.zeros_like(counts)
    sdispls[:, 1:] = torch.cumsum(counts, dim=1)[:, :-1]
    rdispls = torch.zeros_like(counts)                # indexed [receiver, sender]
    ct = counts.t()
    rdispls[:, 1:] = torch.cumsum(ct, dim=1)[:, :-1]
    recv_elems = ct.sum(dim=1)
    if int(counts.max()) >= 2**31 or int(recv_elems.max()) >= 2**31:
        raise ValueError("a block or buffer does not fit int32 element offsets")
    return (send, counts.to(torch.int32), sdispls.to(torch.int32), rdispls.to(torch.int32),
            [int(x) for x in recv_elems])
