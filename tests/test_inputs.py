"""The seeded input recipes, on the CPU: the shapes, distributions and structure that the
workloads are stated with (uniform and normal buffers, the 25 MiB FSDP bucket, the MoE
token dispatch with top-2 routing over a Zipf(1.2) expert popularity)."""
from __future__ import annotations

import torch

from collective_communication_virtual_gb300 import inputs


def test_uniform_and_int_ranges_and_seeding():
    a = inputs.uniform_ranks(3, 10_000, torch.float32, 5)
    b = inputs.uniform_ranks(3, 10_000, torch.float32, 5)
    assert all(torch.equal(x, y) for x, y in zip(a, b))              # seeded
    assert not torch.equal(a[0], a[1])                               # ranks differ
    for x in a:
        assert float(x.min()) >= -1.0 and float(x.max()) < 1.0
        assert abs(float(x.mean())) < 0.05
    for x in inputs.uniform_ranks(2, 10_000, torch.int32, 5):
        assert x.dtype == torch.int32
        assert int(x.min()) >= inputs.INT32_LO and int(x.max()) <= inputs.INT32_HI
    for x in inputs.uniform_ranks(2, 1000, torch.bfloat16, 5):
        assert x.dtype == torch.bfloat16


def test_fsdp_bucket_is_normal_with_the_stated_spread():
    g = inputs.normal_ranks(2, 13_107_200 // 64, 1e-3, torch.bfloat16, 2)
    for x in g:
        assert x.dtype == torch.bfloat16
        assert abs(float(x.float().std()) - 1e-3) < 5e-5
        assert abs(float(x.float().mean())) < 5e-5


def test_moe_dispatch_structure():
    n, tokens, hidden = 8, 512, 16
    send, counts, sd, rd, recv_elems = inputs.moe_dispatch(n_ranks=n, tokens=tokens, hidden=hidden)
    assert counts.dtype == sd.dtype == rd.dtype == torch.int32
    # every token goes to exactly 2 distinct experts, one expert per rank here
    assert torch.equal(counts.sum(1), torch.full((n,), 2 * tokens * hidden, dtype=torch.int64).to(counts.dtype))
    for r in range(n):
        assert send[r].numel() == int(counts[r].sum())
    # displacements: exclusive prefix sums, senders' blocks ordered by destination and the
    # receivers' blocks by source
    assert torch.equal(sd, (torch.cumsum(counts, 1) - counts).to(torch.int32))
    assert torch.equal(rd, (torch.cumsum(counts, 0) - counts).t().contiguous().to(torch.int32))
    assert [int(v) for v in recv_elems] == [int(v) for v in counts.sum(0)]
    # Zipf(1.2) popularity: expert 0 (rank 0) receives the most, the last expert the least
    per_dest = counts.sum(0).float()
    assert int(per_dest.argmax()) == 0 and int(per_dest.argmin()) == n - 1
    p = inputs.zipf_popularity(8, 1.2)
    assert abs(float(p.sum()) - 1.0) < 1e-9
    assert all(float(p[i]) > float(p[i + 1]) for i in range(7))
    assert abs(float(p[0] / p[1]) - 2 ** 1.2) < 1e-6


def test_moe_rows_are_the_routed_tokens_in_order():
    n, tokens, hidden = 4, 64, 8
    send, counts, sd, _, _ = inputs.moe_dispatch(n_ranks=n, tokens=tokens, hidden=hidden)
    route = inputs.moe_routing(n, tokens, 8, 2, 1.2, 4)
    g = torch.Generator().manual_seed(3)
    tok = [torch.randn(tokens, hidden, generator=g, dtype=torch.float32).to(torch.bfloat16) for _ in range(n)]
    for r in range(n):
        dest = route[r] % n
        for d in range(n):
            sel = [t for t in range(tokens) if bool((dest[t] == d).any())]
            block = send[r][int(sd[r, d]):int(sd[r, d]) + int(counts[r, d])].view(-1, hidden)
            assert block.shape[0] == len(sel)
            if sel:
                assert torch.equal(block, tok[r][sel])
