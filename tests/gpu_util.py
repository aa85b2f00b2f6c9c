"""Helpers shared by the GPU tests: device copies of seeded inputs, bit comparison, and
a cache of communicators."""
from __future__ import annotations

import torch

from collective_communication_virtual_gb300 import vcomm as V

DEV = torch.device("cuda:0")


def to_dev(xs, pad_elems: int = 0):
    """Device copies; with pad_elems > 0 each buffer starts pad_elems elements into a
    larger allocation (so it is not 16-byte aligned when pad_elems * esz % 16 != 0)."""
    out = []
    for x in xs:
        if pad_elems:
            big = torch.empty(x.numel() + pad_elems, dtype=x.dtype, device=DEV)
            v = big[pad_elems:]
            v.copy_(x)
            out.append(v)
        else:
            out.append(x.to(DEV))
    return out


def empty_dev(n, count, dtype, pad_elems: int = 0, fill=None):
    out = []
    for _ in range(n):
        big = torch.empty(count + pad_elems, dtype=dtype, device=DEV)
        if fill is not None:
            big.fill_(fill)
        out.append(big[pad_elems:] if pad_elems else big)
    return out


def bits(t: torch.Tensor) -> torch.Tensor:
    t = t.detach().cpu().contiguous()
    return t.view({4: torch.int32, 2: torch.int16}[t.element_size()])


def assert_bits_equal(got, want, what=""):
    assert len(got) == len(want)
    for r, (g, w) in enumerate(zip(got, want)):
        gb, wb = bits(g), bits(w)
        if not torch.equal(gb, wb):
            diff = (gb != wb).nonzero().flatten()
            i = int(diff[0])
            raise AssertionError(f"{what}: rank {r}: {diff.numel()} elements differ, first at {i}: "
                                 f"got {g.cpu()[i].item()!r} want {w[i].item()!r}")


class Comms:
    """Communicators keyed by (nRanks, nChannels, protocol); destroyed at the end."""

    def __init__(self):
        self._c = {}

    def get(self, n, channels=1, proto=V.vProtoSimple, algo="auto", chunk=None, timeout_ms=2000):
        key = (n, channels, proto)
        if key not in self._c:
            self._c[key] = V.vcommInit(n, channels, proto)
        c = self._c[key]
        V.vcommSetAlgo(c, algo)
        V.vcommSetTimeoutMs(c, timeout_ms)
        V.vcommSetChunkBytes(c, chunk or 0)
        return c

    def close(self):
        for c in self._c.values():
            V.vcommDestroy(c)
        self._c.clear()
