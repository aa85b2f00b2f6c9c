"""CPU oracle for the virtual-rank collectives -- TEST INFRASTRUCTURE.

A thin ctypes layer over ``oracle.c`` (plain C, built with gcc).  Only the tests, the
smoke check and the benchmark's CPU-baseline / reference arm use it; the product path
(``collective_communication_virtual_gb300``) never imports it.

Every function takes a list of N contiguous CPU tensors, one per virtual rank, and
returns new CPU tensors.  The arithmetic lives in ``oracle.c``; this module only
allocates outputs and passes pointers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

DTYPE_CODE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.int32: 3}
OP_CODE = {"sum": 0, "prod": 1, "min": 2, "max": 3}

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (gcc, -O2, no FP contraction, no fast-math)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                        "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm", "-lpthread"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        pp = ctypes.POINTER(ctypes.c_void_p)
        ip = ctypes.POINTER(ctypes.c_int32)
        for name, args in {
            "orc_allreduce": [i32, i32, i32, sz, pp, pp, i32],
            "orc_reduce_scatter": [i32, i32, i32, sz, pp, pp, i32],
            "orc_reduce_scatter_scale": [i32, i32, i32, sz, i32, ctypes.c_float, pp, pp, i32],
            "orc_allgather": [sz, i32, sz, pp, pp],
            "orc_broadcast": [sz, i32, sz, i32, pp, pp],
            "orc_alltoall": [sz, i32, sz, pp, pp],
            "orc_alltoallv": [sz, i32, ip, ip, ip, pp, pp],
            "orc_reduce": [i32, i32, i32, sz, i32, pp, pp, i32],
            "orc_allreduce_tree": [i32, i32, i32, sz, pp, pp, i32],
            "orc_gather": [sz, i32, sz, i32, pp, pp],
            "orc_scatter": [sz, i32, sz, i32, pp, pp],
        }.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, ctypes.c_int
        L.orc_block_elems.argtypes, L.orc_block_elems.restype = [sz, i32, sz], sz
        ipn = ctypes.POINTER(ctypes.c_int)
        L.orc_btree.argtypes, L.orc_btree.restype = [i32, i32, ipn, ipn, ipn], None
        L.orc_dtree.argtypes, L.orc_dtree.restype = [i32, i32, i32, ipn, ipn, ipn], None
        L.orc_f32_to_type.argtypes, L.orc_f32_to_type.restype = [i32, sz, vp, vp], None
        L.orc_type_to_f32.argtypes, L.orc_type_to_f32.restype = [i32, sz, vp, vp], None
        _lib = L
    return _lib


def _ptrs(ts) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = None if t is None else t.data_ptr()
    return arr


def _check(xs):
    for t in xs:
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError("oracle inputs must be contiguous CPU tensors")


def _ok(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def block_elems(count: int, n_ranks: int, elem_size: int) -> int:
    """All-reduce block size B = alignUp(ceil(count/N), 16/elem_size) in elements."""
    return int(lib().orc_block_elems(count, n_ranks, elem_size))


def allreduce(xs, op: str = "sum", nthreads: int = 1):
    _check(xs)
    n, count = len(xs), xs[0].numel()
    out = [torch.empty_like(xs[0]) for _ in range(n)]
    _ok(lib().orc_allreduce(DTYPE_CODE[xs[0].dtype], OP_CODE[op], n, count, _ptrs(xs), _ptrs(out),
                            nthreads), "allreduce")
    return out


def allreduce_tree(xs, op: str = "sum", nthreads: int = 1):
    """Double-binary-tree all-reduce (first half up tree 0, second half up tree 1)."""
    _check(xs)
    n, count = len(xs), xs[0].numel()
    out = [torch.empty_like(xs[0]) for _ in range(n)]
    _ok(lib().orc_allreduce_tree(DTYPE_CODE[xs[0].dtype], OP_CODE[op], n, count, _ptrs(xs), _ptrs(out),
                                 nthreads), "allreduce_tree")
    return out


def tree_links(n: int, rank: int, tree: int = 0):
    """(parent, child0, child1) of `rank` in tree 0 or 1 of the double binary tree."""
    u, a, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    lib().orc_dtree(n, rank, tree, ctypes.byref(u), ctypes.byref(a), ctypes.byref(b))
    return u.value, a.value, b.value


def reduce_scatter(xs, op: str = "sum", nthreads: int = 1):
    _check(xs)
    n, count = len(xs), xs[0].numel()
    if count % n:
        raise ValueError("reduce-scatter send count must be a multiple of N")
    rc = count // n
    out = [torch.empty(rc, dtype=xs[0].dtype) for _ in range(n)]
    _ok(lib().orc_reduce_scatter(DTYPE_CODE[xs[0].dtype], OP_CODE[op], n, rc, _ptrs(xs), _ptrs(out),
                                 nthreads), "reduce_scatter")
    return out


def reduce_scatter_scale(xs, op: str, scale: float, out_dtype=torch.float32, nthreads: int = 1):
    """Reduce-scatter with the fused epilogue out = (float)acc * scale, stored as out_dtype."""
    _check(xs)
    n, count = len(xs), xs[0].numel()
    if count % n:
        raise ValueError("reduce-scatter send count must be a multiple of N")
    rc = count // n
    out = [torch.empty(rc, dtype=out_dtype) for _ in range(n)]
    _ok(lib().orc_reduce_scatter_scale(DTYPE_CODE[xs[0].dtype], OP_CODE[op], n, rc,
                                       DTYPE_CODE[out_dtype], ctypes.c_float(scale), _ptrs(xs),
                                       _ptrs(out), nthreads), "reduce_scatter_scale")
    return out


def reduce(xs, op: str = "sum", root: int = 0, nthreads: int = 1):
    """Reduce to root; returns the root's result (one tensor)."""
    _check(xs)
    n, count = len(xs), xs[0].numel()
    out = [None] * n
    out[root] = torch.empty_like(xs[0])
    _ok(lib().orc_reduce(DTYPE_CODE[xs[0].dtype], OP_CODE[op], n, count, root, _ptrs(xs), _ptrs(out),
                         nthreads), "reduce")
    return out[root]


def gather(xs, root: int = 0):
    """Gather to root; returns the root's buffer (N * sendcount elements)."""
    _check(xs)
    n, sc = len(xs), xs[0].numel()
    out = [None] * n
    out[root] = torch.empty(n * sc, dtype=xs[0].dtype)
    _ok(lib().orc_gather(xs[0].element_size(), n, sc, root, _ptrs(xs), _ptrs(out)), "gather")
    return out[root]


def scatter(src, n: int, root: int = 0):
    """Scatter the root's buffer (n blocks) to n ranks; returns the n receive buffers."""
    _check([src])
    if src.numel() % n:
        raise ValueError("scatter source must hold n equal blocks")
    rc = src.numel() // n
    send = [None] * n
    send[root] = src
    out = [torch.empty(rc, dtype=src.dtype) for _ in range(n)]
    _ok(lib().orc_scatter(src.element_size(), n, rc, root, _ptrs(send), _ptrs(out)), "scatter")
    return out


def allgather(xs):
    _check(xs)
    n, sc = len(xs), xs[0].numel()
    out = [torch.empty(n * sc, dtype=xs[0].dtype) for _ in range(n)]
    _ok(lib().orc_allgather(xs[0].element_size(), n, sc, _ptrs(xs), _ptrs(out)), "allgather")
    return out


def broadcast(xs, root: int = 0):
    _check(xs)
    src = xs[root]
    n = len(xs)
    out = [torch.empty_like(src) for _ in range(n)]
    _ok(lib().orc_broadcast(src.element_size(), n, src.numel(), root, _ptrs(xs), _ptrs(out)),
        "broadcast")
    return out


def alltoall(xs):
    _check(xs)
    n, total = len(xs), xs[0].numel()
    if total % n:
        raise ValueError("uniform all-to-all buffers must hold N equal blocks")
    out = [torch.empty_like(xs[0]) for _ in range(n)]
    _ok(lib().orc_alltoall(xs[0].element_size(), n, total // n, _ptrs(xs), _ptrs(out)), "alltoall")
    return out


def alltoallv(xs, counts, sdispls, rdispls, recv_elems):
    """counts/sdispls indexed [sender, receiver]; rdispls indexed [receiver, sender]."""
    _check(xs)
    n = len(xs)
    tabs = [t.to(torch.int32).contiguous() for t in (counts, sdispls, rdispls)]
    ip = ctypes.POINTER(ctypes.c_int32)
    out = [torch.zeros(int(recv_elems[j]), dtype=xs[0].dtype) for j in range(n)]
    _ok(lib().orc_alltoallv(xs[0].element_size(), n,
                            *[ctypes.cast(t.data_ptr(), ip) for t in tabs],
                            _ptrs(xs), _ptrs(out)), "alltoallv")
    return out


def from_f32(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Round fp32 values to ``dtype`` with the oracle's own converter (for pinning it)."""
    x = x.to(torch.float32).contiguous()
    out = torch.empty(x.numel(), dtype=dtype)
    lib().orc_f32_to_type(DTYPE_CODE[dtype], x.numel(), x.data_ptr(), out.data_ptr())
    return out


def to_f32(x: torch.Tensor) -> torch.Tensor:
    """Widen fp16/bf16 values to fp32 with the oracle's own converter."""
    x = x.contiguous()
    out = torch.empty(x.numel(), dtype=torch.float32)
    lib().orc_type_to_f32(DTYPE_CODE[x.dtype], x.numel(), x.data_ptr(), out.data_ptr())
    return out
