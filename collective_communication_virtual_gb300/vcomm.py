"""ctypes binding of libvcomm (include/vcomm.h): the same entry points, argument
marshalling only.  Every collective runs in the library's CUDA kernels; there is no
Python or CPU fallback -- if the library is missing or a call fails, an exception is
raised.

Buffers may be given as torch tensors or as integer device addresses; ``datatype`` as a
torch dtype or a ``vDataType_t`` value; ``stream`` as a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or ``None`` for torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

# ---- enums (values of include/vcomm.h) ---------------------------------------------------
vSuccess, vUnhandledCudaError, vSystemError, vInternalError = 0, 1, 2, 3
vInvalidArgument, vInvalidUsage, vTimeout, vInProgress, vAborted = 4, 5, 6, 7, 8
vFloat32, vFloat16, vBFloat16, vInt32 = 0, 1, 2, 3
vSum, vProd, vMin, vMax = 0, 1, 2, 3
vProtoSimple, vProtoLL, vProtoLL128, vProtoAuto = 0, 1, 2, 3
vAlgoAuto, vAlgoOnePass, vAlgoRing, vAlgoTree = 0, 1, 2, 3
vCollAllReduce, vCollReduceScatter, vCollAllGather = 0, 1, 2
vCollBroadcast, vCollAllToAll, vCollAllToAllv = 3, 4, 5
vCollReduce, vCollGather, vCollScatter = 6, 7, 8
VCOMM_MAX_RANKS = 64

RESULT_NAMES = {0: "vSuccess", 1: "vUnhandledCudaError", 2: "vSystemError", 3: "vInternalError",
                4: "vInvalidArgument", 5: "vInvalidUsage", 6: "vTimeout", 7: "vInProgress",
                8: "vAborted"}
OPS = {"sum": vSum, "prod": vProd, "min": vMin, "max": vMax}
PROTOCOLS = {"simple": vProtoSimple, "ll": vProtoLL, "ll128": vProtoLL128, "auto": vProtoAuto}
ALGOS = {"auto": vAlgoAuto, "onepass": vAlgoOnePass, "ring": vAlgoRing, "tree": vAlgoTree}


class VcommError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {RESULT_NAMES.get(code, code)}")


class vPlanRequest_t(ctypes.Structure):
    _fields_ = [("nRanks", ctypes.c_int), ("nChannels", ctypes.c_int), ("proto", ctypes.c_int),
                ("algo", ctypes.c_int), ("coll", ctypes.c_int), ("datatype", ctypes.c_int),
                ("count", ctypes.c_size_t), ("chunkBytes", ctypes.c_size_t),
                ("aligned16", ctypes.c_int), ("smCount", ctypes.c_int), ("l2Bytes", ctypes.c_size_t),
                ("aligned32", ctypes.c_int), ("noBulkCopy", ctypes.c_int), ("persistentGrid", ctypes.c_int)]


class vPlanInfo_t(ctypes.Structure):
    _fields_ = [("algo", ctypes.c_int), ("proto", ctypes.c_int), ("nChannels", ctypes.c_int),
                ("ctasPerChannel", ctypes.c_int), ("gridCtas", ctypes.c_int),
                ("threadsPerCta", ctypes.c_int), ("vectorized", ctypes.c_int),
                ("launches", ctypes.c_int), ("blockElems", ctypes.c_size_t),
                ("channelElems", ctypes.c_size_t), ("chunkElems", ctypes.c_size_t),
                ("slotPayloadElems", ctypes.c_size_t), ("slotBytes", ctypes.c_size_t),
                ("fifoBytes", ctypes.c_size_t), ("minBytes", ctypes.c_double),
                ("busFactor", ctypes.c_double), ("vecBytes", ctypes.c_int), ("bulkCopy", ctypes.c_int),
                ("predictedUs", ctypes.c_double), ("tileBytes", ctypes.c_size_t), ("tmaStages", ctypes.c_int)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None

_SIGNATURES = {
    "vcommInit": ([ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_int, ctypes.c_int], ctypes.c_int),
    "vcommDestroy": ([ctypes.c_void_p], ctypes.c_int),
    "vcommGetAsyncError": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "vcommAbort": ([ctypes.c_void_p], ctypes.c_int),
    "vcommGetErrorString": ([ctypes.c_int], ctypes.c_char_p),
    "vcommSetAlgo": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "vcommGroupStart": ([ctypes.c_void_p], ctypes.c_int),
    "vcommGroupEnd": ([ctypes.c_void_p], ctypes.c_int),
    "vcommSetProtocol": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "vcommSetChunkBytes": ([ctypes.c_void_p, ctypes.c_size_t], ctypes.c_int),
    "vcommSetTimeoutMs": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "vcommTestSetStallRank": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "vcommQueryPlan": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                        ctypes.POINTER(vPlanInfo_t)], ctypes.c_int),
    "vPlanCompute": ([ctypes.POINTER(vPlanRequest_t), ctypes.POINTER(vPlanInfo_t)], ctypes.c_int),
    "vPlanTreeLinks": ([ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "vPlanChannelRange": ([ctypes.POINTER(vPlanInfo_t), ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                           ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "vAllReduce": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                    ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vReduceScatter": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                        ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vReduceScatterScaleCast": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vAllGather": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                    ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vBroadcast": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                    ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vAllToAll": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vcommCount": ([ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vcommTestSetJitterNs": ([ctypes.c_void_p, ctypes.c_uint], ctypes.c_int),
    "vcommTestSetBadFlagRank": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "vAllToAllv": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                    ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vReduce": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                 ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vGather": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                 ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vScatter": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "vAllReduceNoAlloc": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
}


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libvcomm.so (built in-tree by ``build.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libvcomm.so is not built ({path}); run "
                               "collective_communication_virtual_gb300.build.build() first")
        L = ctypes.CDLL(path)
        for name, (args, res) in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, res
        _lib = L
    return _lib


# ---- marshalling helpers -------------------------------------------------------------------

_DTYPE_CODES: dict = {}
_ARRAY_TYPES: dict = {}


def _dtype_code(dt) -> int:
    if isinstance(dt, int):
        return dt
    if not _DTYPE_CODES:
        import torch
        _DTYPE_CODES.update({torch.float32: vFloat32, torch.float16: vFloat16, torch.bfloat16: vBFloat16,
                             torch.int32: vInt32})
    return _DTYPE_CODES[dt]


def _op_code(op) -> int:
    return OPS[op] if isinstance(op, str) else int(op)


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _ptr_array(bufs, n_ranks: int):
    """A C array of the buffers' device addresses (None for NULL).  The library reads
    exactly n_ranks entries, so a list of another length is refused here."""
    n = len(bufs)
    if n != n_ranks:
        raise VcommError(vInvalidArgument, f"expected {n_ranks} buffers (one per rank), got {n}")
    arr_t = _ARRAY_TYPES.get(n)
    if arr_t is None:
        arr_t = _ARRAY_TYPES[n] = ctypes.c_void_p * n
    return arr_t(*[None if b is None else (b if isinstance(b, int) else b.data_ptr()) for b in bufs])


_N_RANKS: dict = {}


def _handle(comm) -> int | None:
    return comm.value if isinstance(comm, ctypes.c_void_p) else comm


def _n_ranks(comm) -> int:
    """The communicator's rank count, asked of the library once per handle."""
    key = _handle(comm)
    n = _N_RANKS.get(key)
    if n is None:
        v = ctypes.c_int(0)
        _check(lib().vcommCount(comm, ctypes.byref(v)), "vcommCount")
        n = _N_RANKS[key] = v.value
    return n


def _pair(comm, sendbuffs, recvbuffs):
    n = _n_ranks(comm)
    return _ptr_array(sendbuffs, n), _ptr_array(recvbuffs, n)


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != vSuccess:
        raise VcommError(code, where)


# ---- the C ABI, one wrapper per entry point --------------------------------------------------

def vcommInit(n_ranks: int, n_channels: int = 1, protocol=vProtoSimple) -> ctypes.c_void_p:
    comm = ctypes.c_void_p()
    proto = PROTOCOLS[protocol] if isinstance(protocol, str) else protocol
    _check(lib().vcommInit(ctypes.byref(comm), n_ranks, n_channels, proto), "vcommInit")
    _N_RANKS[comm.value] = n_ranks
    return comm


def vcommDestroy(comm) -> None:
    _N_RANKS.pop(_handle(comm), None)
    _check(lib().vcommDestroy(comm), "vcommDestroy")


def vcommCount(comm) -> int:
    v = ctypes.c_int(0)
    _check(lib().vcommCount(comm, ctypes.byref(v)), "vcommCount")
    return v.value


def vcommGetAsyncError(comm) -> int:
    err = ctypes.c_int(0)
    _check(lib().vcommGetAsyncError(comm, ctypes.byref(err)), "vcommGetAsyncError")
    return err.value


def vcommAbort(comm) -> None:
    _check(lib().vcommAbort(comm), "vcommAbort")


def vcommGetErrorString(code: int) -> str:
    return lib().vcommGetErrorString(code).decode()


def vcommGroupStart(comm) -> None:
    _check(lib().vcommGroupStart(comm), "vcommGroupStart")


def vcommGroupEnd(comm) -> None:
    _check(lib().vcommGroupEnd(comm), "vcommGroupEnd")


def vcommSetAlgo(comm, algo) -> None:
    _check(lib().vcommSetAlgo(comm, ALGOS[algo] if isinstance(algo, str) else algo), "vcommSetAlgo")


def vcommSetProtocol(comm, protocol) -> None:
    proto = PROTOCOLS[protocol] if isinstance(protocol, str) else protocol
    _check(lib().vcommSetProtocol(comm, proto), "vcommSetProtocol")


def vcommSetChunkBytes(comm, chunk_bytes: int) -> None:
    _check(lib().vcommSetChunkBytes(comm, chunk_bytes), "vcommSetChunkBytes")


def vcommSetTimeoutMs(comm, ms: int) -> None:
    _check(lib().vcommSetTimeoutMs(comm, ms), "vcommSetTimeoutMs")


def vcommTestSetStallRank(comm, rank: int) -> None:
    _check(lib().vcommTestSetStallRank(comm, rank), "vcommTestSetStallRank")


def vcommTestSetBadFlagRank(comm, rank: int) -> None:
    _check(lib().vcommTestSetBadFlagRank(comm, rank), "vcommTestSetBadFlagRank")


def vcommTestSetJitterNs(comm, max_ns: int) -> None:
    _check(lib().vcommTestSetJitterNs(comm, max_ns), "vcommTestSetJitterNs")


def vcommQueryPlan(comm, coll: int, count: int, datatype, aligned: int = 32) -> dict:
    """The plan for buffers whose pointers share `aligned`-byte alignment (1..32)."""
    info = vPlanInfo_t()
    _check(lib().vcommQueryPlan(comm, coll, count, _dtype_code(datatype), int(aligned),
                                ctypes.byref(info)), "vcommQueryPlan")
    return info.as_dict()


def vPlanCompute(**req) -> vPlanInfo_t:
    q = vPlanRequest_t()
    for k, v in req.items():
        setattr(q, k, v)
    info = vPlanInfo_t()
    _check(lib().vPlanCompute(ctypes.byref(q), ctypes.byref(info)), "vPlanCompute")
    return info


def vPlanTreeLinks(n_ranks: int, rank: int, tree: int = 0) -> tuple[int, int, int]:
    u, a, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().vPlanTreeLinks(n_ranks, rank, tree, ctypes.byref(u), ctypes.byref(a), ctypes.byref(b)),
           "vPlanTreeLinks")
    return u.value, a.value, b.value


def vPlanChannelRange(plan: vPlanInfo_t, count: int, channel: int, block: int) -> tuple[int, int]:
    lo, hi = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().vPlanChannelRange(ctypes.byref(plan), count, channel, block, ctypes.byref(lo),
                                   ctypes.byref(hi)), "vPlanChannelRange")
    return lo.value, hi.value


def vAllReduce(sendbuffs, recvbuffs, count: int, datatype, op, comm, stream=None) -> None:
    _check(lib().vAllReduce(*_pair(comm, sendbuffs, recvbuffs), count, _dtype_code(datatype),
                            _op_code(op), comm, _stream(stream)), "vAllReduce")


def vReduceScatter(sendbuffs, recvbuffs, recvcount: int, datatype, op, comm, stream=None) -> None:
    _check(lib().vReduceScatter(*_pair(comm, sendbuffs, recvbuffs), recvcount,
                                _dtype_code(datatype), _op_code(op), comm, _stream(stream)), "vReduceScatter")


def vReduceScatterScaleCast(sendbuffs, recvbuffs, recvcount: int, datatype, op, out_type, scale: float,
                            comm, stream=None) -> None:
    _check(lib().vReduceScatterScaleCast(*_pair(comm, sendbuffs, recvbuffs), recvcount,
                                         _dtype_code(datatype), _op_code(op), _dtype_code(out_type),
                                         ctypes.c_float(scale), comm, _stream(stream)),
           "vReduceScatterScaleCast")


def vAllGather(sendbuffs, recvbuffs, sendcount: int, datatype, op, comm, stream=None) -> None:
    _check(lib().vAllGather(*_pair(comm, sendbuffs, recvbuffs), sendcount, _dtype_code(datatype),
                            _op_code(op), comm, _stream(stream)), "vAllGather")


def vBroadcast(sendbuffs, recvbuffs, count: int, datatype, op, root: int, comm, stream=None) -> None:
    _check(lib().vBroadcast(*_pair(comm, sendbuffs, recvbuffs), count, _dtype_code(datatype),
                            _op_code(op), root, comm, _stream(stream)), "vBroadcast")


def vAllToAll(sendbuffs, recvbuffs, count: int, datatype, op, comm, stream=None) -> None:
    _check(lib().vAllToAll(*_pair(comm, sendbuffs, recvbuffs), count, _dtype_code(datatype),
                           _op_code(op), comm, _stream(stream)), "vAllToAll")


def vReduce(sendbuffs, recvbuffs, count: int, datatype, op, root: int, comm, stream=None) -> None:
    _check(lib().vReduce(*_pair(comm, sendbuffs, recvbuffs), count, _dtype_code(datatype),
                         _op_code(op), root, comm, _stream(stream)), "vReduce")


def vGather(sendbuffs, recvbuffs, sendcount: int, datatype, root: int, comm, stream=None) -> None:
    _check(lib().vGather(*_pair(comm, sendbuffs, recvbuffs), sendcount, _dtype_code(datatype),
                         root, comm, _stream(stream)), "vGather")


def vScatter(sendbuffs, recvbuffs, recvcount: int, datatype, root: int, comm, stream=None) -> None:
    _check(lib().vScatter(*_pair(comm, sendbuffs, recvbuffs), recvcount, _dtype_code(datatype),
                          root, comm, _stream(stream)), "vScatter")


def vAllToAllv(sendbuffs, recvbuffs, counts, sdispls, rdispls, datatype, comm, stream=None) -> None:
    _check(lib().vAllToAllv(*_pair(comm, sendbuffs, recvbuffs), _addr(counts), _addr(sdispls),
                            _addr(rdispls), _dtype_code(datatype), comm, _stream(stream)), "vAllToAllv")


def vAllReduceNoAlloc(sendbuffs, recvbuffs, count: int, datatype, op, n_ranks: int, n_channels: int = 1,
                      protocol=vProtoSimple, stream=None) -> None:
    """The ring all-reduce that allocates nothing (see include/vcomm.h)."""
    proto = PROTOCOLS[protocol] if isinstance(protocol, str) else protocol
    _check(lib().vAllReduceNoAlloc(_ptr_array(sendbuffs, n_ranks), _ptr_array(recvbuffs, n_ranks), count, _dtype_code(datatype),
                                   _op_code(op), n_ranks, n_channels, proto, _stream(stream)),
           "vAllReduceNoAlloc")
