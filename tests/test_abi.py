"""The C-ABI library without a GPU: it builds, loads, exports every entry point that
include/vcomm.h declares, and rejects bad arguments before touching CUDA."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest
import torch

from collective_communication_virtual_gb300 import build, vcomm as V

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "vcomm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return V.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^(?:vResult_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_collectives():
    names = declared_functions()
    for n in ["vcommInit", "vcommDestroy", "vcommGetAsyncError", "vAllReduce", "vReduceScatter",
              "vReduceScatterScaleCast", "vAllGather", "vBroadcast", "vAllToAll", "vAllToAllv",
              "vReduce", "vGather", "vScatter",
              "vPlanCompute"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", V.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None
    # and the other way round: every unmangled function the library exports is declared
    text_syms = {line.split()[-1] for line in out.splitlines() if len(line.split()) == 3 and line.split()[1] == "T"}
    undeclared = sorted(n for n in text_syms if not n.startswith("_Z") and n not in declared_functions())
    assert not undeclared, undeclared


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "vcomm.h"\nint main(void){vcomm_t c = 0; (void)c; return 0;}\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c",
                    str(src), "-o", str(tmp_path / "t.o")], check=True)


def test_init_rejects_bad_arguments_before_cuda(lib):
    comm = ctypes.c_void_p(123)
    for n, ch, proto in [(0, 1, 0), (65, 1, 0), (4, 0, 0), (4, 65, 0), (4, 1, 7), (-1, 1, 0)]:
        assert lib.vcommInit(ctypes.byref(comm), n, ch, proto) == V.vInvalidArgument
        assert comm.value is None
    assert lib.vcommInit(None, 4, 1, 0) == V.vInvalidArgument


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_init_without_gpu_reports_cuda_error(lib):
    comm = ctypes.c_void_p()
    assert lib.vcommInit(ctypes.byref(comm), 4, 1, 0) == V.vUnhandledCudaError
    assert comm.value is None


def test_null_or_garbage_comm_is_refused(lib):
    arr = (ctypes.c_void_p * 4)()
    garbage = ctypes.create_string_buffer(4096)
    for comm in (None, ctypes.addressof(garbage)):
        assert lib.vAllReduce(arr, arr, 16, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vReduceScatter(arr, arr, 16, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vAllGather(arr, arr, 16, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vBroadcast(arr, arr, 16, 0, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vAllToAll(arr, arr, 16, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vAllToAllv(arr, arr, None, None, None, 0, comm, None) == V.vInvalidArgument
        assert lib.vReduce(arr, arr, 16, 0, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vGather(arr, arr, 16, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vScatter(arr, arr, 16, 0, 0, comm, None) == V.vInvalidArgument
        assert lib.vcommGroupStart(comm) == V.vInvalidArgument
        assert lib.vcommGroupEnd(comm) == V.vInvalidArgument
        assert lib.vcommDestroy(comm) == V.vInvalidArgument
        assert lib.vcommAbort(comm) == V.vInvalidArgument
        err = ctypes.c_int()
        assert lib.vcommGetAsyncError(comm, ctypes.byref(err)) == V.vInvalidArgument
        assert lib.vcommCount(comm, ctypes.byref(err)) == V.vInvalidArgument


def test_binding_refuses_a_buffer_list_of_the_wrong_length(monkeypatch):
    # the library reads exactly N pointers from each array, so the binding checks the
    # lengths against the communicator's rank count before calling it
    calls = []

    class FakeLib:
        def vAllReduce(self, *args):
            calls.append(args)
            return V.vSuccess

    monkeypatch.setattr(V, "lib", lambda: FakeLib())
    monkeypatch.setitem(V._N_RANKS, 0x1234, 4)
    comm = ctypes.c_void_p(0x1234)
    with pytest.raises(V.VcommError) as e:
        V.vAllReduce([1, 2, 3], [4, 5, 6, 7], 16, V.vFloat32, "sum", comm, stream=0)
    assert e.value.code == V.vInvalidArgument and not calls
    with pytest.raises(V.VcommError):
        V.vAllReduce([1, 2, 3, 4], [4, 5, 6, 7, 8], 16, V.vFloat32, "sum", comm, stream=0)
    assert not calls
    V.vAllReduce([1, 2, 3, 4], [5, 6, 7, 8], 16, V.vFloat32, "sum", comm, stream=0)
    assert len(calls) == 1 and list(calls[0][0]) == [1, 2, 3, 4] and list(calls[0][1]) == [5, 6, 7, 8]


def test_error_strings(lib):
    assert V.vcommGetErrorString(V.vSuccess) == "no error"
    assert V.vcommGetErrorString(V.vInvalidUsage) == "invalid usage"
    assert V.vcommGetErrorString(V.vTimeout) == "timeout"
    assert V.vcommGetErrorString(99) == "unknown result code"


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(V, "_lib", None)
    monkeypatch.setattr(V, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        V.lib()
