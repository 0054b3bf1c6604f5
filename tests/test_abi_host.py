"""CPU-side checks of the C-ABI library: it loads, it exports every entry point
include/diffuser.h declares, and host-side argument checks reject bad input
before touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from sparse_long_sequence_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    path = cuda_build.build()
    return ctypes.CDLL(path)


def declared_entry_points():
    names = []
    for fname in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fname.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fname)).read()
            names += re.findall(r"DIFFUSER_API\s+[\w\s\*]*?\b(diffuser_\w+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for must in ("diffuser_build_graph", "diffuser_build_causal_graph",
                 "diffuser_build_block_graph", "diffuser_forward",
                 "diffuser_workspace_size", "diffuser_graph_copy_csr", "diffuser_graph_free"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), f"{name} declared but not exported"


def test_only_the_c_abi_is_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", cuda_build.LIB], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_entry_points())


def test_status_strings(lib):
    lib.diffuser_status_string.restype = ctypes.c_char_p
    assert lib.diffuser_status_string(0) == b"ok"
    for code in range(1, 8):
        assert lib.diffuser_status_string(code) not in (b"ok", b"unknown status")
    assert lib.diffuser_status_string(99) == b"unknown status"


def test_invalid_arguments_rejected_on_host(lib):
    vp = ctypes.c_void_p
    out = vp()
    i64, i32, u64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
    f = lib.diffuser_build_graph
    f.argtypes = [i64, i32, i32, ctypes.POINTER(i32), i32, u64, ctypes.POINTER(vp)]
    assert f(0, 1, 0, None, 0, 0, ctypes.byref(out)) == 1          # n < 1
    assert f(10, -1, 0, None, 0, 0, ctypes.byref(out)) == 1        # r < 0
    assert f(10, 1, 11, None, 0, 0, ctypes.byref(out)) == 1        # g > n
    assert f(10, 1, 0, None, 2000, 0, ctypes.byref(out)) == 1      # R too large
    bad = (i32 * 2)(5, 3)                                          # not increasing
    assert f(10, 1, 2, bad, 0, 0, ctypes.byref(out)) == 1
    assert f(10, 1, 0, None, 0, 0, None) == 1                      # null out
    fc = lib.diffuser_build_causal_graph
    fc.argtypes = f.argtypes
    assert fc(0, 1, 0, None, 0, 0, ctypes.byref(out)) == 1         # n < 1
    assert fc(10, -1, 0, None, 0, 0, ctypes.byref(out)) == 1       # r < 0
    assert fc(10, 1, 2, bad, 0, 0, ctypes.byref(out)) == 1         # not increasing
    fd = lib.diffuser_build_dilated_graph
    fd.argtypes = [i64, i32, i32, i32, ctypes.POINTER(i32), i32, u64, i32, ctypes.POINTER(vp)]
    assert fd(10, 1, 0, 0, None, 0, 0, 0, ctypes.byref(out)) == 1   # dilation < 1
    assert fd(10, -1, 2, 0, None, 0, 0, 0, ctypes.byref(out)) == 1  # r < 0
    fb = lib.diffuser_build_block_graph
    fb.argtypes = [i64, i32, i32, i32, i32, u64, ctypes.POINTER(vp)]
    assert fb(100, 16, 2, 1, 1, 0, ctypes.byref(out)) == 1         # even window
    assert fb(100, 16, 3, 1, 9, 0, ctypes.byref(out)) == 1         # too many global blocks
    assert fb(100, 0, 3, 1, 1, 0, ctypes.byref(out)) == 1          # block < 1
    ws = lib.diffuser_workspace_size
    ws.argtypes = [vp, i64, i64, i32, i32, ctypes.POINTER(ctypes.c_size_t)]
    nbytes = ctypes.c_size_t()
    assert ws(None, 1, 1, 64, 1, ctypes.byref(nbytes)) == 1        # null graph
    fw = lib.diffuser_forward
    fw.argtypes = [vp, vp, vp, i32, i64, i64, i32, vp, i32, ctypes.c_float, vp, vp,
                   ctypes.c_size_t, vp]
    assert fw(None, None, None, 1, 1, 1, 64, None, 5, 0.1, None, None, 0, None) == 1
    bws = lib.diffuser_backward_workspace_size
    bws.argtypes = [vp, i64, i64, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)]
    assert bws(None, 1, 1, 64, 1, 5, ctypes.byref(nbytes)) == 1   # null graph
    bw = lib.diffuser_backward
    bw.argtypes = [vp, vp, vp, vp, i32, i64, i64, i32, vp, i32, ctypes.c_float, vp, vp, vp, vp,
                   ctypes.c_size_t, vp]
    assert bw(None, None, None, None, 1, 1, 1, 64, None, 5, 0.1, None, None, None, None, 0,
              None) == 1
    lib.diffuser_last_error.restype = ctypes.c_char_p
    assert lib.diffuser_last_error() != b""


def test_launch_counter_and_profiler_without_gpu(lib):
    arr = (ctypes.c_int64 * 5)()
    lib.diffuser_launch_count.restype = ctypes.c_int64
    before = lib.diffuser_launch_count(arr)
    assert before == sum(arr)
    assert lib.diffuser_profile_begin() == 0
    assert lib.diffuser_profile_begin() == 1     # one profile at a time
    ms = (ctypes.c_double * 5)()
    cnt = (ctypes.c_int64 * 5)()
    assert lib.diffuser_profile_end(ms, cnt) == 0
    assert list(cnt) == [0, 0, 0, 0, 0]
    assert lib.diffuser_profile_end(ms, cnt) == 1
    assert lib.diffuser_launch_count(None) == before   # failed calls launched nothing
