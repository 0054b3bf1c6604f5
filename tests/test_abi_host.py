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


def test_every_other_entry_point_rejects_bad_arguments_on_host(lib):
    # each of these returns before any device call: INVALID_ARG (1) for a NULL or an
    # out-of-range argument, UNSUPPORTED (2) for a head width or model width it lacks
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    out, nbytes = vp(), sz()
    fu = lib.diffuser_build_uniform_graph
    fu.argtypes = [i64, i32, i32, ctypes.POINTER(i32), i32, i32, ctypes.POINTER(vp)]
    assert fu(0, 1, 0, None, 4, 0, ctypes.byref(out)) == 1          # n < 1
    assert fu(10, -1, 0, None, 4, 0, ctypes.byref(out)) == 1        # r < 0
    assert fu(10, 1, 0, None, 2000, 0, ctypes.byref(out)) == 1      # too many positions per row
    assert fu(10, 1, 0, None, 4, 0, None) == 1                      # null out
    lib.diffuser_graph_info.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    assert lib.diffuser_graph_info(None, None, None) == 1
    lib.diffuser_graph_copy_csr.argtypes = [vp, vp, vp]
    assert lib.diffuser_graph_copy_csr(None, None, None) == 1
    hws = lib.diffuser_host_workspace_size
    hws.argtypes = [vp, i64, i64, i32, i32, ctypes.POINTER(sz)]
    assert hws(None, 1, 1, 64, 1, ctypes.byref(nbytes)) == 1        # null graph
    assert hws(None, 1, 1, 64, 1, None) == 1                        # null result
    fh = lib.diffuser_forward_host
    fh.argtypes = [vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp, vp, sz, vp]
    assert fh(None, None, None, 1, 1, 1, 64, None, 5, 0.1, None, None, 0, None) == 1
    phws = lib.diffuser_per_head_workspace_size
    phws.argtypes = [vp, i64, i64, i32, i32, ctypes.POINTER(sz)]
    assert phws(None, 1, 2, 64, 1, ctypes.byref(nbytes)) == 1       # null graph list
    heads = (vp * 1)(None)
    assert phws(ctypes.cast(heads, vp), 1, 0, 64, 1, ctypes.byref(nbytes)) == 1   # H < 1
    assert phws(ctypes.cast(heads, vp), 1, 1, 64, 1, ctypes.byref(nbytes)) == 1   # a NULL head graph
    assert phws(ctypes.cast(heads, vp), 1, 1, 64, 1, None) == 1
    fph = lib.diffuser_forward_per_head
    fph.argtypes = [vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp, vp, sz, vp]
    assert fph(None, None, None, 1, 1, 1, 64, None, 5, 0.1, None, None, 0, None) == 1
    fq = lib.diffuser_qkv_projection
    fq.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, vp, vp, vp]
    assert fq(None, None, 0, 16, 768, 12, 64, None, None, None, None) == 1     # B < 1
    assert fq(None, None, 1, 16, 768, 12, 32, None, None, None, None) == 2     # d != 64
    assert fq(None, None, 1, 16, 770, 12, 64, None, None, None, None) == 2     # D not a multiple of 8
    assert fq(None, None, 1, 16, 768, 12, 64, None, None, None, None) == 1     # null tensors
    fo = lib.diffuser_output_projection
    fo.argtypes = [vp, vp, i64, i64, i32, i32, i32, vp, vp]
    assert fo(None, None, 1, 0, 768, 12, 64, None, None) == 1                  # n < 1
    assert fo(None, None, 1, 16, 768, 12, 64, None, None) == 1                 # null tensors
    lib.diffuser_projection_status.argtypes = [vp, ctypes.c_int]
    assert lib.diffuser_projection_status(None, 0) == 1
    lws = lib.diffuser_layer_workspace_size
    lws.argtypes = [vp, i64, i32, i32, i32, ctypes.POINTER(sz)]
    assert lws(None, 1, 768, 12, 64, ctypes.byref(nbytes)) == 1
    lf = lib.diffuser_layer_forward
    lf.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp, i32, f32, vp, vp, sz, vp]
    assert lf(None, None, None, 1, 768, 12, 64, None, 5, 0.1, None, None, 0, None) == 1
    na = lib.diffuser_forward_no_alloc
    na.argtypes = [vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp, vp]
    assert na(None, None, None, 1, 1, 1, 64, None, 5, 0.1, None, None) == 1
    lib.diffuser_no_alloc_scratch_bytes.restype = sz
    assert lib.diffuser_no_alloc_scratch_bytes() == 32 << 20
    aw = lib.diffuser_attention_weights
    aw.argtypes = [vp, vp, i32, i64, i64, i32, vp, vp, vp, sz, vp]
    assert aw(None, None, 1, 1, 1, 64, None, None, None, 0, None) == 1
    dc = lib.diffuser_diffuse_csr
    dc.argtypes = [vp, vp, vp, i32, i64, i64, i32, i32, f32, vp, vp, sz, vp]
    assert dc(None, None, None, 1, 1, 1, 64, 5, 0.1, None, None, 0, None) == 1
    assert lib.diffuser_set_path(7) == 1
    assert lib.diffuser_get_path() == 0                              # unchanged by the refusal
    assert lib.diffuser_set_path(1) == 0 and lib.diffuser_get_path() == 1
    assert lib.diffuser_set_path(0) == 0 and lib.diffuser_get_path() == 0
    lib.diffuser_kernels_for.argtypes = [vp, i32, vp]
    assert lib.diffuser_kernels_for(None, 1, None) == 1
    lib.diffuser_graph_status.argtypes = [vp, vp, ctypes.c_int]
    assert lib.diffuser_graph_status(None, None, 0) == 1
    lib.diffuser_graph_set_status.argtypes = [vp, ctypes.c_int]
    assert lib.diffuser_graph_set_status(None, 6) == 1


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
