"""Thin ctypes binding of libdiffuser.so (include/diffuser.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Functions keep the C names.  Device tensors are torch tensors
(PyTorch provides device memory and streams); the graph is an opaque handle
freed when its Python object dies.

If the library is missing or cannot be loaded this module raises on import:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdiffuser.so")

DIFFUSER_OK = 0
DIFFUSER_DTYPE_FP32 = 0
DIFFUSER_DTYPE_BF16 = 1
DIFFUSER_PATH_AUTO = 0
DIFFUSER_PATH_CSR = 1
KERNEL_KINDS = ("build", "score", "hop", "aux", "gather")


class DiffuserError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status} ({message})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libdiffuser.so is not built ({LIB_PATH}); run "
                          "`python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(LIB_PATH)
    c = ctypes
    vp, i32, i64, u64, f32 = c.c_void_p, c.c_int32, c.c_int64, c.c_uint64, c.c_float
    i64p, i32p = c.POINTER(c.c_int64), c.POINTER(c.c_int32)
    sig = {
        "diffuser_status_string": (c.c_char_p, [c.c_int]),
        "diffuser_last_error": (c.c_char_p, []),
        "diffuser_version": (c.c_int, []),
        "diffuser_build_graph": (c.c_int, [i64, i32, i32, i32p, i32, u64, c.POINTER(vp)]),
        "diffuser_build_causal_graph": (c.c_int, [i64, i32, i32, i32p, i32, u64, c.POINTER(vp)]),
        "diffuser_build_dilated_graph": (c.c_int, [i64, i32, i32, i32, i32p, i32, u64, i32,
                                                   c.POINTER(vp)]),
        "diffuser_build_block_graph": (c.c_int, [i64, i32, i32, i32, i32, u64, c.POINTER(vp)]),
        "diffuser_graph_info": (c.c_int, [vp, i64p, i64p]),
        "diffuser_graph_copy_csr": (c.c_int, [vp, i64p, i32p]),
        "diffuser_graph_free": (None, [vp]),
        "diffuser_workspace_size": (c.c_int, [vp, i64, i64, i32, i32, c.POINTER(c.c_size_t)]),
        "diffuser_forward": (c.c_int, [vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp, vp,
                                       c.c_size_t, vp]),
        "diffuser_host_workspace_size": (c.c_int, [vp, i64, i64, i32, i32,
                                                   c.POINTER(c.c_size_t)]),
        "diffuser_forward_host": (c.c_int, [vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp,
                                            vp, c.c_size_t, vp]),
        "diffuser_backward_workspace_size": (c.c_int, [vp, i64, i64, i32, i32, i32,
                                                       c.POINTER(c.c_size_t)]),
        "diffuser_backward": (c.c_int, [vp, vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp, vp,
                                        vp, vp, c.c_size_t, vp]),
        "diffuser_attention_weights": (c.c_int, [vp, vp, i32, i64, i64, i32, vp, vp, vp,
                                                 c.c_size_t, vp]),
        "diffuser_diffuse_csr": (c.c_int, [vp, vp, vp, i32, i64, i64, i32, i32, f32, vp, vp,
                                           c.c_size_t, vp]),
        "diffuser_forward_no_alloc": (c.c_int, [vp, vp, vp, i32, i64, i64, i32, vp, i32, f32, vp,
                                                vp]),
        "diffuser_no_alloc_scratch_bytes": (c.c_size_t, []),
        "diffuser_set_path": (c.c_int, [c.c_int]),
        "diffuser_get_path": (c.c_int, []),
        "diffuser_build_uniform_graph": (c.c_int, [i64, i32, i32, c.POINTER(c.c_int32), i32, i32,
                                                   c.POINTER(vp)]),
        "diffuser_per_head_workspace_size": (c.c_int, [c.POINTER(vp), i64, i64, i32, i32,
                                                       c.POINTER(c.c_size_t)]),
        "diffuser_forward_per_head": (c.c_int, [vp, vp, vp, i32, i64, i64, i32, c.POINTER(vp), i32,
                                                c.c_float, vp, vp, c.c_size_t, vp]),
        "diffuser_kernels_for": (c.c_int, [vp, i32, c.POINTER(c.c_int)]),
        "diffuser_qkv_projection": (c.c_int, [vp, vp, i64, i64, i32, i32, i32, vp, vp, vp, vp]),
        "diffuser_output_projection": (c.c_int, [vp, vp, i64, i64, i32, i32, i32, vp, vp]),
        "diffuser_projection_status": (c.c_int, [c.POINTER(c.c_int), c.c_int]),
        "diffuser_layer_workspace_size": (c.c_int, [vp, i64, i32, i32, i32, c.POINTER(c.c_size_t)]),
        "diffuser_layer_forward": (c.c_int, [vp, vp, vp, i64, i32, i32, i32, vp, i32, c.c_float, vp,
                                             vp, c.c_size_t, vp]),
        "diffuser_graph_status": (c.c_int, [vp, c.POINTER(c.c_int), c.c_int]),
        "diffuser_graph_set_status": (c.c_int, [vp, c.c_int]),
        "diffuser_launch_count": (c.c_int64, [i64p]),
        "diffuser_profile_begin": (c.c_int, []),
        "diffuser_profile_end": (c.c_int, [c.POINTER(c.c_double), i64p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status: int, where: str) -> None:
    if status != DIFFUSER_OK:
        msg = _lib.diffuser_last_error().decode() or _lib.diffuser_status_string(status).decode()
        raise DiffuserError(status, where, msg)


def diffuser_status_string(status: int) -> str:
    return _lib.diffuser_status_string(status).decode()


def diffuser_version() -> int:
    return int(_lib.diffuser_version())


class Graph:
    """Owning handle of a diffuser_graph."""

    def __init__(self, handle: int):
        self.handle = ctypes.c_void_p(handle)
        n, nnz = ctypes.c_int64(), ctypes.c_int64()
        _check(_lib.diffuser_graph_info(self.handle, ctypes.byref(n), ctypes.byref(nnz)),
               "diffuser_graph_info")
        self.n, self.nnz = n.value, nnz.value

    def free(self) -> None:
        if self.handle:
            _lib.diffuser_graph_free(self.handle)
            self.handle = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def _build_token(fn, name, n, r, n_globals, global_idx, rand_per_row, seed) -> Graph:
    gp = None
    if global_idx is not None:
        g = np.ascontiguousarray(np.asarray(global_idx, dtype=np.int32))
        n_globals = int(g.size)
        gp = g.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    out = ctypes.c_void_p()
    _check(fn(n, r, n_globals, gp, rand_per_row, seed & 0xFFFFFFFFFFFFFFFF, ctypes.byref(out)),
           name)
    return Graph(out.value)


def diffuser_build_graph(n: int, r: int, n_globals: int, global_idx=None, rand_per_row: int = 0,
                         seed: int = 0) -> Graph:
    return _build_token(_lib.diffuser_build_graph, "diffuser_build_graph", n, r, n_globals,
                        global_idx, rand_per_row, seed)


def diffuser_build_causal_graph(n: int, r: int, n_globals: int, global_idx=None,
                                rand_per_row: int = 0, seed: int = 0) -> Graph:
    return _build_token(_lib.diffuser_build_causal_graph, "diffuser_build_causal_graph", n, r,
                        n_globals, global_idx, rand_per_row, seed)


def diffuser_build_dilated_graph(n: int, r: int, dilation: int, n_globals: int, global_idx=None,
                                 rand_per_row: int = 0, seed: int = 0, causal: bool = False) -> Graph:
    gp = None
    if global_idx is not None:
        gl = np.ascontiguousarray(np.asarray(global_idx, dtype=np.int32))
        n_globals = int(gl.size)
        gp = gl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    out = ctypes.c_void_p()
    _check(_lib.diffuser_build_dilated_graph(n, r, dilation, n_globals, gp, rand_per_row,
                                             seed & 0xFFFFFFFFFFFFFFFF, int(causal),
                                             ctypes.byref(out)), "diffuser_build_dilated_graph")
    return Graph(out.value)


def diffuser_build_uniform_graph(n: int, r: int, n_globals: int, global_idx=None,
                                 positions_per_row: int = 0, causal: bool = False) -> Graph:
    """Token graph whose extras sit on a uniform grid ("w uni."), no seed."""
    gp = None
    if global_idx is not None:
        gl = np.ascontiguousarray(np.asarray(global_idx, dtype=np.int32))
        n_globals = int(gl.size)
        gp = gl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    out = ctypes.c_void_p()
    _check(_lib.diffuser_build_uniform_graph(n, r, n_globals, gp, positions_per_row, int(causal),
                                             ctypes.byref(out)), "diffuser_build_uniform_graph")
    return Graph(out.value)


def diffuser_build_block_graph(n: int, block: int, window_blocks: int, rand_blocks: int,
                               global_blocks: int, seed: int = 0) -> Graph:
    out = ctypes.c_void_p()
    _check(_lib.diffuser_build_block_graph(n, block, window_blocks, rand_blocks, global_blocks,
                                           seed & 0xFFFFFFFFFFFFFFFF, ctypes.byref(out)),
           "diffuser_build_block_graph")
    return Graph(out.value)


def diffuser_graph_info(g: Graph) -> tuple[int, int]:
    return g.n, g.nnz


def diffuser_graph_copy_csr(g: Graph) -> tuple[np.ndarray, np.ndarray]:
    row_ptr = np.zeros(g.n + 1, dtype=np.int64)
    col = np.zeros(max(g.nnz, 1), dtype=np.int32)
    _check(_lib.diffuser_graph_copy_csr(g.handle,
                                        row_ptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                        col.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
           "diffuser_graph_copy_csr")
    return row_ptr, col[: g.nnz]


def diffuser_graph_free(g: Graph) -> None:
    g.free()


# ---------------------------------------------------------------- torch marshalling
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DIFFUSER_DTYPE_FP32
    if t.dtype == torch.bfloat16:
        return DIFFUSER_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; use float32 or bfloat16")


def _shape(t, g: Graph):
    if t.dim() != 4 or t.shape[2] != g.n:
        raise ValueError(f"expected [B][H][{g.n}][d], got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return int(t.shape[0]), int(t.shape[1]), int(t.shape[3])


def _stream(stream) -> ctypes.c_void_p:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def diffuser_workspace_size(g: Graph, B: int, H: int, d: int, dtype: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.diffuser_workspace_size(g.handle, B, H, d, dtype, ctypes.byref(b)),
           "diffuser_workspace_size")
    return b.value


def diffuser_host_workspace_size(g: Graph, B: int, H: int, d: int, dtype: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.diffuser_host_workspace_size(g.handle, B, H, d, dtype, ctypes.byref(b)),
           "diffuser_host_workspace_size")
    return b.value


def alloc_workspace(nbytes: int, device=None):
    """A 256-byte aligned device buffer (torch caching allocator) of nbytes."""
    import torch
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=device or "cuda")


def diffuser_forward(Q, K, V, g: Graph, hops: int, alpha: float, out=None, workspace=None,
                     stream=None):
    import torch
    B, H, d = _shape(Q, g)
    code = _dtype_code(Q)
    if out is None:
        out = torch.empty_like(V)
    if workspace is None:
        workspace = alloc_workspace(diffuser_workspace_size(g, B, H, d, code), Q.device)
    _check(_lib.diffuser_forward(Q.data_ptr(), K.data_ptr(), V.data_ptr(), code, B, H, d,
                                 g.handle, hops, alpha, out.data_ptr(), workspace.data_ptr(),
                                 workspace.numel(), _stream(stream)), "diffuser_forward")
    return out


def _graph_array(graphs):
    return (ctypes.c_void_p * len(graphs))(*[g.handle.value for g in graphs])


def diffuser_per_head_workspace_size(graphs, B: int, H: int, d: int, dtype: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.diffuser_per_head_workspace_size(_graph_array(graphs), B, H, d, dtype,
                                                 ctypes.byref(b)), "diffuser_per_head_workspace_size")
    return b.value


def diffuser_forward_per_head(Q, K, V, graphs, hops: int, alpha: float, out=None, workspace=None,
                              stream=None):
    """The forward with graphs[h] for head h (device tensors [B][H][n][d])."""
    import torch
    B, H, n, d = Q.shape
    if len(graphs) != H:
        raise ValueError("one graph per head is needed")
    code = _dtype_code(Q)
    if out is None:
        out = torch.empty_like(V)
    if workspace is None:
        workspace = alloc_workspace(diffuser_per_head_workspace_size(graphs, B, H, d, code), Q.device)
    _check(_lib.diffuser_forward_per_head(Q.data_ptr(), K.data_ptr(), V.data_ptr(), code, B, H, d,
                                          _graph_array(graphs), hops, alpha, out.data_ptr(),
                                          workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "diffuser_forward_per_head")
    return out


def diffuser_qkv_projection(X, Wqkv, H: int, Q=None, K=None, V=None, stream=None):
    """Per-head Q, K, V [B][H][n][64] of X [B][n][D] by Wqkv [3 H 64][D] (bf16 tensors)."""
    import torch
    B, n, D = X.shape
    shape = (B, H, n, 64)
    Q = torch.empty(shape, dtype=torch.bfloat16, device=X.device) if Q is None else Q
    K = torch.empty(shape, dtype=torch.bfloat16, device=X.device) if K is None else K
    V = torch.empty(shape, dtype=torch.bfloat16, device=X.device) if V is None else V
    _check(_lib.diffuser_qkv_projection(X.data_ptr(), Wqkv.data_ptr(), B, n, D, H, 64, Q.data_ptr(),
                                        K.data_ptr(), V.data_ptr(), _stream(stream)),
           "diffuser_qkv_projection")
    return Q, K, V


def diffuser_output_projection(Z, Wo, Y=None, stream=None):
    """Y [B][n][D] = the heads of Z [B][H][n][64] concatenated, times Wo^T (Wo [D][H 64])."""
    import torch
    B, H, n, d = Z.shape
    D = Wo.shape[0]
    Y = torch.empty((B, n, D), dtype=torch.bfloat16, device=Z.device) if Y is None else Y
    _check(_lib.diffuser_output_projection(Z.data_ptr(), Wo.data_ptr(), B, n, D, H, d, Y.data_ptr(),
                                           _stream(stream)), "diffuser_output_projection")
    return Y


def diffuser_projection_status(reset: bool = False) -> int:
    st = ctypes.c_int()
    _check(_lib.diffuser_projection_status(ctypes.byref(st), int(reset)), "diffuser_projection_status")
    return st.value


def diffuser_layer_workspace_size(g: Graph, B: int, D: int, H: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.diffuser_layer_workspace_size(g.handle, B, D, H, 64, ctypes.byref(b)),
           "diffuser_layer_workspace_size")
    return b.value


def diffuser_layer_forward(X, Wqkv, Wo, g: Graph, H: int, hops: int, alpha: float, Y=None,
                           workspace=None, stream=None):
    """The module: projections, the forward on graph g, concatenation and W_O (bf16)."""
    import torch
    B, n, D = X.shape
    Y = torch.empty_like(X) if Y is None else Y
    if workspace is None:
        workspace = alloc_workspace(diffuser_layer_workspace_size(g, B, D, H), X.device)
    _check(_lib.diffuser_layer_forward(X.data_ptr(), Wqkv.data_ptr(), Wo.data_ptr(), B, D, H, 64,
                                       g.handle, hops, alpha, Y.data_ptr(), workspace.data_ptr(),
                                       workspace.numel(), _stream(stream)), "diffuser_layer_forward")
    return Y


def diffuser_backward_workspace_size(g: Graph, B: int, H: int, d: int, dtype: int,
                                     hops: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.diffuser_backward_workspace_size(g.handle, B, H, d, dtype, hops, ctypes.byref(b)),
           "diffuser_backward_workspace_size")
    return b.value


def diffuser_backward(Q, K, V, dOut, g: Graph, hops: int, alpha: float, dQ=None, dK=None, dV=None,
                      workspace=None, stream=None):
    """Gradients (dQ, dK, dV) of <dOut, forward(Q, K, V)>; device tensors in one dtype."""
    import torch
    B, H, d = _shape(Q, g)
    code = _dtype_code(Q)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    if workspace is None:
        workspace = alloc_workspace(diffuser_backward_workspace_size(g, B, H, d, code, hops),
                                    Q.device)
    _check(_lib.diffuser_backward(Q.data_ptr(), K.data_ptr(), V.data_ptr(), dOut.data_ptr(), code,
                                  B, H, d, g.handle, hops, alpha, dQ.data_ptr(), dK.data_ptr(),
                                  dV.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                  _stream(stream)), "diffuser_backward")
    return dQ, dK, dV


def diffuser_forward_host(Q, K, V, g: Graph, hops: int, alpha: float, out, workspace,
                          stream=None):
    """Q, K, V, out: host (ideally pinned) torch tensors; enqueues copies + forward."""
    B, H, d = _shape(Q, g)
    code = _dtype_code(Q)
    _check(_lib.diffuser_forward_host(Q.data_ptr(), K.data_ptr(), V.data_ptr(), code, B, H, d,
                                      g.handle, hops, alpha, out.data_ptr(),
                                      workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "diffuser_forward_host")
    return out


def diffuser_forward_no_alloc(Q, K, V, g: Graph, hops: int, alpha: float, out, stream=None):
    """The forward with the library's fixed device scratch array (no workspace)."""
    B, H, d = _shape(Q, g)
    code = _dtype_code(Q)
    _check(_lib.diffuser_forward_no_alloc(Q.data_ptr(), K.data_ptr(), V.data_ptr(), code, B, H, d,
                                          g.handle, hops, alpha, out.data_ptr(), _stream(stream)),
           "diffuser_forward_no_alloc")
    return out


def diffuser_no_alloc_scratch_bytes() -> int:
    return int(_lib.diffuser_no_alloc_scratch_bytes())


def diffuser_attention_weights(Q, K, g: Graph, A_out=None, workspace=None, stream=None):
    import torch
    B, H, d = _shape(Q, g)
    code = _dtype_code(Q)
    if A_out is None:
        A_out = torch.empty((B * H, g.nnz), dtype=torch.float32, device=Q.device)
    if workspace is None:
        workspace = alloc_workspace(diffuser_workspace_size(g, B, H, d, code), Q.device)
    _check(_lib.diffuser_attention_weights(Q.data_ptr(), K.data_ptr(), code, B, H, d, g.handle,
                                           A_out.data_ptr(), workspace.data_ptr(),
                                           workspace.numel(), _stream(stream)),
           "diffuser_attention_weights")
    return A_out


def diffuser_diffuse_csr(g: Graph, A, V, hops: int, alpha: float, out=None, workspace=None,
                         stream=None):
    import torch
    B, H, d = _shape(V, g)
    code = _dtype_code(V)
    if A.dtype != torch.float32 or not A.is_contiguous() or A.numel() != B * H * g.nnz:
        raise ValueError("A must be contiguous float32 with B*H*nnz entries")
    if out is None:
        out = torch.empty_like(V)
    if workspace is None:
        workspace = alloc_workspace(diffuser_workspace_size(g, B, H, d, code), V.device)
    _check(_lib.diffuser_diffuse_csr(g.handle, A.data_ptr(), V.data_ptr(), code, B, H, d, hops,
                                     alpha, out.data_ptr(), workspace.data_ptr(),
                                     workspace.numel(), _stream(stream)), "diffuser_diffuse_csr")
    return out


def diffuser_set_path(path: int) -> None:
    _check(_lib.diffuser_set_path(path), "diffuser_set_path")


def diffuser_get_path() -> int:
    return int(_lib.diffuser_get_path())


DIFFUSER_KERNELS_CSR, DIFFUSER_KERNELS_BAND, DIFFUSER_KERNELS_BLOCK = 1, 2, 3


def diffuser_kernels_for(g: Graph, dtype: int) -> int:
    """The kernel family a forward on g with this dtype runs (DIFFUSER_KERNELS_*)."""
    k = ctypes.c_int()
    _check(_lib.diffuser_kernels_for(g.handle, dtype, ctypes.byref(k)), "diffuser_kernels_for")
    return k.value


def diffuser_graph_status(g: Graph, reset: bool = False) -> int:
    st = ctypes.c_int()
    _check(_lib.diffuser_graph_status(g.handle, ctypes.byref(st), int(reset)),
           "diffuser_graph_status")
    return st.value


def diffuser_graph_set_status(g: Graph, status: int) -> None:
    _check(_lib.diffuser_graph_set_status(g.handle, int(status)), "diffuser_graph_set_status")


def diffuser_launch_count() -> tuple[int, dict]:
    arr = (ctypes.c_int64 * len(KERNEL_KINDS))()
    total = int(_lib.diffuser_launch_count(arr))
    return total, dict(zip(KERNEL_KINDS, list(arr)))


def diffuser_profile_begin() -> None:
    _check(_lib.diffuser_profile_begin(), "diffuser_profile_begin")


def diffuser_profile_end() -> dict:
    ms = (ctypes.c_double * len(KERNEL_KINDS))()
    cnt = (ctypes.c_int64 * len(KERNEL_KINDS))()
    _check(_lib.diffuser_profile_end(ms, cnt), "diffuser_profile_end")
    return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNEL_KINDS)}


def raw_library() -> ctypes.CDLL:
    """The loaded ctypes library (for tests that call the C ABI directly)."""
    return _lib
