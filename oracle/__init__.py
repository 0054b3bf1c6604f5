"""fp64 CPU oracle for the Diffuser hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and the
oracle imports nothing from the product package: the two share only the seeded
input buffers that a test hands to both.

The arithmetic lives in ``diffuser_oracle.c`` (plain C, double precision);
this module compiles it with gcc on first use and marshals numpy arrays.

Sources, cited by page title and section/equation:
  * "Diffuser: modelling long sequences with multi-hop attention diffusion"
    (reading notes, arXiv 2210.11794v2): sec 2.1 eq S.1-S.5 (weights A; the
    per-head projections and W_O), sec 2.4 eq S.7 (PPR recursion), sec 2.6
    (training through the unrolled recursion; causal use, A lower-triangular).
  * "1.2.1 Static sparsity: Longformer, BigBird and sliding windows":
    eq 1-6 (scores, softmax, window; the causal window), eq 11 (dilated
    window), eq 12 (globals), sec 2 eq 13 (blocks).
  * "038 BigBird": sec 2 (window u random u global; global rows read all).

Pins: every function here is checked against values the pages print, closed
forms, brute force, finite differences and invariants, in
``tests/test_oracle_pins.py``, ``tests/test_oracle_backward_pins.py`` and
``tests/test_oracle_layer_pins.py``.  The random-edge draws
themselves are a definition (SplitMix64 keyed by row and draw index), pinned
only through the published SplitMix64 test vector: parity unpinned beyond it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "diffuser_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE fp64, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared",
           "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_splitmix64.restype = ctypes.c_uint64
        lib.oracle_splitmix64.argtypes = [ctypes.c_uint64]
        lib.oracle_token_graph.restype = ctypes.c_int
        lib.oracle_token_graph.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _i32p,
                                           ctypes.c_int32, ctypes.c_uint64, _i64p, _i32p,
                                           ctypes.c_int64, _i64p]
        lib.oracle_token_graph_causal.restype = ctypes.c_int
        lib.oracle_token_graph_causal.argtypes = lib.oracle_token_graph.argtypes
        lib.oracle_token_graph_dilated.restype = ctypes.c_int
        lib.oracle_token_graph_dilated.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32, _i32p, ctypes.c_int32,
                                                   ctypes.c_uint64, ctypes.c_int32, _i64p, _i32p,
                                                   ctypes.c_int64, _i64p]
        lib.oracle_token_graph_uniform.restype = ctypes.c_int
        lib.oracle_token_graph_uniform.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                   _i32p, ctypes.c_int32, ctypes.c_int32, _i64p,
                                                   _i32p, ctypes.c_int64, _i64p]
        lib.oracle_block_graph.restype = ctypes.c_int
        lib.oracle_block_graph.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_uint64, _i64p,
                                           _i32p, ctypes.c_int64, _i64p]
        lib.oracle_attention_weights.restype = None
        lib.oracle_attention_weights.argtypes = [_f64p, _f64p, ctypes.c_int64, ctypes.c_int32,
                                                 _i64p, _i32p, _f64p]
        lib.oracle_diffuse.restype = ctypes.c_int
        lib.oracle_diffuse.argtypes = [_f64p, _i64p, _i32p, _f64p, ctypes.c_int64, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_double, _f64p]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [_f64p, _f64p, _f64p, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int32, _i64p, _i32p, ctypes.c_int32, ctypes.c_double,
                                       _f64p, ctypes.c_int32]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [_f64p, _f64p, _f64p, _f64p, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int32, _i64p, _i32p, ctypes.c_int32,
                                        ctypes.c_double, _f64p, _f64p, _f64p]
        _lib = lib
        return lib


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def splitmix64(x: int) -> int:
    """SplitMix64 output function applied to one state value."""
    return int(_load().oracle_splitmix64(ctypes.c_uint64(x & 0xFFFFFFFFFFFFFFFF)))


def _check(status: int, what: str) -> None:
    if status != 0:
        raise ValueError(f"oracle {what} failed with status {status}")


def token_graph(n: int, r: int, n_globals: int, rand_per_row: int, seed: int = 0,
                globals_idx=None, causal: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """CSR (row_ptr int64[n+1], col int32[nnz]) of window u globals u random draws.

    ``causal``: the same edge set with the mask j <= i applied to every edge
    kind (Diffuser notes sec 2.6; window of the r+1 history positions).
    """
    lib = _load()
    fn = lib.oracle_token_graph_causal if causal else lib.oracle_token_graph
    g = None
    if globals_idx is not None:
        g = np.ascontiguousarray(np.asarray(globals_idx, dtype=np.int32))
        n_globals = int(g.size)
    gp = _p(g, _i32p) if g is not None else None
    nnz = ctypes.c_int64(0)
    _check(fn(n, r, n_globals, gp, rand_per_row, seed, None, None, 0, ctypes.byref(nnz)),
           "token_graph(count)")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    col = np.zeros(max(nnz.value, 1), dtype=np.int32)
    _check(fn(n, r, n_globals, gp, rand_per_row, seed, _p(row_ptr, _i64p), _p(col, _i32p),
              col.size, ctypes.byref(nnz)), "token_graph")
    return row_ptr, col[: nnz.value]


def dilated_graph(n: int, r: int, dilation: int, n_globals: int, rand_per_row: int, seed: int = 0,
                  globals_idx=None, causal: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """CSR of the token graph whose window is {i + k dilation : |k| <= r} (sliding-window
    page, sec 1.2 eq 11)."""
    lib = _load()
    g = None
    if globals_idx is not None:
        g = np.ascontiguousarray(np.asarray(globals_idx, dtype=np.int32))
        n_globals = int(g.size)
    gp = _p(g, _i32p) if g is not None else None
    nnz = ctypes.c_int64(0)
    _check(lib.oracle_token_graph_dilated(n, r, dilation, n_globals, gp, rand_per_row, seed,
                                          int(causal), None, None, 0, ctypes.byref(nnz)),
           "dilated_graph(count)")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    col = np.zeros(max(nnz.value, 1), dtype=np.int32)
    _check(lib.oracle_token_graph_dilated(n, r, dilation, n_globals, gp, rand_per_row, seed,
                                          int(causal), _p(row_ptr, _i64p), _p(col, _i32p),
                                          col.size, ctypes.byref(nnz)), "dilated_graph")
    return row_ptr, col[: nnz.value]


def uniform_graph(n: int, r: int, n_globals: int, rand_per_row: int, globals_idx=None,
                  causal: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """CSR of the token graph whose R extras of row i sit on the uniform grid
    j_t = (i + floor((2t + 1) n / (2R))) mod n ("w uni.", Diffuser notes sec 4.5,
    Tab S.7), with the causal mask when ``causal``."""
    lib = _load()
    g = None
    if globals_idx is not None:
        g = np.ascontiguousarray(np.asarray(globals_idx, dtype=np.int32))
        n_globals = int(g.size)
    gp = _p(g, _i32p) if g is not None else None
    nnz = ctypes.c_int64(0)
    _check(lib.oracle_token_graph_uniform(n, r, n_globals, gp, rand_per_row, int(causal), None,
                                          None, 0, ctypes.byref(nnz)), "uniform_graph(count)")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    col = np.zeros(max(nnz.value, 1), dtype=np.int32)
    _check(lib.oracle_token_graph_uniform(n, r, n_globals, gp, rand_per_row, int(causal),
                                          _p(row_ptr, _i64p), _p(col, _i32p), col.size,
                                          ctypes.byref(nnz)), "uniform_graph")
    return row_ptr, col[: nnz.value]


def forward_per_head(Q: np.ndarray, K: np.ndarray, V: np.ndarray, graphs, hops: int,
                     alpha: float, nthreads: int = 1) -> np.ndarray:
    """The forward with one graph per head (Diffuser notes sec 2.2: the random
    sets may differ per layer and per head): head h of every batch item runs on
    graphs[h] = (row_ptr, col).  Q, K, V float64 [B][H][n][d]."""
    Q, K, V = (np.asarray(x, dtype=np.float64) for x in (Q, K, V))
    out = np.zeros_like(V)
    for h, (row_ptr, col) in enumerate(graphs):
        out[:, h] = forward(Q[:, h], K[:, h], V[:, h], row_ptr, col, hops, alpha, nthreads=nthreads)
    return out


def block_graph(n: int, block: int, window_blocks: int, rand_blocks: int, global_blocks: int,
                seed: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """CSR of the BigBird ITC block pattern, expanded to tokens."""
    lib = _load()
    nnz = ctypes.c_int64(0)
    _check(lib.oracle_block_graph(n, block, window_blocks, rand_blocks, global_blocks, seed,
                                  None, None, 0, ctypes.byref(nnz)), "block_graph(count)")
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    col = np.zeros(max(nnz.value, 1), dtype=np.int32)
    _check(lib.oracle_block_graph(n, block, window_blocks, rand_blocks, global_blocks, seed,
                                  _p(row_ptr, _i64p), _p(col, _i32p), col.size,
                                  ctypes.byref(nnz)), "block_graph")
    return row_ptr, col[: nnz.value]


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of an input buffer to float64.

    ``dtype`` "fp32": x is float32.  "bf16": x holds bfloat16 bit patterns as
    uint16 (a bfloat16 is the top half of a float32).
    """
    if dtype == "fp32":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        bits = np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def attention_weights(Q: np.ndarray, K: np.ndarray, row_ptr: np.ndarray,
                      col: np.ndarray) -> np.ndarray:
    """Row-softmax weights A (one per CSR edge) for one unit; Q, K float64 [n][d]."""
    Q = np.ascontiguousarray(Q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    n, d = Q.shape
    A = np.zeros(max(int(row_ptr[-1]), 1), dtype=np.float64)
    _load().oracle_attention_weights(_p(Q, _f64p), _p(K, _f64p), n, d,
                                     _p(np.ascontiguousarray(row_ptr, dtype=np.int64), _i64p),
                                     _p(np.ascontiguousarray(col, dtype=np.int32), _i32p),
                                     _p(A, _f64p))
    return A[: int(row_ptr[-1])]


def diffuse(A: np.ndarray, row_ptr: np.ndarray, col: np.ndarray, V: np.ndarray, hops: int,
            alpha: float) -> np.ndarray:
    """Z_hops of the PPR recursion for one unit; V float64 [n][dv]."""
    V = np.ascontiguousarray(V, dtype=np.float64)
    n, dv = V.shape
    A = np.ascontiguousarray(A, dtype=np.float64)
    if A.size == 0:
        A = np.zeros(1, dtype=np.float64)
    Z = np.zeros_like(V)
    _check(_load().oracle_diffuse(_p(A, _f64p),
                                  _p(np.ascontiguousarray(row_ptr, dtype=np.int64), _i64p),
                                  _p(np.ascontiguousarray(col, dtype=np.int32), _i32p),
                                  _p(V, _f64p), n, dv, hops, alpha, _p(Z, _f64p)), "diffuse")
    return Z


def forward(Q: np.ndarray, K: np.ndarray, V: np.ndarray, row_ptr: np.ndarray, col: np.ndarray,
            hops: int, alpha: float, nthreads: int = 1) -> np.ndarray:
    """Whole forward over [units][n][d] float64 inputs; returns Z_hops float64."""
    Q = np.ascontiguousarray(Q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    units = int(np.prod(Q.shape[:-2])) if Q.ndim > 2 else 1
    n, d = Q.shape[-2], Q.shape[-1]
    out = np.zeros_like(V)
    _check(_load().oracle_forward(_p(Q, _f64p), _p(K, _f64p), _p(V, _f64p), units, n, d,
                                  _p(np.ascontiguousarray(row_ptr, dtype=np.int64), _i64p),
                                  _p(np.ascontiguousarray(col, dtype=np.int32), _i32p),
                                  hops, alpha, _p(out, _f64p), max(1, int(nthreads))), "forward")
    return out


def backward(Q: np.ndarray, K: np.ndarray, V: np.ndarray, dOut: np.ndarray, row_ptr: np.ndarray,
             col: np.ndarray, hops: int, alpha: float):
    """Gradients (dQ, dK, dV) of <dOut, Z_hops> over [units][n][d] float64 inputs (or [n][d])."""
    Q, K, V, dOut = (np.ascontiguousarray(x, dtype=np.float64) for x in (Q, K, V, dOut))
    units = int(np.prod(Q.shape[:-2])) if Q.ndim > 2 else 1
    n, d = Q.shape[-2], Q.shape[-1]
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    _check(_load().oracle_backward(_p(Q, _f64p), _p(K, _f64p), _p(V, _f64p), _p(dOut, _f64p),
                                   units, n, d,
                                   _p(np.ascontiguousarray(row_ptr, dtype=np.int64), _i64p),
                                   _p(np.ascontiguousarray(col, dtype=np.int32), _i32p),
                                   hops, alpha, _p(dQ, _f64p), _p(dK, _f64p), _p(dV, _f64p)),
           "backward")
    return dQ, dK, dV


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bfloat16 value (8 significant bits), ties to even,
    returned as float64: x = m 2^e with 0.5 <= |m| < 1, m rounded to a multiple
    of 2^-8 (normal range; no overflow handling)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def layer_forward(X: np.ndarray, Wq: np.ndarray, Wk: np.ndarray, Wv: np.ndarray, Wo: np.ndarray,
                  row_ptr: np.ndarray, col: np.ndarray, hops: int, alpha: float,
                  bf16_interfaces: bool = False) -> np.ndarray:
    """The diffusion module with its projections (Diffuser notes sec 2.1: per head
    Q = X W_Q, K = X W_K, V = X W_V; the heads' outputs are concatenated and
    projected by W_O; sec 2.4: residual and feed-forward lie outside the module).

    X [B][n][D]; Wq, Wk, Wv [H][D][d]; Wo [H*d][D]; all float64.  Returns [B][n][D].
    ``bf16_interfaces``: the tensors passed between the stages (Q, K, V, the heads'
    outputs Z and the result) are bf16, each rounded once to nearest-even from the
    exact value of its stage; the arithmetic inside every stage stays float64.
    """
    r = round_bf16 if bf16_interfaces else (lambda t: t)
    X = np.asarray(X, dtype=np.float64)
    B, n, _ = X.shape
    H, _, d = Wq.shape
    Q = r(np.einsum("bnD,hDd->bhnd", X, Wq))
    K = r(np.einsum("bnD,hDd->bhnd", X, Wk))
    V = r(np.einsum("bnD,hDd->bhnd", X, Wv))
    Z = r(forward(Q, K, V, row_ptr, col, hops, alpha))              # [B][H][n][d]
    heads = np.transpose(Z, (0, 2, 1, 3)).reshape(B, n, H * d)      # concatenation
    return r(heads @ Wo)
