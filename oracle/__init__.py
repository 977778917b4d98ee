"""CPU oracle for CSR sparse aggregation: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never calls it
and shares no code with it; it is the independent, slow, obviously correct
statement of what the CUDA path must compute.

The arithmetic lives in ``oracle.c`` (plain C loops, double accumulation);
this module compiles it with gcc on first use and marshals numpy arrays.
Each function names the passage it follows:

* AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN Aggregation
  (SpMM/SDDMM) and CSR Attention", Abstract: CSR SpMM, SDDMM and the CSR
  attention pipeline SDDMM -> row-softmax -> SpMM.
* Benchmark page "fused sparse attention-value aggregation", problem
  statement and kernel: rows are destinations, ``col_idx`` holds sources,
  the row softmax subtracts the row maximum, empty rows give zero output.

Parity status of each function (what pins it) is listed in the tests
(``tests/test_oracle_pins.py``); the plan fingerprint and row statistics
are definitions of this library's own (no passage), pinned by brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP across rows)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_spmm.argtypes = [_i64, _ptr, _ptr, _ptr, _i64, _i64, _ptr, _i64, _ptr, _i64, _ptr]
    lib.oracle_sddmm.argtypes = [_i64, _ptr, _ptr, _i64, _i64, _ptr, _i64, _ptr, _i64,
                                 ctypes.c_double, _ptr, _i64, _ptr, _ptr]
    lib.oracle_row_softmax.argtypes = [_i64, _ptr, _i64, _ptr, _ptr]
    lib.oracle_csr_attention.argtypes = [_i64, _ptr, _ptr, _i64, _i64, _ptr, _i64, _ptr, _i64,
                                         _ptr, _i64, ctypes.c_double, _ptr, _i64, _ptr]
    lib.oracle_transpose.argtypes = [_i64, _i64, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]
    lib.oracle_spmm_t_scatter.argtypes = [_i64, _i64, _ptr, _ptr, _ptr, _ptr, _i64, _i64, _ptr]
    lib.oracle_row_stats.argtypes = [_i64, _ptr, _i64, _ptr, _ptr]
    lib.oracle_csr_attention_backward.argtypes = [_i64, _i64, _ptr, _ptr, _i64, _i64, _ptr, _ptr, _ptr, _ptr,
                                                  ctypes.c_double, _ptr, _ptr, _ptr]
    lib.oracle_csr_attention_backward.restype = None
    lib.oracle_spmm_typed.argtypes = [_i64, _i64, _ptr, _ptr, _ptr, _ptr, _ptr, _i64, _i64, _ptr]
    lib.oracle_spmm_typed.restype = None
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads.restype = None
    lib.oracle_fingerprint.argtypes = [_i64, _ptr, _ptr]
    lib.oracle_fingerprint.restype = ctypes.c_uint64
    for name in ("oracle_spmm", "oracle_sddmm", "oracle_row_softmax", "oracle_csr_attention",
                 "oracle_transpose", "oracle_spmm_t_scatter", "oracle_row_stats"):
        getattr(lib, name).restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


class use_library:
    """Context manager: route every oracle call to another build of oracle.c
    (the pin tests use it to check that planted mistakes are caught)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _rows(rows, n_rows):
    if rows is None:
        return None, n_rows
    r = np.ascontiguousarray(rows, dtype=np.int64)
    if r.size and (r.min() < 0 or r.max() >= n_rows):
        raise IndexError("row out of range")
    return r, int(r.size)


def _matrix(X):
    X = np.asarray(X, dtype=np.float32)
    if X.ndim != 2 or X.strides[1] != 4 or X.strides[0] % 4:
        X = np.ascontiguousarray(X)
    return X, X.strides[0] // 4


def spmm(row_ptr, col_idx, vals, X, rows=None, heads: int = 1):
    """Y = A X in double (Abstract: CSR SpMM).

    ``vals`` is [nnz] (or [nnz, heads] with ``heads > 1``) or None for all
    ones; X is [n_cols, heads * D]. Returns [len(rows) or n_rows, F] float64.
    """
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    n_rows = row_ptr.shape[0] - 1
    X, ldx = _matrix(X)
    F = X.shape[1]
    if F % heads:
        raise ValueError("F must be a multiple of heads")
    v = None if vals is None else _f32(vals).reshape(-1)
    r, n_out = _rows(rows, n_rows)
    Y = np.zeros((n_out, F), dtype=np.float64)
    lib.oracle_spmm(n_rows, _p(row_ptr), _p(col_idx), _p(v), heads, F // heads, _p(X), ldx,
                    _p(r), n_out, _p(Y))
    return Y


def sddmm(row_ptr, col_idx, Q, K, alpha: float = 1.0, heads: int = 1, rows=None):
    """S[p, h] = alpha * <Q[row(p), h, :], K[col_idx[p], h, :]> in double (Abstract: SDDMM).

    Returns [nnz, heads] (or the edges of ``rows``, concatenated in order).
    """
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    n_rows = row_ptr.shape[0] - 1
    Q, ldq = _matrix(Q)
    K, ldk = _matrix(K)
    F = Q.shape[1]
    if K.shape[1] != F or F % heads:
        raise ValueError("bad feature shapes")
    r, n_out = _rows(rows, n_rows)
    if r is None:
        off = None
        n_e = int(row_ptr[-1])
    else:
        deg = (row_ptr[r + 1].astype(np.int64) - row_ptr[r])
        off = np.zeros(n_out + 1, dtype=np.int64)
        np.cumsum(deg, out=off[1:])
        n_e = int(off[-1])
    S = np.zeros((n_e, heads), dtype=np.float64)
    lib.oracle_sddmm(n_rows, _p(row_ptr), _p(col_idx), heads, F // heads, _p(Q), ldq, _p(K), ldk,
                     float(alpha), _p(r), n_out, _p(off), _p(S))
    return S


def row_softmax(row_ptr, S):
    """Per-row (per-head) max-subtracted softmax of edge scores, in double."""
    lib = _load()
    row_ptr = _i32(row_ptr)
    S = np.ascontiguousarray(S, dtype=np.float64)
    S2 = S.reshape(S.shape[0], -1)
    W = np.zeros_like(S2)
    lib.oracle_row_softmax(row_ptr.shape[0] - 1, _p(row_ptr), S2.shape[1], _p(S2), _p(W))
    return W.reshape(S.shape)


def csr_attention(row_ptr, col_idx, Q, K, V, heads: int, scale: float, rows=None):
    """O = softmax_row(scale * Q K^T on the pattern) V per head, all in double."""
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    n_rows = row_ptr.shape[0] - 1
    Q, ldq = _matrix(Q)
    K, ldk = _matrix(K)
    V, ldv = _matrix(V)
    F = Q.shape[1]
    if K.shape[1] != F or V.shape[1] != F or F % heads:
        raise ValueError("bad feature shapes")
    r, n_out = _rows(rows, n_rows)
    O = np.zeros((n_out, F), dtype=np.float64)
    lib.oracle_csr_attention(n_rows, _p(row_ptr), _p(col_idx), heads, F // heads, _p(Q), ldq,
                             _p(K), ldk, _p(V), ldv, float(scale), _p(r), n_out, _p(O))
    return O


def csr_attention_backward(row_ptr, col_idx, Q, K, V, dO, heads: int, scale: float):
    """Gradients (dQ, dK, dV) of CSR attention for an upstream gradient dO, in
    double: the chain rule through the weighted sum and the row softmax."""
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    Q, K, V, dO = (np.ascontiguousarray(a, dtype=np.float32) for a in (Q, K, V, dO))
    n_rows, n_cols, F = Q.shape[0], K.shape[0], Q.shape[1]
    if F % heads or K.shape[1] != F or V.shape != K.shape or dO.shape != Q.shape:
        raise ValueError("bad shapes")
    dQ = np.zeros((n_rows, F))
    dK = np.zeros((n_cols, F))
    dV = np.zeros((n_cols, F))
    lib.oracle_csr_attention_backward(n_rows, n_cols, _p(row_ptr), _p(col_idx), heads, F // heads, _p(Q), _p(K),
                                      _p(V), _p(dO), float(scale), _p(dQ), _p(dK), _p(dV))
    return dQ, dK, dV


def spmm_typed(row_ptr, col_idx, edge_type, vals, Z):
    """Multi-relation SpMM: Y[i] = sum_p vals[p] Z[edge_type[p], col_idx[p]]; Z is [R, n_cols, F]."""
    lib = _load()
    row_ptr, col_idx, edge_type = _i32(row_ptr), _i32(col_idx), _i32(edge_type)
    Z = np.ascontiguousarray(Z, dtype=np.float32)
    R, n_cols, F = Z.shape
    if edge_type.size and (edge_type.min() < 0 or edge_type.max() >= R):
        raise ValueError("edge type out of range")
    v = None if vals is None else _f32(vals)
    Y = np.zeros((row_ptr.size - 1, F))
    lib.oracle_spmm_typed(row_ptr.size - 1, n_cols, _p(row_ptr), _p(col_idx), _p(edge_type), _p(v),
                          _p(Z.reshape(R * n_cols, F)), F, F, _p(Y))
    return Y


def edge_softmax_aggregate(row_ptr, col_idx, scores, V, heads: int = 1, rows=None):
    """The benchmark page's op: softmax of given edge scores per row, then the
    weighted sum of source values. Composed from row_softmax and spmm."""
    W = row_softmax(row_ptr, np.asarray(scores, dtype=np.float64).reshape(-1, heads))
    # weights are used as float64 here; round-trip through float32 would lose
    # precision, so aggregate directly in double.
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    V = np.asarray(V, dtype=np.float32)
    n_rows = row_ptr.shape[0] - 1
    rr = np.arange(n_rows) if rows is None else np.asarray(rows, dtype=np.int64)
    D = V.shape[1] // heads
    out = np.zeros((rr.size, V.shape[1]), dtype=np.float64)
    for k, i in enumerate(rr):
        b, e = int(row_ptr[i]), int(row_ptr[i + 1])
        if e == b:
            continue
        src = col_idx[b:e]
        for h in range(heads):
            out[k, h * D:(h + 1) * D] = W[b:e, h] @ V[src, h * D:(h + 1) * D].astype(np.float64)
    return out


def transpose(row_ptr, col_idx, vals, n_cols: int):
    """CSR of A^T by a stable counting sort (entries of each column keep row order)."""
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    n_rows = row_ptr.shape[0] - 1
    nnz = int(row_ptr[-1])
    v = None if vals is None else _f32(vals)
    rpt = np.zeros(n_cols + 1, dtype=np.int32)
    cit = np.zeros(nnz, dtype=np.int32)
    vt = None if v is None else np.zeros(nnz, dtype=np.float32)
    lib.oracle_transpose(n_rows, n_cols, _p(row_ptr), _p(col_idx), _p(v), _p(rpt), _p(cit), _p(vt))
    return rpt, cit, vt


def spmm_t(row_ptr, col_idx, vals, G, n_cols: int, rows=None):
    """G_X = A^T G: transpose by counting sort, then the SpMM loop."""
    rpt, cit, vt = transpose(row_ptr, col_idx, vals, n_cols)
    return spmm(rpt, cit, vt, G, rows=rows)


def spmm_t_scatter(row_ptr, col_idx, vals, G, n_cols: int):
    """G_X = A^T G by scattering each edge's contribution (second route)."""
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    G, ldg = _matrix(G)
    v = None if vals is None else _f32(vals)
    out = np.zeros((n_cols, G.shape[1]), dtype=np.float64)
    lib.oracle_spmm_t_scatter(row_ptr.shape[0] - 1, n_cols, _p(row_ptr), _p(col_idx), _p(v), _p(G),
                              ldg, G.shape[1], _p(out))
    return out


def row_stats(row_ptr, long_threshold: int = 1024):
    """Row-length statistics: (ints[40], reals[2]); layout documented in oracle.c."""
    lib = _load()
    row_ptr = _i32(row_ptr)
    ints = np.zeros(40, dtype=np.int64)
    reals = np.zeros(2, dtype=np.float64)
    lib.oracle_row_stats(row_ptr.shape[0] - 1, _p(row_ptr), int(long_threshold), _p(ints), _p(reals))
    return ints, reals


def fingerprint(row_ptr, col_idx) -> int:
    """64-bit order-independent fingerprint of a CSR structure (see oracle.c)."""
    lib = _load()
    row_ptr, col_idx = _i32(row_ptr), _i32(col_idx)
    return int(lib.oracle_fingerprint(row_ptr.shape[0] - 1, _p(row_ptr), _p(col_idx)))


def set_threads(n: int) -> None:
    """Threads of the oracle's row-parallel loops (timing only; results do not depend on it)."""
    _load().oracle_set_threads(int(n))


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return os.cpu_count() or 1
