"""Python binding of libautosage (CSR SpMM / SDDMM / CSR attention on GB300).

Argument marshalling only: every step runs in the library's CUDA kernels
behind the C ABI in ``include/autosage.h``. PyTorch supplies device memory
and the current stream; there is no CPU or vendor-library path. Nothing
works until the native library is built (run
``python -m sparse_gnn_aggregation_gb300.build`` or ``__graft_entry__.build()``):
the first call into the library raises ImportError.

Operations (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN
Aggregation (SpMM/SDDMM) and CSR Attention", Abstract): SpMM, SDDMM, the
CSR attention pipeline SDDMM -> row-softmax -> SpMM, schedule planning with
a cost estimate and micro-probes, and a persistent plan cache.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libautosage.so")

# ---------------------------------------------------------------- constants (autosage.h)
OK, ERR_INVALID_ARG, ERR_INVALID_CSR, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3, 4
ERR_CACHE_IO, ERR_CACHE_FORMAT, ERR_PROBE, ERR_PLAN_MISMATCH = 5, 6, 7, 8
F32, BF16 = 0, 1
OP_SPMM, OP_SPMM_T, OP_SDDMM, OP_ATTN, OP_ATTN_UNFUSED, OP_SOFTMAX, OP_ATTN_BACKWARD = 0, 1, 2, 3, 4, 5, 6
SCHED_AUTO, SCHED_ROWGROUP, SCHED_SPLIT, SCHED_MERGEPATH, SCHED_BINNED, SCHED_HYBRID = -1, 0, 1, 2, 3, 4
PLAN_PROBE, PLAN_NO_CACHE, PLAN_VERIFY, PLAN_FIXED_VALUES = 1, 2, 4, 8

EXPORTS = [
    "autosage_spmm", "autosage_sddmm", "autosage_row_softmax", "autosage_csr_attention",
    "autosage_edge_softmax_aggregate", "autosage_plan", "autosage_plan_with_schedule",
    "autosage_plan_destroy", "autosage_plan_describe", "autosage_plan_schedule",
    "autosage_cache_load", "autosage_cache_save", "autosage_cache_clear", "autosage_cache_size",
    "autosage_row_stats", "autosage_fingerprint", "autosage_validate_csr", "autosage_csr_transpose",
    "autosage_status_string", "autosage_last_error", "autosage_version",
    "autosage_csr_attention_unfused_noalloc", "autosage_csr_attention_backward",
    "autosage_plan_typed", "autosage_spmm_typed", "autosage_plan_rebind",
    "autosage_partition_rows", "autosage_shard_halo", "autosage_gather_rows", "autosage_measure_gather",
]


class AutosageError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class _Csr(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("n_cols", ctypes.c_int64), ("nnz", ctypes.c_int64),
                ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p), ("vals", ctypes.c_void_p)]


class _Schedule(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("lanes_f", ctypes.c_int), ("lanes_e", ctypes.c_int),
                ("split", ctypes.c_int), ("per_edge", ctypes.c_int), ("lanes_f_agg", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libautosage.so is not built ({LIB_PATH}); run "
                          "`python -m sparse_gnn_aggregation_gb300.build` first")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I, F, U = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint
    CSR = ctypes.POINTER(_Csr)
    sig = {
        "autosage_spmm": [CSR, P, I64, P, I64, I64, I, I, P, P],
        "autosage_sddmm": [CSR, P, I64, P, I64, I64, I, F, P, P, P],
        "autosage_row_softmax": [CSR, P, I, P, P],
        "autosage_csr_attention": [CSR, P, P, P, I, I64, I, F, P, I, P, P],
        "autosage_csr_attention_unfused_noalloc": [CSR, P, P, P, I, I64, I, F, P, P],
        "autosage_csr_attention_backward": [CSR, P, P, P, P, I, I64, I, F, P, P, P, P, P],
        "autosage_plan_typed": [CSR, P, I, I64, I, U, ctypes.POINTER(P), P],
        "autosage_spmm_typed": [CSR, P, I, P, I64, P, I64, I64, I, P, P],
        "autosage_edge_softmax_aggregate": [CSR, P, P, I, I64, I, P, P, P],
        "autosage_plan": [CSR, I, I64, I, I, U, ctypes.POINTER(P), P],
        "autosage_plan_with_schedule": [CSR, I, I64, I, I, ctypes.POINTER(_Schedule), ctypes.POINTER(P), P],
        "autosage_plan_destroy": [P],
        "autosage_plan_rebind": [P, CSR, P],
        "autosage_plan_describe": [P, ctypes.c_char_p, ctypes.c_size_t],
        "autosage_plan_schedule": [P, ctypes.POINTER(_Schedule), ctypes.POINTER(ctypes.c_double)],
        "autosage_cache_load": [ctypes.c_char_p],
        "autosage_cache_save": [ctypes.c_char_p],
        "autosage_cache_clear": [],
        "autosage_row_stats": [CSR, I64, P, P, P],
        "autosage_fingerprint": [CSR, ctypes.POINTER(ctypes.c_uint64), P],
        "autosage_validate_csr": [CSR, P],
        "autosage_csr_transpose": [CSR, P, P, P, P],
        "autosage_partition_rows": [P, I64, I, P],
        "autosage_shard_halo": [P, P, I64, I64, I64, P, P, P],
        "autosage_gather_rows": [P, I64, P, I64, I64, I, P, I64, P],
        "autosage_measure_gather": [I64, I, I64, I, ctypes.POINTER(ctypes.c_double), P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.autosage_cache_size.argtypes = []
    lib.autosage_cache_size.restype = ctypes.c_int64
    for name in ("autosage_status_string",):
        getattr(lib, name).argtypes = [ctypes.c_int]
        getattr(lib, name).restype = ctypes.c_char_p
    for name in ("autosage_last_error", "autosage_version"):
        getattr(lib, name).argtypes = []
        getattr(lib, name).restype = ctypes.c_char_p
    return lib


class _LazyLib:
    """Loads libautosage.so on first use; raises ImportError if it is not built."""

    _handle = None

    def __getattr__(self, name):
        if _LazyLib._handle is None:
            _LazyLib._handle = _load()
        return getattr(_LazyLib._handle, name)


_lib = _LazyLib()


def _check(status: int):
    if status != OK:
        msg = _lib.autosage_last_error().decode() or _lib.autosage_status_string(status).decode()
        raise AutosageError(status, msg)


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}; float32 or bfloat16")


def _ld(t) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("feature matrices must be 2-D with unit column stride")
    return int(t.stride(0))


def _head_width(T, heads: int):
    """(W, D) of a [n, heads * D] or [n, heads, D] attention tensor; rejects heads that do not divide W."""
    heads = int(heads)
    if heads < 1:
        raise ValueError("heads must be >= 1")
    W = int(T.shape[-1]) if T.dim() == 2 else int(T.shape[-1] * T.shape[-2])
    if W % heads:
        raise ValueError(f"row width {W} is not a multiple of heads = {heads}")
    return W, W // heads


def _same_layout(ref, rows: int, what: str, *tensors):
    """Every tensor: contiguous, ref's dtype and device, ``rows`` rows of ref's row width."""
    for name, t in tensors:
        if not t.is_contiguous():
            raise ValueError(f"{what}: {name} must be contiguous")
        if t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError(f"{what}: {name} must have the dtype and device of the first input")
        if int(t.shape[0]) != rows or tuple(t.shape[1:]) != tuple(ref.shape[1:]):
            raise ValueError(f"{what}: {name} has shape {tuple(t.shape)}, expected {(rows,) + tuple(ref.shape[1:])}")


# ---------------------------------------------------------------- CSR handle

@dataclasses.dataclass
class CsrMatrix:
    """A CSR graph in device memory (int32 row_ptr/col_idx, float32 vals or None)."""

    row_ptr: "object"
    col_idx: "object"
    vals: "object" = None
    n_cols: int | None = None

    def __post_init__(self):
        torch = _torch()
        for name in ("row_ptr", "col_idx"):
            t = getattr(self, name)
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous int32 tensor")
        if self.vals is not None and (self.vals.dtype != torch.float32 or not self.vals.is_contiguous()):
            raise TypeError("vals must be a contiguous float32 tensor")
        self.n_rows = int(self.row_ptr.numel()) - 1
        self.nnz = int(self.col_idx.numel())
        if self.n_cols is None:
            self.n_cols = self.n_rows
        self._c = _Csr(self.n_rows, int(self.n_cols), self.nnz, self.row_ptr.data_ptr(),
                       self.col_idx.data_ptr() if self.nnz else 0,
                       self.vals.data_ptr() if self.vals is not None else 0)

    @property
    def c(self):
        return ctypes.byref(self._c)

    @classmethod
    def from_numpy(cls, row_ptr, col_idx, vals=None, n_cols=None, device="cuda"):
        torch = _torch()
        rp = torch.from_numpy(np.ascontiguousarray(row_ptr, dtype=np.int32)).to(device)
        ci = torch.from_numpy(np.ascontiguousarray(col_idx, dtype=np.int32)).to(device)
        v = None if vals is None else torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32)).to(device)
        return cls(rp, ci, v, n_cols)


# ---------------------------------------------------------------- plans

class Plan:
    """Owns an autosage_plan_t; destroyed with the object."""

    def __init__(self, handle: int, op: int):
        self.handle = ctypes.c_void_p(handle)
        self.op = op

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(512)
        _check(_lib.autosage_plan_describe(self.handle, buf, 512))
        return buf.value.decode()

    def schedule(self):
        s = _Schedule()
        ms = ctypes.c_double()
        _check(_lib.autosage_plan_schedule(self.handle, ctypes.byref(s), ctypes.byref(ms)))
        return {"kind": s.kind, "lanes_f": s.lanes_f, "lanes_e": s.lanes_e, "split": s.split,
                "per_edge": s.per_edge, "lanes_f_agg": s.lanes_f_agg, "probe_ms": ms.value}

    def rebind(self, A: "CsrMatrix", stream=None):
        """Bind the plan to a copy of its graph's structure in other device memory
        (checked by fingerprint on the GPU; raises ERR_PLAN_MISMATCH for another graph)."""
        _check(_lib.autosage_plan_rebind(self.handle, A.c, _stream(stream)))
        return self

    def close(self):
        if self.handle and self.handle.value:
            _lib.autosage_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _plan_handle(plan):
    return plan.handle if plan is not None else ctypes.c_void_p(0)


def autosage_plan(A: CsrMatrix, op: int, F: int, heads: int = 1, dtype=None, flags: int = 0, stream=None,
                  allow_probe_failure: bool = False) -> Plan:
    torch = _torch()
    dt = BF16 if dtype == torch.bfloat16 else F32
    h = ctypes.c_void_p()
    st = _lib.autosage_plan(A.c, op, int(F), int(heads), dt, int(flags), ctypes.byref(h), _stream(stream))
    if st == ERR_PROBE and allow_probe_failure and h.value:
        return Plan(h.value, op)
    _check(st)
    return Plan(h.value, op)


def autosage_plan_with_schedule(A: CsrMatrix, op: int, F: int, kind: int, lanes_f: int = 0, lanes_e: int = 0,
                                split: int = 0, heads: int = 1, dtype=None, stream=None, per_edge: int = 0,
                                lanes_f_agg: int = 0) -> Plan:
    torch = _torch()
    dt = BF16 if dtype == torch.bfloat16 else F32
    s = _Schedule(kind, lanes_f, lanes_e, split, int(bool(per_edge)), int(lanes_f_agg))
    h = ctypes.c_void_p()
    _check(_lib.autosage_plan_with_schedule(A.c, op, int(F), int(heads), dt, ctypes.byref(s), ctypes.byref(h),
                                            _stream(stream)))
    return Plan(h.value, op)


def autosage_plan_rebind(plan: Plan, A: CsrMatrix, stream=None) -> Plan:
    """Bind ``plan`` to A's structure arrays when they moved (same graph in other
    device memory). Raises AutosageError(ERR_PLAN_MISMATCH) for another graph."""
    return plan.rebind(A, stream)


# ---------------------------------------------------------------- ops

def autosage_spmm(A: CsrMatrix, X, Y=None, transpose: bool = False, plan: Plan | None = None, stream=None):
    """Y = A X (or A^T X with a plan built for OP_SPMM_T). Returns Y."""
    torch = _torch()
    F = int(X.shape[1])
    rows = A.n_cols if transpose else A.n_rows
    if Y is None:
        Y = torch.empty((rows, F), dtype=X.dtype, device=X.device)
    if Y.dtype != X.dtype:
        raise TypeError("X and Y must have the same dtype")
    _check(_lib.autosage_spmm(A.c, _ptr(X), _ld(X), _ptr(Y), _ld(Y), F, _dt(X), int(bool(transpose)),
                              _plan_handle(plan), _stream(stream)))
    return Y


def autosage_sddmm(A: CsrMatrix, Q, K, alpha: float = 1.0, out=None, plan: Plan | None = None, stream=None):
    """out[p] = alpha * <Q[row(p)], K[col_idx[p]]> (fp32, CSR order). Returns out."""
    torch = _torch()
    if out is None:
        out = torch.empty(A.nnz, dtype=torch.float32, device=Q.device)
    if Q.dtype != K.dtype:
        raise TypeError("Q and K must have the same dtype")
    _check(_lib.autosage_sddmm(A.c, _ptr(Q), _ld(Q), _ptr(K), _ld(K), int(Q.shape[1]), _dt(Q), float(alpha),
                               _ptr(out), _plan_handle(plan), _stream(stream)))
    return out


def autosage_row_softmax(A: CsrMatrix, scores, heads: int = 1, plan: Plan | None = None, stream=None):
    """Row softmax of fp32 edge scores [nnz, heads], in place. Returns scores."""
    _check(_lib.autosage_row_softmax(A.c, _ptr(scores), int(heads), _plan_handle(plan), _stream(stream)))
    return scores


def autosage_csr_attention(A: CsrMatrix, Q, K, V, heads: int, scale: float, fused: bool = True, out=None,
                           plan: Plan | None = None, stream=None):
    """CSR attention; Q, K, V, out are [n, heads * D] (= [n, heads, D] contiguous)."""
    torch = _torch()
    _, D = _head_width(Q, heads)
    if out is None:
        out = torch.empty_like(Q)
    _same_layout(Q, A.n_rows, "attention", ("Q", Q), ("out", out))
    _same_layout(Q, A.n_cols, "attention", ("K", K), ("V", V))
    _check(_lib.autosage_csr_attention(A.c, _ptr(Q), _ptr(K), _ptr(V), int(heads), D, _dt(Q), float(scale),
                                       _ptr(out), int(bool(fused)), _plan_handle(plan), _stream(stream)))
    return out


def autosage_plan_typed(A: CsrMatrix, edge_type, num_types: int, F: int, dtype=None, flags: int = 0,
                        stream=None) -> Plan:
    """Plan for the multi-relation SpMM (checks the edge types on the GPU)."""
    torch = _torch()
    dt = BF16 if dtype == torch.bfloat16 else F32
    if edge_type.dtype != torch.int32 or not edge_type.is_contiguous():
        raise TypeError("edge_type must be a contiguous int32 tensor")
    h = ctypes.c_void_p()
    _check(_lib.autosage_plan_typed(A.c, _ptr(edge_type), int(num_types), int(F), dt, int(flags), ctypes.byref(h),
                                    _stream(stream)))
    return Plan(h.value, OP_SPMM)


def autosage_spmm_typed(A: CsrMatrix, edge_type, Z, Y=None, plan: Plan | None = None, stream=None):
    """Y[i] = sum_p vals[p] Z[edge_type[p], col_idx[p]] with Z [num_types, n_cols, F]."""
    torch = _torch()
    if Z.dim() != 3 or not Z.is_contiguous():
        raise ValueError("Z must be a contiguous [num_types, n_cols, F] tensor")
    R, _, F = (int(x) for x in Z.shape)
    if Y is None:
        Y = torch.empty((A.n_rows, F), dtype=Z.dtype, device=Z.device)
    _check(_lib.autosage_spmm_typed(A.c, _ptr(edge_type), R, _ptr(Z), F, _ptr(Y), _ld(Y), F, _dt(Z),
                                    _plan_handle(plan), _stream(stream)))
    return Y


def autosage_csr_attention_backward(A: CsrMatrix, Q, K, V, dO, heads: int, scale: float, dQ=None, dK=None,
                                    dV=None, plan: Plan | None = None, stream=None):
    """Gradients (dQ, dK, dV) of CSR attention for the upstream gradient dO.

    All tensors are [n, heads * D] contiguous of one dtype. ``plan`` should be
    built for OP_ATTN_BACKWARD with F = D; without one the call builds a
    temporary plan (allocating and synchronising)."""
    torch = _torch()
    _, D = _head_width(Q, heads)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    _same_layout(Q, A.n_rows, "attention backward", ("Q", Q), ("dO", dO), ("dQ", dQ))
    _same_layout(Q, A.n_cols, "attention backward", ("K", K), ("V", V), ("dK", dK), ("dV", dV))
    _check(_lib.autosage_csr_attention_backward(A.c, _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), int(heads), D,
                                                _dt(Q), float(scale), _ptr(dQ), _ptr(dK), _ptr(dV),
                                                _plan_handle(plan), _stream(stream)))
    return dQ, dK, dV


NOALLOC_MAX_SCORES = 4 * 1024 * 1024


def autosage_csr_attention_unfused_noalloc(A: CsrMatrix, Q, K, V, heads: int, scale: float, out, stream=None):
    """Unfused CSR attention that allocates no device memory in the library.

    For callers that must not allocate inside their work loop. The caller
    passes every input and the output (``out`` is required); the score array
    lives in a fixed 16 MiB device array inside the library, so nnz * heads
    may not exceed NOALLOC_MAX_SCORES. Calls that overlap on the GPU share
    that array and must be serialised by the caller.
    """
    _, D = _head_width(Q, heads)
    _same_layout(Q, A.n_rows, "attention", ("Q", Q), ("out", out))
    _same_layout(Q, A.n_cols, "attention", ("K", K), ("V", V))
    _check(_lib.autosage_csr_attention_unfused_noalloc(A.c, _ptr(Q), _ptr(K), _ptr(V), int(heads), D,
                                                       _dt(Q), float(scale), _ptr(out), _stream(stream)))
    return out


def autosage_edge_softmax_aggregate(A: CsrMatrix, scores, V, heads: int = 1, out=None, plan: Plan | None = None,
                                    stream=None):
    """Softmax of given fp32 scores [nnz, heads] per row, then weighted sum of V rows."""
    torch = _torch()
    _, D = _head_width(V, heads)
    if out is None:
        out = torch.empty((A.n_rows,) + tuple(V.shape[1:]), dtype=V.dtype, device=V.device)
    _same_layout(V, A.n_cols, "edge softmax aggregation", ("V", V))
    _same_layout(V, A.n_rows, "edge softmax aggregation", ("out", out))
    if scores.dtype != torch.float32 or not scores.is_contiguous() or scores.numel() != A.nnz * int(heads):
        raise ValueError("scores must be a contiguous float32 tensor of nnz * heads elements")
    _check(_lib.autosage_edge_softmax_aggregate(A.c, _ptr(scores), _ptr(V), int(heads), D, _dt(V),
                                                _ptr(out), _plan_handle(plan), _stream(stream)))
    return out


# ---------------------------------------------------------------- utilities

def autosage_row_stats(A: CsrMatrix, long_threshold: int = 1024, stream=None):
    ints = np.zeros(40, dtype=np.int64)
    reals = np.zeros(2, dtype=np.float64)
    _check(_lib.autosage_row_stats(A.c, int(long_threshold), ints.ctypes.data_as(ctypes.c_void_p),
                                   reals.ctypes.data_as(ctypes.c_void_p), _stream(stream)))
    return ints, reals


def autosage_fingerprint(A: CsrMatrix, stream=None) -> int:
    out = ctypes.c_uint64()
    _check(_lib.autosage_fingerprint(A.c, ctypes.byref(out), _stream(stream)))
    return int(out.value)


def autosage_validate_csr(A: CsrMatrix, stream=None) -> int:
    """Returns OK or ERR_INVALID_CSR (does not raise for an invalid structure)."""
    st = _lib.autosage_validate_csr(A.c, _stream(stream))
    if st not in (OK, ERR_INVALID_CSR):
        _check(st)
    return st


def autosage_csr_transpose(A: CsrMatrix, stream=None):
    """CSR of A^T on the GPU: (row_ptr_t, col_idx_t, vals_t or None)."""
    torch = _torch()
    dev = A.row_ptr.device
    rpt = torch.empty(A.n_cols + 1, dtype=torch.int32, device=dev)
    cit = torch.empty(max(A.nnz, 1), dtype=torch.int32, device=dev)[:A.nnz]
    vt = None if A.vals is None else torch.empty(max(A.nnz, 1), dtype=torch.float32, device=dev)[:A.nnz]
    _check(_lib.autosage_csr_transpose(A.c, _ptr(rpt), _ptr(cit), _ptr(vt), _stream(stream)))
    return rpt, cit, vt


def autosage_partition_rows(row_ptr, parts: int):
    """Equal-nnz row ranges of a HOST CSR: int64 bounds [parts + 1] (part k = rows bounds[k]..bounds[k+1])."""
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    bounds = np.zeros(int(parts) + 1, dtype=np.int64)
    _check(_lib.autosage_partition_rows(rp.ctypes.data_as(ctypes.c_void_p), rp.size - 1, int(parts),
                                        bounds.ctypes.data_as(ctypes.c_void_p)))
    return bounds


def autosage_shard_halo(row_ptr, col_idx, n_cols: int, row_begin: int, row_end: int):
    """(halo, local_col) of the shard rows [row_begin, row_end) of a HOST CSR: the sorted distinct
    columns its edges reference, and each edge's column as a position in that list."""
    rp = np.ascontiguousarray(row_ptr, dtype=np.int32)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    halo = np.empty(max(int(n_cols), 1), dtype=np.int32)
    local = np.empty(max(int(rp[row_end] - rp[row_begin]), 1), dtype=np.int32)
    nh = ctypes.c_int64()
    _check(_lib.autosage_shard_halo(rp.ctypes.data_as(ctypes.c_void_p), ci.ctypes.data_as(ctypes.c_void_p),
                                    int(n_cols), int(row_begin), int(row_end), halo.ctypes.data_as(ctypes.c_void_p),
                                    ctypes.byref(nh), local.ctypes.data_as(ctypes.c_void_p)))
    return halo[:nh.value].copy(), local[:int(rp[row_end] - rp[row_begin])].copy()


def autosage_gather_rows(X, idx, out=None, stream=None):
    """out[k] = X[idx[k]] on the GPU (X 2-D float32/bfloat16 with unit column stride, idx int32)."""
    torch = _torch()
    if idx.dtype != torch.int32 or not idx.is_contiguous():
        raise TypeError("idx must be a contiguous int32 tensor")
    F = int(X.shape[1])
    if out is None:
        out = torch.empty((int(idx.numel()), F), dtype=X.dtype, device=X.device)
    _check(_lib.autosage_gather_rows(_ptr(X), _ld(X), _ptr(idx), int(idx.numel()), F, _dt(X), _ptr(out), _ld(out),
                                     _stream(stream)))
    return out


def autosage_measure_gather(table_bytes: int, row_bytes: int = 1024, n_gathers: int = 1 << 24, reps: int = 5,
                            stream=None) -> float:
    """Read rate (GB/s) of random row gathers from a table of table_bytes on the
    current GPU: L2-resident tables give the L2 rate for hot rows, large ones
    the DRAM rate. Synchronises the stream."""
    g = ctypes.c_double()
    _check(_lib.autosage_measure_gather(int(table_bytes), int(row_bytes), int(n_gathers), int(reps), ctypes.byref(g),
                                        _stream(stream)))
    return g.value


def autosage_cache_load(path: str):
    _check(_lib.autosage_cache_load(os.fsencode(path)))


def autosage_cache_save(path: str):
    _check(_lib.autosage_cache_save(os.fsencode(path)))


def autosage_cache_clear():
    _check(_lib.autosage_cache_clear())


def autosage_cache_size() -> int:
    return int(_lib.autosage_cache_size())


def autosage_version() -> str:
    return _lib.autosage_version().decode()


def library():
    """The loaded ctypes library (for symbol checks)."""
    _lib.autosage_version  # force the load
    return _LazyLib._handle
