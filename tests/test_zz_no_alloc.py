"""The allocation-free unfused attention entry point.

Some callers cannot allocate device memory inside their work loop: a server
that reserved all device memory for its own pool up front, or a
latency-critical loop that must not enter the driver's allocator (an
allocation can synchronise the device and take unbounded time). For them the
library offers autosage_csr_attention_unfused_noalloc, which keeps the fp32
score array in a fixed device array of the library instead of allocating it.

These tests call it through the C ABI and check its output against the fp64
oracle (the same tolerance as every fp32 parity test) on two calls in a row
with different inputs, on a skewed graph whose hub rows are over a thousand
edges long, check that a call leaves the device's memory pool and free
memory untouched, and that an over-size call is refused before any launch.
The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_F32, assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402


def _inputs(g, seed, heads, D):
    W = heads * D
    Q = synth.normal(g.n_rows, W, seed, synth.STREAM_Q)
    K = synth.normal(g.n_cols, W, seed, synth.STREAM_K)
    V = synth.normal(g.n_cols, W, seed, synth.STREAM_V)
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    return A, Q, K, V


def _call_c_abi(A, Qd, Kd, Vd, heads, D, out):
    lib = sga.library()
    stream = torch.cuda.current_stream()
    return lib.autosage_csr_attention_unfused_noalloc(
        A.c, ctypes.c_void_p(Qd.data_ptr()), ctypes.c_void_p(Kd.data_ptr()), ctypes.c_void_p(Vd.data_ptr()),
        heads, D, sga.F32, ctypes.c_float(1.0 / np.sqrt(D)), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("heads,D", [(1, 32), (4, 16)])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(heads, D):
    outs = []
    for seed in (1, 2):  # two calls in a row, different graphs and inputs, one shared scratch
        g = synth.rmat_skew(12, seed=seed)
        A, Q, K, V = _inputs(g, seed, heads, D)
        assert g.nnz * heads <= sga.NOALLOC_MAX_SCORES
        Qd, Kd, Vd = (torch.from_numpy(x).cuda() for x in (Q, K, V))
        out = torch.full_like(Qd, float("nan"))
        st = _call_c_abi(A, Qd, Kd, Vd, heads, D, out)
        assert st == sga.OK, sga.library().autosage_last_error().decode()
        torch.cuda.synchronize()
        want = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, heads, 1.0 / np.sqrt(D))
        assert_close(out.cpu().numpy(), want, TOL_F32, f"no-alloc call {seed}")
        outs.append(out.cpu())
    assert outs[0].shape != outs[1].shape or not torch.equal(outs[0], outs[1])


def test_noalloc_hub_rows_longer_than_any_chunk():
    # R-MAT scale 13: hub rows of over a thousand edges, which the default
    # schedule walks whole (one lane group per row, no cutting)
    g = synth.rmat_skew(13, seed=3)
    heads, D = 2, 16
    assert int(g.degrees().max()) > 1024
    A, Q, K, V = _inputs(g, 5, heads, D)
    Qd, Kd, Vd = (torch.from_numpy(x).cuda() for x in (Q, K, V))
    out = torch.empty_like(Qd)
    assert _call_c_abi(A, Qd, Kd, Vd, heads, D, out) == sga.OK
    torch.cuda.synchronize()
    want = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, heads, 1.0 / np.sqrt(D))
    assert_close(out.cpu().numpy(), want, TOL_F32, "no-alloc on hub rows")


def _cudart():
    return ctypes.CDLL("libcudart.so.13")


def _pool_attr(rt, pool, attr):
    v = ctypes.c_uint64(0)
    assert rt.cudaMemPoolGetAttribute(pool, attr, ctypes.byref(v)) == 0
    return v.value


def test_noalloc_call_allocates_nothing():
    # The first call on a device loads the library's device code, which holds
    # the fixed score array; from then on a call must neither take memory from
    # the device's stream-ordered pool nor change the free device memory.
    USED_CURRENT, USED_HIGH = 7, 8  # cudaMemPoolAttrUsedMemCurrent / UsedMemHigh
    g = synth.rmat_skew(12, seed=4)
    heads, D = 2, 16
    A, Q, K, V = _inputs(g, 4, heads, D)
    Qd, Kd, Vd = (torch.from_numpy(x).cuda() for x in (Q, K, V))
    out = torch.empty_like(Qd)
    assert _call_c_abi(A, Qd, Kd, Vd, heads, D, out) == sga.OK
    torch.cuda.synchronize()
    rt = _cudart()
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), torch.cuda.current_device()) == 0
    used = _pool_attr(rt, pool, USED_CURRENT)
    zero = ctypes.c_uint64(0)
    assert rt.cudaMemPoolSetAttribute(pool, USED_HIGH, ctypes.byref(zero)) == 0  # reset the high watermark
    free0, free1, total = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    assert rt.cudaMemGetInfo(ctypes.byref(free0), ctypes.byref(total)) == 0
    assert _call_c_abi(A, Qd, Kd, Vd, heads, D, out) == sga.OK
    torch.cuda.synchronize()
    assert rt.cudaMemGetInfo(ctypes.byref(free1), ctypes.byref(total)) == 0
    assert _pool_attr(rt, pool, USED_HIGH) <= used, "the call took memory from the stream-ordered pool"
    assert free1.value == free0.value, "the call changed the free device memory"
    want = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, heads, 1.0 / np.sqrt(D))
    assert_close(out.cpu().numpy(), want, TOL_F32, "no-alloc, measured call")


def test_noalloc_refuses_oversize():
    g = synth.Csr(4, 4, np.array([0, 1, 2, 3, 4], np.int32), np.array([0, 1, 2, 3], np.int32), None)
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, None, 4)
    heads = sga.NOALLOC_MAX_SCORES // 4 + 1  # nnz * heads just above the scratch size
    x = torch.zeros(4, heads, device="cuda")
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_csr_attention_unfused_noalloc(A, x, x, x, heads, 1.0, torch.empty_like(x))
    assert e.value.status == sga.ERR_UNSUPPORTED
    assert "AUTOSAGE_NOALLOC_MAX_SCORES" in str(e.value)
