"""The allocation-free unfused attention entry point.

Some callers cannot allocate device memory inside their work loop (a server
that reserved all device memory for its own pool up front, or a
latency-critical loop that must not enter the driver's allocator). For them
the library offers autosage_csr_attention_unfused_noalloc, which keeps the
score array in a fixed device array instead of allocating it. This test calls
it through the C ABI twice in a row and checks each result against the
regular autosage_csr_attention (fused = 0, no plan), within the fp32 parity
tolerance, and checks that an over-size call is refused before any launch.
The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import TOL_F32, assert_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402


def _inputs(seed, heads, D):
    g = synth.rmat_skew(12, seed=seed)
    W = heads * D
    Q = torch.from_numpy(synth.normal(g.n_rows, W, seed, synth.STREAM_Q)).cuda()
    K = torch.from_numpy(synth.normal(g.n_cols, W, seed, synth.STREAM_K)).cuda()
    V = torch.from_numpy(synth.normal(g.n_cols, W, seed, synth.STREAM_V)).cuda()
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    return g, A, Q, K, V


@pytest.mark.parametrize("heads,D", [(1, 32), (4, 16)])
def test_noalloc_matches_regular_entry_point_twice(heads, D):
    lib = sga.library()
    outs = []
    for seed in (1, 2):  # two calls in a row on different inputs share the scratch
        g, A, Q, K, V = _inputs(seed, heads, D)
        assert g.nnz * heads <= sga.NOALLOC_MAX_SCORES
        out = torch.full_like(Q, float("nan"))
        stream = torch.cuda.current_stream()
        st = lib.autosage_csr_attention_unfused_noalloc(A.c, ctypes.c_void_p(Q.data_ptr()),
                                                        ctypes.c_void_p(K.data_ptr()),
                                                        ctypes.c_void_p(V.data_ptr()), heads, D, sga.F32,
                                                        ctypes.c_float(1.0 / np.sqrt(D)),
                                                        ctypes.c_void_p(out.data_ptr()),
                                                        ctypes.c_void_p(stream.cuda_stream))
        assert st == sga.OK, lib.autosage_last_error().decode()
        ref = sga.autosage_csr_attention(A, Q, K, V, heads, 1.0 / np.sqrt(D), fused=False)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref.cpu().numpy(), TOL_F32, f"no-alloc call {seed}")
        outs.append(out)
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_refuses_oversize():
    g = synth.Csr(4, 4, np.array([0, 1, 2, 3, 4], np.int32), np.array([0, 1, 2, 3], np.int32), None)
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, None, 4)
    heads = sga.NOALLOC_MAX_SCORES // 4 + 1  # nnz * heads just above the scratch size
    x = torch.zeros(4, heads, device="cuda")
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_csr_attention_unfused_noalloc(A, x, x, x, heads, 1.0, torch.empty_like(x))
    assert e.value.status == sga.ERR_UNSUPPORTED
    assert "AUTOSAGE_NOALLOC_MAX_SCORES" in str(e.value)
