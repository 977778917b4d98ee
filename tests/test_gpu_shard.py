"""Row-sharded aggregation on one GPU: the shards of a 2- and 3-way split run
one after the other through the C ABI, and their outputs, concatenated, are
compared with the whole-graph oracle element by element.

The exchange step is emulated on the one device by concatenating the row
blocks each shard owns (the multi-process all-gather itself is tested with
gloo ranks on the CPU); the halo rows are packed by the library's GPU gather
(checked bit-exact), and each shard runs the library's planned kernels on its
own CSR: SpMM, SDDMM, fused attention, and SpMM with A^T over the rows of A^T.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_F32, assert_close, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402
from sparse_gnn_aggregation_gb300 import shard as sh  # noqa: E402

FLAGS = sga.PLAN_PROBE | sga.PLAN_NO_CACHE


@pytest.fixture(scope="module")
def graph():
    g = synth.rmat_skew(14, seed=8)
    return g.with_vals(synth.uniform_vals(g, 8))


def owned_then_exchanged(M, bounds):
    """The exchange on one device: each shard's owned block, concatenated."""
    blocks = [torch.from_numpy(np.ascontiguousarray(M[bounds[k]:bounds[k + 1]])).cuda()
              for k in range(len(bounds) - 1)]
    return torch.cat(blocks)


@pytest.mark.parametrize("world", [2, 3])
def test_shards_match_the_whole_graph(graph, world):
    g = graph
    F, H, D = 32, 4, 16
    X = synth.normal(g.n_cols, F, 9, synth.STREAM_X)
    Q = synth.normal(g.n_rows, H * D, 9, synth.STREAM_Q)
    K = synth.normal(g.n_cols, H * D, 9, synth.STREAM_K)
    V = synth.normal(g.n_cols, H * D, 9, synth.STREAM_V)
    bounds = sga.autosage_partition_rows(g.row_ptr, world)
    Xf, Kf, Vf = (owned_then_exchanged(M, bounds) for M in (X, K, V))
    Ys, Ss, Os = [], [], []
    for r in range(world):
        s = sh.make_shard(g.row_ptr, g.col_idx, g.vals, g.n_cols, r, world, bounds)
        A = s.csr()
        halo = torch.from_numpy(s.halo).cuda()
        Xh = sh.halo_rows(Xf, halo)
        assert torch.equal(Xh.cpu(), torch.from_numpy(X[s.halo])), "halo gather is not exact"
        Kh, Vh = sh.halo_rows(Kf, halo), sh.halo_rows(Vf, halo)
        Qr = torch.from_numpy(np.ascontiguousarray(Q[s.row_begin:s.row_end])).cuda()
        Ys.append(to_np(sga.autosage_spmm(A, Xh, plan=sga.autosage_plan(A, sga.OP_SPMM, F, flags=FLAGS))))
        Ss.append(to_np(sga.autosage_sddmm(A, Qr, Kh, 0.25,
                                           plan=sga.autosage_plan(A, sga.OP_SDDMM, H * D, flags=FLAGS))))
        Os.append(to_np(sga.autosage_csr_attention(A, Qr, Kh, Vh, H, 0.25,
                                                   plan=sga.autosage_plan(A, sga.OP_ATTN, D, heads=H, flags=FLAGS))))
    assert_close(np.concatenate(Ys), oracle.spmm(g.row_ptr, g.col_idx, g.vals, X), TOL_F32, f"{world} shards: spmm")
    assert_close(np.concatenate(Ss), oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 0.25)[:, 0], TOL_F32,
                 f"{world} shards: sddmm")
    assert_close(np.concatenate(Os), oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, H, 0.25), TOL_F32,
                 f"{world} shards: attention")


def test_transpose_shards_over_the_rows_of_a_transposed(graph):
    g = graph
    world, F = 2, 24
    G = synth.normal(g.n_rows, F, 10, synth.STREAM_G)
    rpt, cit, vt = sh.transpose_host(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    ort, oct_, ovt = oracle.transpose(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    np.testing.assert_array_equal(rpt, ort)
    np.testing.assert_array_equal(cit, oct_)
    in_bounds = sga.autosage_partition_rows(g.row_ptr, world)  # who owns which rows of G
    Gf = owned_then_exchanged(G, in_bounds)
    out = []
    for r in range(world):
        s = sh.make_shard(rpt, cit, vt, g.n_rows, r, world)
        A = s.csr()
        Gh = sh.halo_rows(Gf, torch.from_numpy(s.halo).cuda())
        out.append(to_np(sga.autosage_spmm(A, Gh, plan=sga.autosage_plan(A, sga.OP_SPMM, F, flags=FLAGS))))
    assert_close(np.concatenate(out), oracle.spmm_t(g.row_ptr, g.col_idx, g.vals, G, g.n_cols), TOL_F32,
                 "sharded SpMM with A^T")


def test_gather_rows_widths_and_dtypes():
    rng = np.random.default_rng(3)
    for F, dt in ((1, torch.float32), (3, torch.float32), (64, torch.float32), (5, torch.bfloat16),
                  (64, torch.bfloat16)):
        X = torch.from_numpy(rng.standard_normal((500, F + 3), dtype=np.float32)).to(dt).cuda()[:, :F]
        idx = torch.from_numpy(rng.integers(0, 500, 777).astype(np.int32)).cuda()
        got = sga.autosage_gather_rows(X, idx)
        assert torch.equal(got.cpu(), X.cpu()[idx.cpu().long()]), f"gather F={F} {dt}"
