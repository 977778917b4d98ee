"""GPU parity at the full workload sizes, in the launch configuration the
benchmark uses (schedules from the planner with probes). SpMM, SpMM with A^T,
SDDMM and the forward attention are compared with the oracle on EVERY row
(the oracle runs with OpenMP on the host's cores), so every chunk, fix-up and
merge-path boundary the chosen schedules create is covered. The attention
backward's dQ is compared on every row longer than 2048 edges (each cut
into at least four chunks), an even spread of the other cut rows and of
the short rows; dK and dV through two identities at full size.

Workloads (synthetic stand-ins, seeded): R-MAT scale 20 and its uniform
control; a lognormal power-law graph shaped like OGBN-Products (2,449,029
nodes, 123.7M edges, mean aggregation); a 50-community power-law graph
shaped like Reddit (232,965 nodes, 114.6M edges); multi-head bf16 attention
on R-MAT scale 20.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_BF16, TOL_F32, assert_close, bf16_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402

FLAGS = sga.PLAN_PROBE | sga.PLAN_VERIFY


def assert_close_rows(gpu, ref, tol, what, chunk=1 << 18):
    """assert_close over blocks of rows (bounded host memory for the largest outputs)."""
    for b in range(0, ref.shape[0], chunk):
        got = gpu[b:b + chunk]
        got = got.float().cpu().numpy() if hasattr(got, "cpu") else got
        assert_close(got, ref[b:b + chunk], tol, f"{what} rows {b}..")


def mat(g):
    return sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)


@pytest.fixture(scope="module")
def rmat20():
    return synth.rmat_skew(20, seed=0)


@pytest.fixture(scope="module")
def control(rmat20):
    return synth.uniform_control(rmat20, seed=0)


def check_spmm(g, F, transpose=False, seed=0):
    A = mat(g)
    src = g.n_rows if transpose else g.n_cols
    X = synth.normal(src, F, seed, synth.STREAM_X)
    plan = sga.autosage_plan(A, sga.OP_SPMM_T if transpose else sga.OP_SPMM, F, flags=FLAGS)
    Y = sga.autosage_spmm(A, torch.from_numpy(X).cuda(), transpose=transpose, plan=plan)
    if transpose:
        rpt, cit, vt = oracle.transpose(g.row_ptr, g.col_idx, g.vals, g.n_cols)
        ref = oracle.spmm(rpt, cit, vt, X)
    else:
        ref = oracle.spmm(g.row_ptr, g.col_idx, g.vals, X)
    assert_close_rows(Y, ref, TOL_F32, f"spmm F={F} T={transpose} [{plan.describe()}]")


def check_sddmm(g, F, seed=0):
    A = mat(g)
    Q = synth.normal(g.n_rows, F, seed, synth.STREAM_Q)
    K = synth.normal(g.n_cols, F, seed, synth.STREAM_K)
    plan = sga.autosage_plan(A, sga.OP_SDDMM, F, flags=FLAGS)
    S = sga.autosage_sddmm(A, torch.from_numpy(Q).cuda(), torch.from_numpy(K).cuda(), 1.0, plan=plan)
    ref = oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 1.0)[:, 0]
    assert_close_rows(S, ref, TOL_F32, f"sddmm F={F} [{plan.describe()}]", chunk=1 << 24)


@pytest.mark.parametrize("F", [4, 16, 64, 256])
def test_rmat20_spmm(rmat20, F):
    check_spmm(rmat20, F)


@pytest.mark.parametrize("F", [4, 64, 256])
def test_rmat20_sddmm(rmat20, F):
    check_sddmm(rmat20, F)


@pytest.mark.parametrize("F", [8, 128])
def test_control_spmm_sddmm(control, F):
    check_spmm(control, F)
    check_sddmm(control, F)


def test_rmat20_spmm_transpose(rmat20):
    check_spmm(rmat20, 64, transpose=True)


@pytest.mark.parametrize("fused", [True, False])
def test_rmat20_attention_bf16(rmat20, fused):
    g = rmat20
    A = mat(g)
    H, D = 8, 64
    Qb, Q32 = bf16_tensor(synth.normal(g.n_rows, H * D, 0, synth.STREAM_Q))
    Kb, K32 = bf16_tensor(synth.normal(g.n_cols, H * D, 0, synth.STREAM_K))
    Vb, V32 = bf16_tensor(synth.normal(g.n_cols, H * D, 0, synth.STREAM_V))
    plan = sga.autosage_plan(A, sga.OP_ATTN if fused else sga.OP_ATTN_UNFUSED, D, heads=H,
                             dtype=torch.bfloat16, flags=FLAGS)
    O = sga.autosage_csr_attention(A, Qb, Kb, Vb, H, 0.125, fused=fused, plan=plan)
    ref = oracle.csr_attention(g.row_ptr, g.col_idx, Q32, K32, V32, H, 0.125)
    assert_close_rows(O, ref, TOL_BF16, f"attention fused={fused} [{plan.describe()}]")


def test_rmat20_attention_backward_bf16(rmat20):
    # the backward in the benchmark's configuration (bf16, H = 8, D = 64,
    # default backward plan). dQ of a row depends on that row's edges only,
    # so the oracle runs on the sub-graph of sampled rows (columns renumbered
    # to the ones they touch); dK and dV are checked at full size through two
    # identities of the chain rule: sum_j dV_j = sum of dO over non-empty rows
    # (each row's weights sum to 1) and sum_j dK_j = 0 (each row's score
    # gradients sum to 0).
    g = rmat20
    A = mat(g)
    H, D = 8, 64
    W = H * D
    Qb, Q32 = bf16_tensor(synth.normal(g.n_rows, W, 11, synth.STREAM_Q))
    Kb, K32 = bf16_tensor(synth.normal(g.n_cols, W, 11, synth.STREAM_K))
    Vb, V32 = bf16_tensor(synth.normal(g.n_cols, W, 11, synth.STREAM_V))
    Gb, G32 = bf16_tensor(synth.normal(g.n_rows, W, 11, synth.STREAM_G))
    plan = sga.autosage_plan(A, sga.OP_ATTN_BACKWARD, D, heads=H, dtype=torch.bfloat16)
    dQ, dK, dV = sga.autosage_csr_attention_backward(A, Qb, Kb, Vb, Gb, H, 0.125, plan=plan)
    torch.cuda.synchronize()

    deg_all = g.degrees()
    cut = np.flatnonzero(deg_all > 512)  # the rows the backward plan cuts into chunks
    longest = cut[deg_all[cut] > 2048]
    other_cut = cut[deg_all[cut] <= 2048]
    short = np.flatnonzero(deg_all <= 512)
    rows = np.unique(np.concatenate([longest, other_cut[::16], short[::500], [0, g.n_rows - 1]]))
    deg = (g.row_ptr[rows + 1] - g.row_ptr[rows]).astype(np.int64)
    sub_ptr = np.zeros(rows.size + 1, np.int32)
    np.cumsum(deg, out=sub_ptr[1:])
    cols = np.concatenate([g.col_idx[g.row_ptr[r]:g.row_ptr[r + 1]] for r in rows])
    used, sub_cols = np.unique(cols, return_inverse=True)
    rQ, _, _ = oracle.csr_attention_backward(sub_ptr, sub_cols.astype(np.int32), Q32[rows], K32[used],
                                             V32[used], G32[rows], H, 0.125)
    got = dQ[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert_close(got, rQ, TOL_BF16, f"backward dQ [{plan.describe()}]")

    nonempty = np.diff(g.row_ptr) > 0
    want_dv = G32.astype(np.float64)[nonempty].sum(0)
    dv_sum = dV.double().sum(0).cpu().numpy()
    dk_sum = dK.double().sum(0).cpu().numpy()
    # bf16 outputs carry at most 2^-9 relative rounding each
    tol_dv = 4e-3 * dV.double().abs().sum(0).cpu().numpy() + 1e-3
    tol_dk = 4e-3 * dK.double().abs().sum(0).cpu().numpy() + 1e-3
    assert np.all(np.abs(dv_sum - want_dv) <= tol_dv), "sum of dV != sum of dO over non-empty rows"
    assert np.all(np.abs(dk_sum) <= tol_dk), "sum of dK != 0"


@pytest.fixture(scope="module")
def products():
    return synth.products_like(seed=0)


@pytest.mark.parametrize("F", [32, 100])
def test_products_spmm_forward_and_transpose(products, F):
    check_spmm(products, F)
    check_spmm(products, F, transpose=True, seed=1)


@pytest.fixture(scope="module")
def reddit():
    return synth.reddit_like(seed=0)


@pytest.mark.parametrize("F", [128, 602])
def test_reddit_spmm(reddit, F):
    check_spmm(reddit, F)


def test_reddit_sddmm(reddit):
    check_sddmm(reddit, 128)
