"""A planned call computes on the A it is given.

A plan is built from A's structure (row_ptr, col_idx): its chunk lists, row
order, merge-path partitions and A^T come from it. The edge values are not
part of the plan: every call reads the values it is passed, which is the
normal case of a GNN whose edge weights change per layer or step. These
tests build a plan on A and then:
  - call it with new edge values (a new allocation, and the same allocation
    overwritten in place) and compare with the oracle on those values;
  - call it with a copy of the structure in new device memory: refused with
    ERR_PLAN_MISMATCH until autosage_plan_rebind accepts the copy (same
    fingerprint), after which results match the oracle;
  - rebind to a different graph of the same size: refused.
Covers SpMM (every schedule family), SpMM with A^T, SDDMM, fused and unfused
attention, the attention backward and the typed SpMM.
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.fixture(scope="module")
def graphs():
    g = synth.rmat_skew(12, seed=21)
    g = g.with_vals(synth.uniform_vals(g, 21))
    v2 = synth.uniform_vals(g, 22)
    # same sizes, another structure: the rows of g in reverse order
    deg = np.diff(g.row_ptr)[::-1]
    rp = np.zeros_like(g.row_ptr)
    np.cumsum(deg, out=rp[1:])
    ci = np.concatenate([g.col_idx[g.row_ptr[r]:g.row_ptr[r + 1]] for r in range(g.n_rows - 1, -1, -1)])
    other = synth.Csr(g.n_rows, g.n_cols, rp.astype(np.int32), ci.astype(np.int32), g.vals)
    assert not np.array_equal(other.row_ptr, g.row_ptr)
    return g, v2, other


def copy_of(A: sga.CsrMatrix, vals=None):
    """The same structure in new device memory (and optionally other values)."""
    v = A.vals.clone() if vals is None else vals
    return sga.CsrMatrix(A.row_ptr.clone(), A.col_idx.clone(), v, A.n_cols)


SCHEDS = [
    ("rowgroup", sga.SCHED_ROWGROUP, 0),
    ("split", sga.SCHED_SPLIT, 64),
    ("binned", sga.SCHED_BINNED, 32),
    ("mergepath", sga.SCHED_MERGEPATH, 64),
]


@pytest.mark.parametrize("name,kind,split", SCHEDS, ids=[s[0] for s in SCHEDS])
def test_spmm_plan_reads_the_calls_values_and_structure(graphs, name, kind, split):
    g, v2, other = graphs
    F = 24
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    X = synth.normal(g.n_cols, F, 3, synth.STREAM_X)
    plan = sga.autosage_plan_with_schedule(A, sga.OP_SPMM, F, kind, split=split)
    want1 = oracle.spmm(g.row_ptr, g.col_idx, g.vals, X)
    want2 = oracle.spmm(g.row_ptr, g.col_idx, v2, X)
    assert_close(to_np(sga.autosage_spmm(A, dev(X), plan=plan)), want1, TOL_F32, f"{name}: plan-time values")
    # new values in a new allocation, same structure arrays
    A2 = sga.CsrMatrix(A.row_ptr, A.col_idx, dev(v2), A.n_cols)
    assert_close(to_np(sga.autosage_spmm(A2, dev(X), plan=plan)), want2, TOL_F32, f"{name}: new value array")
    # the plan-time value array overwritten in place
    A.vals.copy_(dev(v2))
    assert_close(to_np(sga.autosage_spmm(A, dev(X), plan=plan)), want2, TOL_F32, f"{name}: values in place")
    # a copy of the structure: refused until rebound
    A3 = copy_of(A)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm(A3, dev(X), plan=plan)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
    del A  # the plan-time arrays may go away once the plan is rebound
    plan.rebind(A3)
    assert_close(to_np(sga.autosage_spmm(A3, dev(X), plan=plan)), want2, TOL_F32, f"{name}: rebound copy")
    # a different graph of the same size is refused, and the plan stays bound to A3
    B = sga.CsrMatrix.from_numpy(other.row_ptr, other.col_idx, other.vals, other.n_cols)
    with pytest.raises(sga.AutosageError) as e:
        plan.rebind(B)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm(B, dev(X), plan=plan)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
    assert_close(to_np(sga.autosage_spmm(A3, dev(X), plan=plan)), want2, TOL_F32, f"{name}: still bound")


def test_spmm_transpose_plan_gathers_the_calls_values(graphs):
    g, v2, other = graphs
    F = 16
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    G = synth.normal(g.n_rows, F, 4, synth.STREAM_G)
    plan = sga.autosage_plan(A, sga.OP_SPMM_T, F, flags=sga.PLAN_NO_CACHE)
    want1 = oracle.spmm_t(g.row_ptr, g.col_idx, g.vals, G, g.n_cols)
    want2 = oracle.spmm_t(g.row_ptr, g.col_idx, v2, G, g.n_cols)
    assert_close(to_np(sga.autosage_spmm(A, dev(G), transpose=True, plan=plan)), want1, TOL_F32, "A^T values 1")
    A2 = sga.CsrMatrix(A.row_ptr, A.col_idx, dev(v2), A.n_cols)
    assert_close(to_np(sga.autosage_spmm(A2, dev(G), transpose=True, plan=plan)), want2, TOL_F32, "A^T values 2")
    A0 = sga.CsrMatrix(A.row_ptr, A.col_idx, None, A.n_cols)  # no values: every edge 1
    want0 = oracle.spmm_t(g.row_ptr, g.col_idx, None, G, g.n_cols)
    assert_close(to_np(sga.autosage_spmm(A0, dev(G), transpose=True, plan=plan)), want0, TOL_F32, "A^T ones")
    A3 = copy_of(A2)
    with pytest.raises(sga.AutosageError):
        sga.autosage_spmm(A3, dev(G), transpose=True, plan=plan)
    plan.rebind(A3)
    assert_close(to_np(sga.autosage_spmm(A3, dev(G), transpose=True, plan=plan)), want2, TOL_F32, "A^T rebound")


def test_sddmm_and_attention_plans_follow_a_rebound_copy(graphs):
    g, _, other = graphs
    F, H = 16, 2
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    Q = synth.normal(g.n_rows, F * H, 5, synth.STREAM_Q)
    K = synth.normal(g.n_cols, F * H, 5, synth.STREAM_K)
    V = synth.normal(g.n_cols, F * H, 5, synth.STREAM_V)
    sp = sga.autosage_plan_with_schedule(A, sga.OP_SDDMM, F * H, sga.SCHED_SPLIT, split=64)
    fp = sga.autosage_plan_with_schedule(A, sga.OP_ATTN, F, sga.SCHED_BINNED, split=32, heads=H)
    up = sga.autosage_plan_with_schedule(A, sga.OP_ATTN_UNFUSED, F, sga.SCHED_SPLIT, split=64, heads=H)
    A3 = copy_of(A)
    for p in (sp, fp, up):
        with pytest.raises(sga.AutosageError) as e:
            if p is sp:
                sga.autosage_sddmm(A3, dev(Q), dev(K), 0.5, plan=p)
            else:
                sga.autosage_csr_attention(A3, dev(Q), dev(K), dev(V), H, 0.25, fused=p is fp, plan=p)
        assert e.value.status == sga.ERR_PLAN_MISMATCH
        p.rebind(A3)
    del A
    S = sga.autosage_sddmm(A3, dev(Q), dev(K), 0.5, plan=sp)
    assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 0.5)[:, 0], TOL_F32, "sddmm rebound")
    want = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, H, 0.25)
    for p, fused in ((fp, True), (up, False)):
        O = sga.autosage_csr_attention(A3, dev(Q), dev(K), dev(V), H, 0.25, fused=fused, plan=p)
        assert_close(to_np(O), want, TOL_F32, f"attention fused={fused} rebound")
    B = sga.CsrMatrix.from_numpy(other.row_ptr, other.col_idx, other.vals, other.n_cols)
    for p in (sp, fp, up):
        with pytest.raises(sga.AutosageError) as e:
            p.rebind(B)
        assert e.value.status == sga.ERR_PLAN_MISMATCH


def test_backward_plan_follows_a_rebound_copy(graphs):
    g, _, _ = graphs
    H, D = 2, 8
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    x = {st: synth.normal(g.n_rows, H * D, 6, st) for st in
         (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_G)}
    plan = sga.autosage_plan(A, sga.OP_ATTN_BACKWARD, D, heads=H)
    A3 = copy_of(A)
    args = [dev(x[st]) for st in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_G)]
    with pytest.raises(sga.AutosageError):
        sga.autosage_csr_attention_backward(A3, *args, H, 0.3, plan=plan)
    plan.rebind(A3)
    del A
    got = sga.autosage_csr_attention_backward(A3, *args, H, 0.3, plan=plan)
    want = oracle.csr_attention_backward(g.row_ptr, g.col_idx, x[synth.STREAM_Q], x[synth.STREAM_K],
                                         x[synth.STREAM_V], x[synth.STREAM_G], H, 0.3)
    for name, a, b in zip(("dQ", "dK", "dV"), got, want):
        assert_close(to_np(a), b, TOL_F32, f"backward {name} rebound")


def test_typed_plan_reads_the_calls_values_and_checks_its_arrays(graphs):
    g, v2, _ = graphs
    R, F = 3, 8
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    etype = synth.rng_for(7, 9).integers(0, R, g.nnz).astype(np.int32)
    et = dev(etype)
    Z = synth.normal(R * g.n_cols, F, 7, synth.STREAM_X).reshape(R, g.n_cols, F)
    plan = sga.autosage_plan_typed(A, et, R, F, flags=sga.PLAN_NO_CACHE)
    A2 = sga.CsrMatrix(A.row_ptr, A.col_idx, dev(v2), A.n_cols)
    Y = sga.autosage_spmm_typed(A2, et, dev(Z), plan=plan)
    assert_close(to_np(Y), oracle.spmm_typed(g.row_ptr, g.col_idx, etype, v2, Z), TOL_F32, "typed, new values")
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm_typed(A2, et.clone(), dev(Z), plan=plan)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
    with pytest.raises(sga.AutosageError) as e:
        plan.rebind(copy_of(A2))
    assert e.value.status == sga.ERR_UNSUPPORTED


def test_fixed_values_plan_keeps_its_values_and_checks_the_array(graphs):
    # AUTOSAGE_PLAN_FIXED_VALUES: SpMM with A^T gathers the values into A^T's
    # edge order once; a call must pass the same value array, and rebinding
    # takes the new array's values
    g, v2, _ = graphs
    F = 8
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    G = synth.normal(g.n_rows, F, 8, synth.STREAM_G)
    plan = sga.autosage_plan(A, sga.OP_SPMM_T, F, flags=sga.PLAN_NO_CACHE | sga.PLAN_FIXED_VALUES)
    assert "fixed_vals=1" in plan.describe()
    want1 = oracle.spmm_t(g.row_ptr, g.col_idx, g.vals, G, g.n_cols)
    for _ in range(2):
        assert_close(to_np(sga.autosage_spmm(A, dev(G), transpose=True, plan=plan)), want1, TOL_F32, "fixed values")
    A2 = sga.CsrMatrix(A.row_ptr, A.col_idx, dev(v2), A.n_cols)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm(A2, dev(G), transpose=True, plan=plan)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
    plan.rebind(A2)
    want2 = oracle.spmm_t(g.row_ptr, g.col_idx, v2, G, g.n_cols)
    assert_close(to_np(sga.autosage_spmm(A2, dev(G), transpose=True, plan=plan)), want2, TOL_F32, "refixed values")
    # forward ops read the values from the call's array (the same array here)
    fplan = sga.autosage_plan(A2, sga.OP_SPMM, F, flags=sga.PLAN_NO_CACHE | sga.PLAN_FIXED_VALUES)
    X = synth.normal(g.n_cols, F, 8, synth.STREAM_X)
    assert_close(to_np(sga.autosage_spmm(A2, dev(X), plan=fplan)), oracle.spmm(g.row_ptr, g.col_idx, v2, X),
                 TOL_F32, "forward, fixed values")
