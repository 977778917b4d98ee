"""Randomized GPU parity sweep: seeded random CSR graphs (degree mixes from
empty to hub rows, rectangular shapes, optional duplicates) with random
widths, head counts, dtypes and schedules, every operation against the
oracle through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_BF16, TOL_F32, assert_close, bf16_tensor, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402

KINDS = [sga.SCHED_ROWGROUP, sga.SCHED_SPLIT, sga.SCHED_BINNED, sga.SCHED_MERGEPATH]


def random_graph(rng):
    n = int(rng.integers(1, 400))
    m = int(rng.integers(1, 400))
    kind = rng.integers(0, 3)
    if kind == 0:    # power-law-ish degrees
        deg = np.minimum((rng.pareto(1.2, n) * 3).astype(np.int64), m)
    elif kind == 1:  # mostly empty rows and one hub
        deg = np.where(rng.random(n) < 0.7, 0, np.minimum(rng.integers(0, 4, n), m))
        deg[rng.integers(0, n)] = m
    else:            # uniform
        deg = rng.integers(0, min(m, 30) + 1, n)
    rows = np.repeat(np.arange(n), deg)
    cols = np.concatenate([np.sort(rng.choice(m, size=d, replace=False)) for d in deg]) if deg.sum() else np.zeros(0)
    if rng.random() < 0.3 and cols.size:  # duplicate a few edges (separate CSR terms)
        dup = rng.integers(0, cols.size, max(1, cols.size // 10))
        order = np.argsort(np.concatenate([rows, rows[dup]]), kind="stable")
        rows = np.concatenate([rows, rows[dup]])[order]
        cols = np.concatenate([cols, cols[dup]])[order]
    row_ptr = np.zeros(n + 1, np.int32)
    np.cumsum(np.bincount(rows, minlength=n), out=row_ptr[1:])
    vals = rng.uniform(-1, 1, cols.size).astype(np.float32)
    return synth.Csr(n, m, row_ptr, cols.astype(np.int32), vals)


def plan_for(rng, A, op, F, heads, dtype, allow_mergepath):
    kinds = KINDS if allow_mergepath else KINDS[:3]
    kind = int(rng.choice(kinds))
    lanes_e = int(rng.choice([0, 1, 2, 4]))
    split = int(rng.choice([1, 3, 16, 64]))
    if kind == sga.SCHED_ROWGROUP:
        split = 0
    per_edge = int(op == sga.OP_SDDMM and rng.random() < 0.5)
    return sga.autosage_plan_with_schedule(A, op, F, kind, lanes_e=0 if kind == sga.SCHED_MERGEPATH else lanes_e,
                                           split=split, heads=heads, dtype=dtype, per_edge=per_edge)


@pytest.mark.parametrize("seed", range(24))
def test_random_graphs_all_ops(seed):
    rng = np.random.default_rng(1000 + seed)
    g = random_graph(rng)
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    bf16 = bool(rng.random() < 0.3)
    tol = TOL_BF16 if bf16 else TOL_F32
    dtype = torch.bfloat16 if bf16 else torch.float32

    def feat(rows, width, stream):
        x = synth.normal(rows, width, seed, stream)
        if bf16:
            t, x32 = bf16_tensor(x)
            return t, x32
        return torch.from_numpy(x).cuda(), x

    # SpMM
    F = int(rng.choice([1, 2, 3, 4, 8, 12, 32, 40, 64, 128]))
    X, X32 = feat(g.n_cols, F, synth.STREAM_X)
    plan = plan_for(rng, A, sga.OP_SPMM, F, 1, dtype, True)
    Y = sga.autosage_spmm(A, X, plan=plan)
    assert_close(to_np(Y), oracle.spmm(g.row_ptr, g.col_idx, g.vals, X32), tol, f"spmm F={F} {plan.describe()}")
    # SpMM with A^T
    G, G32 = feat(g.n_rows, F, synth.STREAM_G)
    plan = plan_for(rng, A, sga.OP_SPMM_T, F, 1, dtype, True)
    GX = sga.autosage_spmm(A, G, transpose=True, plan=plan)
    assert_close(to_np(GX), oracle.spmm_t(g.row_ptr, g.col_idx, g.vals, G32, g.n_cols), tol, f"spmm_t {plan.describe()}")
    # SDDMM
    Q, Q32 = feat(g.n_rows, F, synth.STREAM_Q)
    K, K32 = feat(g.n_cols, F, synth.STREAM_K)
    plan = plan_for(rng, A, sga.OP_SDDMM, F, 1, dtype, False)
    S = sga.autosage_sddmm(A, Q, K, 0.3, plan=plan)
    if g.nnz:
        assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q32, K32, 0.3)[:, 0], TOL_F32,
                     f"sddmm {plan.describe()}")
    # attention, fused and unfused, and its backward (K and V have a row per source)
    H = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([4, 8, 16, 32]))
    W = H * D
    Qa, Qa32 = feat(g.n_rows, W, synth.STREAM_Q)
    Ka, Ka32 = feat(g.n_cols, W, synth.STREAM_K)
    Va, Va32 = feat(g.n_cols, W, synth.STREAM_V)
    scale = 1.0 / np.sqrt(D)
    ref = oracle.csr_attention(g.row_ptr, g.col_idx, Qa32, Ka32, Va32, H, scale)
    for fused in (True, False):
        plan = plan_for(rng, A, sga.OP_ATTN if fused else sga.OP_ATTN_UNFUSED, D, H, dtype, False)
        O = sga.autosage_csr_attention(A, Qa, Ka, Va, H, scale, fused=fused, plan=plan)
        assert_close(to_np(O), ref, tol, f"attention fused={fused} H={H} D={D} {plan.describe()}")
    if not bf16:
        dO, dO32 = feat(g.n_rows, W, synth.STREAM_G)
        plan = plan_for(rng, A, sga.OP_ATTN_BACKWARD, D, H, dtype, False)
        grads = sga.autosage_csr_attention_backward(A, Qa, Ka, Va, dO, H, scale, plan=plan)
        refs = oracle.csr_attention_backward(g.row_ptr, g.col_idx, Qa32, Ka32, Va32, dO32, H, scale)
        for name, got, r in zip(("dQ", "dK", "dV"), grads, refs):
            assert_close(to_np(got), r, TOL_F32, f"backward {name} H={H} D={D} {plan.describe()}")
