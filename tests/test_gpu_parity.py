"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every test is marked gpu. Inputs come from synth (seeded), expected values
from oracle (fp64). fp32 paths: |gpu - oracle| <= 1e-4 * (1 + |oracle|);
bf16 feature paths: 2e-2 relative; integer/index results bit-exact;
repeated runs of one plan bitwise identical.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_BF16, TOL_F32, assert_close, bf16_tensor, csr_from_lists, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def mat(g: synth.Csr) -> sga.CsrMatrix:
    return sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)


SCHEDULES = [
    ("default", None),
    ("rowgroup-e1", dict(kind=sga.SCHED_ROWGROUP, lanes_e=1)),
    ("rowgroup-e4", dict(kind=sga.SCHED_ROWGROUP, lanes_e=4)),
    ("split-8", dict(kind=sga.SCHED_SPLIT, split=8)),
    ("split-64-e2", dict(kind=sga.SCHED_SPLIT, split=64, lanes_e=2)),
    ("binned-32", dict(kind=sga.SCHED_BINNED, split=32)),
]
SPMM_SCHEDULES = SCHEDULES + [
    ("mergepath-32", dict(kind=sga.SCHED_MERGEPATH, split=32)),
    ("mergepath-300", dict(kind=sga.SCHED_MERGEPATH, split=300)),
    ("hybrid-32", dict(kind=sga.SCHED_HYBRID, split=32)),
    ("hybrid-512-e4", dict(kind=sga.SCHED_HYBRID, split=512, lanes_e=4)),
]


def make_plan(A, op, F, spec, heads=1, dtype=torch.float32):
    if spec is None:
        return None
    spec = dict(spec)
    kind = spec.pop("kind")
    return sga.autosage_plan_with_schedule(A, op, F, kind, heads=heads, dtype=dtype, **spec)


@pytest.fixture(scope="module")
def tiny():
    g = synth.tiny_er(0)
    F = 32
    X = synth.normal(g.n_cols, F, 0, synth.STREAM_X)
    Q = synth.normal(g.n_rows, F, 0, synth.STREAM_Q)
    K = synth.normal(g.n_cols, F, 0, synth.STREAM_K)
    V = synth.normal(g.n_cols, F, 0, synth.STREAM_V)
    return g, X, Q, K, V


@pytest.fixture(scope="module")
def skew():
    """R-MAT scale 13: several tiles, hubs longer than the split sizes, ragged tails."""
    g = synth.rmat_skew(13, seed=3)
    return g


# ---------------------------------------------------------------- SpMM

@pytest.mark.parametrize("name,spec", SPMM_SCHEDULES, ids=[s[0] for s in SPMM_SCHEDULES])
def test_spmm_tiny_er(tiny, name, spec):
    g, X, *_ = tiny
    A = mat(g)
    plan = make_plan(A, sga.OP_SPMM, 32, spec)
    Y = sga.autosage_spmm(A, dev(X), plan=plan)
    assert_close(to_np(Y), oracle.spmm(g.row_ptr, g.col_idx, g.vals, X), TOL_F32, f"spmm {name}")


@pytest.mark.parametrize("F", [1, 2, 3, 4, 5, 8, 16, 33, 64, 100, 128, 256, 602])
@pytest.mark.parametrize("name,spec", SPMM_SCHEDULES, ids=[s[0] for s in SPMM_SCHEDULES])
def test_spmm_width_sweep_skewed(skew, F, name, spec):
    g = skew
    A = mat(g)
    X = synth.normal(g.n_cols, F, 1, synth.STREAM_X)
    plan = make_plan(A, sga.OP_SPMM, F, spec)
    Y = sga.autosage_spmm(A, dev(X), plan=plan)
    assert_close(to_np(Y), oracle.spmm(g.row_ptr, g.col_idx, g.vals, X), TOL_F32, f"spmm F={F} {name}")


def test_spmm_leading_dims_and_bf16(skew):
    g = skew
    A = mat(g)
    big = synth.normal(g.n_cols, 70, 2, synth.STREAM_X)
    Xd = dev(big)[:, 3:67]  # ld 70, offset 3 floats: only 4-byte alignment
    Yfull = torch.full((g.n_rows, 80), 7.0, device="cuda")
    Y = Yfull[:, 5:69]
    sga.autosage_spmm(A, Xd, Y)
    assert_close(to_np(Y), oracle.spmm(g.row_ptr, g.col_idx, g.vals, big[:, 3:67]), TOL_F32, "spmm ld")
    assert torch.all(Yfull[:, :5] == 7.0) and torch.all(Yfull[:, 69:] == 7.0), "wrote outside Y"
    Xb, Xb32 = bf16_tensor(synth.normal(g.n_cols, 64, 3, synth.STREAM_X))
    Yb = sga.autosage_spmm(A, Xb)
    assert Yb.dtype == torch.bfloat16
    assert_close(to_np(Yb), oracle.spmm(g.row_ptr, g.col_idx, g.vals, Xb32), TOL_BF16, "spmm bf16")


def test_spmm_no_values_means_ones(skew):
    g = skew.with_vals(None)
    A = mat(g)
    X = synth.normal(g.n_cols, 16, 4, synth.STREAM_X)
    assert_close(to_np(sga.autosage_spmm(A, dev(X))), oracle.spmm(g.row_ptr, g.col_idx, None, X), TOL_F32)


@pytest.mark.parametrize("items", [32, 300])
@pytest.mark.parametrize("bf16", [False, True])
def test_spmm_mergepath_cut_row_rounded_once(items, bf16):
    # One hub row cut by the merge path into many warps' segments: its first
    # 1501 edges have value +1 and its last 1500 value -1 over identical X
    # rows, so every warp's segment sums to hundreds of X rows while the row's
    # exact result is one X row. The segments must be added in fp32 and the
    # row rounded to the output type once; rounding the finishing segment to
    # bf16 first would be off by up to (its length) * 2^-9.
    k = 1500
    n = 2 * k + 1
    cols = np.arange(n, dtype=np.int32)
    vals = np.concatenate([np.ones(k + 1), -np.ones(k)]).astype(np.float32)
    row_ptr = np.array([0, n] + [n + i + 1 for i in range(n - 1)], dtype=np.int32)  # then one edge per row
    col_idx = np.concatenate([cols, (np.arange(n - 1, dtype=np.int32) * 7) % n]).astype(np.int32)
    vals = np.concatenate([vals, np.full(n - 1, 0.5, np.float32)])
    g = synth.Csr(n, n, row_ptr, col_idx, vals)
    F = 8
    base = synth.normal(1, F, 17, synth.STREAM_X) * 3.0
    X32 = np.repeat(base, n, axis=0)
    if bf16:
        Xd, X32 = bf16_tensor(X32)
    else:
        Xd = dev(X32)
    A = mat(g)
    plan = make_plan(A, sga.OP_SPMM, F, dict(kind=sga.SCHED_MERGEPATH, split=items),
                     dtype=torch.bfloat16 if bf16 else torch.float32)
    Y = sga.autosage_spmm(A, Xd, plan=plan)
    want = oracle.spmm(g.row_ptr, g.col_idx, g.vals, X32)
    assert_close(to_np(Y), want, TOL_BF16 if bf16 else TOL_F32, f"merge path items={items} bf16={bf16}")
    assert "sched=mergepath" in plan.describe()


@pytest.mark.parametrize("name,spec", SPMM_SCHEDULES, ids=[s[0] for s in SPMM_SCHEDULES])
def test_spmm_transpose(skew, name, spec):
    g = skew
    A = mat(g)
    spec = spec or dict(kind=sga.SCHED_ROWGROUP)
    plan = make_plan(A, sga.OP_SPMM_T, 24, spec)
    G = synth.normal(g.n_rows, 24, 5, synth.STREAM_G)
    GX = sga.autosage_spmm(A, dev(G), transpose=True, plan=plan)
    assert_close(to_np(GX), oracle.spmm_t(g.row_ptr, g.col_idx, g.vals, G, g.n_cols), TOL_F32, f"spmm^T {name}")


# ---------------------------------------------------------------- SDDMM

@pytest.mark.parametrize("name,spec", SCHEDULES + [("mergepath-64", dict(kind=sga.SCHED_MERGEPATH, split=64))],
                         ids=[s[0] for s in SCHEDULES] + ["mergepath-64"])
def test_sddmm_tiny_er(tiny, name, spec):
    g, _, Q, K, _ = tiny
    A = mat(g)
    plan = make_plan(A, sga.OP_SDDMM, 32, spec)
    S = sga.autosage_sddmm(A, dev(Q), dev(K), 1.0, plan=plan)
    assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 1.0)[:, 0], TOL_F32, f"sddmm {name}")


# merge path for SDDMM: lane groups of any shape walk equal shares of (rows + edges)
SDDMM_SCHEDULES = SCHEDULES + [
    ("mergepath-32", dict(kind=sga.SCHED_MERGEPATH, split=32)),
    ("mergepath-300-e2", dict(kind=sga.SCHED_MERGEPATH, split=300, lanes_e=2)),
    ("mergepath-1024-pe", dict(kind=sga.SCHED_MERGEPATH, split=1024, per_edge=1)),
]


@pytest.mark.parametrize("F", [1, 3, 4, 8, 16, 32, 64, 100, 128, 256])
@pytest.mark.parametrize("name,spec", SDDMM_SCHEDULES, ids=[s[0] for s in SDDMM_SCHEDULES])
def test_sddmm_width_sweep_skewed(skew, F, name, spec):
    g = skew
    A = mat(g)
    Q = synth.normal(g.n_rows, F, 6, synth.STREAM_Q)
    K = synth.normal(g.n_cols, F, 6, synth.STREAM_K)
    plan = make_plan(A, sga.OP_SDDMM, F, spec)
    S = sga.autosage_sddmm(A, dev(Q), dev(K), 0.5, plan=plan)
    assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 0.5)[:, 0], TOL_F32, f"sddmm F={F} {name}")


PER_EDGE = [
    ("rowgroup-g4", dict(kind=sga.SCHED_ROWGROUP, lanes_f=4, lanes_e=1, per_edge=1)),
    ("rowgroup-g8-e2", dict(kind=sga.SCHED_ROWGROUP, lanes_f=8, lanes_e=2, per_edge=1)),
    ("binned-g16", dict(kind=sga.SCHED_BINNED, lanes_f=16, split=32, per_edge=1)),
    ("split-g4-e4", dict(kind=sga.SCHED_SPLIT, lanes_f=4, lanes_e=4, split=16, per_edge=1)),
]


@pytest.mark.parametrize("F", [16, 20, 64, 100, 256])
@pytest.mark.parametrize("name,spec", PER_EDGE, ids=[s[0] for s in PER_EDGE])
def test_sddmm_per_edge_reduction(skew, F, name, spec):
    # single-head SDDMM with one shuffle reduction per edge instead of batched
    # transpose-reductions (a planner variant); same results within tolerance
    g = skew
    A = mat(g)
    Q = synth.normal(g.n_rows, F, 12, synth.STREAM_Q)
    K = synth.normal(g.n_cols, F, 12, synth.STREAM_K)
    plan = make_plan(A, sga.OP_SDDMM, F, spec)
    assert plan.schedule()["per_edge"] == 1 and "per_edge=1" in plan.describe()
    S = sga.autosage_sddmm(A, dev(Q), dev(K), 0.25, plan=plan)
    assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 0.25)[:, 0], TOL_F32, f"sddmm F={F} {name}")


def test_sddmm_bf16(skew):
    g = skew
    A = mat(g)
    Qb, Q32 = bf16_tensor(synth.normal(g.n_rows, 64, 7, synth.STREAM_Q))
    Kb, K32 = bf16_tensor(synth.normal(g.n_cols, 64, 7, synth.STREAM_K))
    S = sga.autosage_sddmm(A, Qb, Kb, 0.125)
    assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q32, K32, 0.125)[:, 0], TOL_F32, "sddmm bf16")


# ---------------------------------------------------------------- softmax

@pytest.mark.parametrize("heads", [1, 2, 3, 8])
@pytest.mark.parametrize("name,spec", SCHEDULES[:1] + SCHEDULES[3:4] + SCHEDULES[5:6], ids=["default", "split-8", "binned-32"])
def test_row_softmax(skew, heads, name, spec):
    g = skew
    A = mat(g)
    S = synth.normal(g.nnz, heads, 8, synth.STREAM_Q) * 4
    plan = make_plan(A, sga.OP_SOFTMAX, 1, spec, heads=heads)
    W = sga.autosage_row_softmax(A, dev(S), heads, plan=plan)
    assert_close(to_np(W), oracle.row_softmax(g.row_ptr, S.astype(np.float64)), TOL_F32, f"softmax H={heads}")


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name,spec", SCHEDULES, ids=[s[0] for s in SCHEDULES])
def test_attention_tiny_er(tiny, fused, name, spec):
    g, _, Q, K, V = tiny
    A = mat(g)
    op = sga.OP_ATTN if fused else sga.OP_ATTN_UNFUSED
    plan = make_plan(A, op, 32, spec)
    scale = 1.0 / np.sqrt(32.0)
    O = sga.autosage_csr_attention(A, dev(Q), dev(K), dev(V), 1, scale, fused=fused, plan=plan)
    ref = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, 1, scale)
    assert_close(to_np(O), ref, TOL_F32, f"attention fused={fused} {name}")


@pytest.mark.parametrize("heads,D", [(2, 16), (4, 8), (8, 64), (3, 32), (2, 12)])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name,spec", SCHEDULES[:1] + SCHEDULES[3:6], ids=["default", "split-8", "split-64-e2", "binned-32"])
def test_attention_multihead_skewed(skew, heads, D, fused, name, spec):
    g = skew
    A = mat(g)
    W = heads * D
    Q = synth.normal(g.n_rows, W, 9, synth.STREAM_Q)
    K = synth.normal(g.n_cols, W, 9, synth.STREAM_K)
    V = synth.normal(g.n_cols, W, 9, synth.STREAM_V)
    op = sga.OP_ATTN if fused else sga.OP_ATTN_UNFUSED
    plan = make_plan(A, op, D, spec, heads=heads)
    O = sga.autosage_csr_attention(A, dev(Q), dev(K), dev(V), heads, 1 / np.sqrt(D), fused=fused, plan=plan)
    ref = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, heads, 1 / np.sqrt(D))
    assert_close(to_np(O), ref, TOL_F32, f"attention H={heads} D={D} fused={fused} {name}")


@pytest.mark.parametrize("fused", [True, False])
def test_attention_bf16_multihead(skew, fused):
    g = skew
    A = mat(g)
    H, D = 8, 64
    Qb, Q32 = bf16_tensor(synth.normal(g.n_rows, H * D, 10, synth.STREAM_Q))
    Kb, K32 = bf16_tensor(synth.normal(g.n_cols, H * D, 10, synth.STREAM_K))
    Vb, V32 = bf16_tensor(synth.normal(g.n_cols, H * D, 10, synth.STREAM_V))
    plan = sga.autosage_plan(A, sga.OP_ATTN if fused else sga.OP_ATTN_UNFUSED, D, heads=H,
                             dtype=torch.bfloat16, flags=sga.PLAN_NO_CACHE)
    O = sga.autosage_csr_attention(A, Qb, Kb, Vb, H, 0.125, fused=fused, plan=plan)
    assert O.dtype == torch.bfloat16
    ref = oracle.csr_attention(g.row_ptr, g.col_idx, Q32, K32, V32, H, 0.125)
    assert_close(to_np(O), ref, TOL_BF16, f"attention bf16 fused={fused}")


# the aggregation stage of unfused attention with its own feature lanes
# (fewer, more, or the same as the score stage), fp32 and bf16
@pytest.mark.parametrize("kind,G,E,split,agg", [
    (sga.SCHED_BINNED, 16, 1, 512, 32), (sga.SCHED_BINNED, 16, 1, 32, 8), (sga.SCHED_ROWGROUP, 8, 2, 0, 16),
    (sga.SCHED_SPLIT, 16, 2, 16, 8), (sga.SCHED_ROWGROUP, 32, 1, 0, 32),
], ids=["binned-16-agg32", "binned-16-agg8", "rowgroup-8x2-agg16", "split-16x2-agg8", "rowgroup-32-agg32"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_unfused_attention_aggregation_lanes(skew, kind, G, E, split, agg, dtype):
    g = skew
    A = mat(g)
    H, D = 8, 64
    Q = synth.normal(g.n_rows, H * D, 12, synth.STREAM_Q)
    K = synth.normal(g.n_cols, H * D, 12, synth.STREAM_K)
    V = synth.normal(g.n_cols, H * D, 12, synth.STREAM_V)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    if dtype == "bf16":
        (Qd, Q), (Kd, K), (Vd, V) = bf16_tensor(Q), bf16_tensor(K), bf16_tensor(V)
    else:
        Qd, Kd, Vd = dev(Q), dev(K), dev(V)
    plan = sga.autosage_plan_with_schedule(A, sga.OP_ATTN_UNFUSED, D, kind, lanes_f=G, lanes_e=E, split=split,
                                           heads=H, dtype=tdt, lanes_f_agg=agg)
    want = 0 if agg == G else agg
    assert plan.schedule()["lanes_f_agg"] == want and f"agg_lanes={want}" in plan.describe()
    O = sga.autosage_csr_attention(A, Qd, Kd, Vd, H, 0.125, fused=False, plan=plan)
    ref = oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, H, 0.125)
    assert_close(to_np(O), ref, TOL_BF16 if dtype == "bf16" else TOL_F32, f"unfused agg lanes {agg} {dtype}")


def test_edge_softmax_aggregate_benchmark_shape():
    g = synth.attention_benchmark_shape(0)
    A = mat(g)
    scores = synth.normal(g.nnz, 1, 0, synth.STREAM_Q)[:, 0]
    V = synth.normal(g.n_cols, 64, 0, synth.STREAM_V)
    out = sga.autosage_edge_softmax_aggregate(A, dev(scores), dev(V))
    ref = oracle.edge_softmax_aggregate(g.row_ptr, g.col_idx, scores, V)
    assert_close(to_np(out), ref, TOL_F32, "edge softmax aggregation")
    # unfused route over the same scores: row softmax, then SpMM with the weights
    W = sga.autosage_row_softmax(A, dev(scores.copy()), 1)
    B = sga.CsrMatrix(A.row_ptr, A.col_idx, W, A.n_cols)
    assert_close(to_np(sga.autosage_spmm(B, dev(V))), ref, TOL_F32, "softmax + spmm")


# ---------------------------------------------------------------- edge cases

def edge_case_graphs():
    n = 37
    out = []
    out.append(("all-empty", synth.Csr(n, n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32),
                                       np.zeros(0, np.float32))))
    out.append(("single-node-self-loop", csr_from_lists([(0, 0)], 1, 1, [0.5])))
    hub = [(5, c) for c in range(n)] * 3  # duplicates allowed: the plain CSR sum
    out.append(("one-hub-with-duplicates", csr_from_lists(hub, n, n, np.linspace(-1, 1, len(hub)))))
    out.append(("self-loops-only", csr_from_lists([(i, i) for i in range(n)], n, n, np.ones(n))))
    out.append(("empty-tail-rows", csr_from_lists([(0, 1), (0, 2), (1, 0)], n, 3, [1.0, 2.0, 3.0])))
    return out


@pytest.mark.parametrize("name,g", edge_case_graphs(), ids=[e[0] for e in edge_case_graphs()])
@pytest.mark.parametrize("sched", ["default", "split", "mergepath", "binned", "hybrid"])
def test_edge_cases(name, g, sched):
    A = mat(g)
    F = 6
    X = synth.normal(g.n_cols, F, 11, synth.STREAM_X)
    Q = synth.normal(g.n_rows, F, 11, synth.STREAM_Q)
    K = synth.normal(g.n_cols, F, 11, synth.STREAM_K)
    spec = {"default": None, "split": dict(kind=sga.SCHED_SPLIT, split=2),
            "mergepath": dict(kind=sga.SCHED_MERGEPATH, split=3), "binned": dict(kind=sga.SCHED_BINNED, split=2),
            "hybrid": dict(kind=sga.SCHED_HYBRID, split=8)}[sched]
    plan = make_plan(A, sga.OP_SPMM, F, spec)
    Y = sga.autosage_spmm(A, dev(X), plan=plan)
    assert_close(to_np(Y), oracle.spmm(g.row_ptr, g.col_idx, g.vals, X), TOL_F32, f"{name} spmm")
    if sched != "hybrid":  # SpMM only
        plan = make_plan(A, sga.OP_SDDMM, F, spec)
        S = sga.autosage_sddmm(A, dev(Q), dev(K), plan=plan)
        assert_close(to_np(S), oracle.sddmm(g.row_ptr, g.col_idx, Q, K)[:, 0], TOL_F32, f"{name} sddmm")
    if sched in ("mergepath", "hybrid"):  # the attention ops take neither family
        return
    for fused in (True, False):
        plan = make_plan(A, sga.OP_ATTN if fused else sga.OP_ATTN_UNFUSED, F, spec)
        O = sga.autosage_csr_attention(A, dev(Q), dev(K), dev(X), 1, 0.7, fused=fused, plan=plan)
        assert_close(to_np(O), oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, X, 1, 0.7), TOL_F32,
                     f"{name} attention fused={fused}")


def test_zero_rows_is_a_no_op():
    g = synth.Csr(0, 0, np.zeros(1, np.int32), np.zeros(0, np.int32), None)
    A = mat(g)
    Y = sga.autosage_spmm(A, torch.zeros((0, 4), device="cuda"))
    assert Y.shape == (0, 4)


def test_argument_errors_are_reported_before_launch(tiny):
    g, X, *_ = tiny
    A = mat(g)
    Xd = dev(X)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm(A, Xd, torch.empty((g.n_rows, 16), device="cuda"))  # ld < F
    assert e.value.status == sga.ERR_INVALID_ARG
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm(A, Xd, transpose=True)  # no A^T plan
    assert e.value.status == sga.ERR_INVALID_ARG
    plan = sga.autosage_plan(A, sga.OP_SDDMM, 32, flags=sga.PLAN_NO_CACHE)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm(A, Xd, plan=plan)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
    bad = g.col_idx.copy()
    bad[10] = g.n_cols + 5
    B = sga.CsrMatrix.from_numpy(g.row_ptr, bad, g.vals, g.n_cols)
    assert sga.autosage_validate_csr(B) == sga.ERR_INVALID_CSR
    assert sga.autosage_validate_csr(A) == sga.OK


# ---------------------------------------------------------------- determinism

@pytest.mark.parametrize("name,spec", SPMM_SCHEDULES[1:], ids=[s[0] for s in SPMM_SCHEDULES[1:]])
def test_repeat_runs_are_bitwise_identical(skew, name, spec):
    g = skew
    A = mat(g)
    X = dev(synth.normal(g.n_cols, 64, 12, synth.STREAM_X))
    plan = make_plan(A, sga.OP_SPMM, 64, spec)
    first = sga.autosage_spmm(A, X, plan=plan).clone()
    for _ in range(3):
        assert torch.equal(sga.autosage_spmm(A, X, plan=plan), first)
    if spec["kind"] not in (sga.SCHED_MERGEPATH, sga.SCHED_HYBRID):  # SpMM-only families
        aplan = make_plan(A, sga.OP_ATTN, 16, spec, heads=4)
        Q = dev(synth.normal(g.n_rows, 64, 12, synth.STREAM_Q))
        o1 = sga.autosage_csr_attention(A, Q, Q, X, 4, 0.25, plan=aplan).clone()
        for _ in range(3):
            assert torch.equal(sga.autosage_csr_attention(A, Q, Q, X, 4, 0.25, plan=aplan), o1)


# ---------------------------------------------------------------- graph utilities

def test_row_stats_fingerprint_transpose_bit_exact(skew):
    g = skew
    A = mat(g)
    ints, reals = sga.autosage_row_stats(A, 100)
    oi, orl = oracle.row_stats(g.row_ptr, 100)
    np.testing.assert_array_equal(ints, oi)
    np.testing.assert_allclose(reals, orl, rtol=1e-12)
    assert sga.autosage_fingerprint(A) == oracle.fingerprint(g.row_ptr, g.col_idx)
    rpt, cit, vt = sga.autosage_csr_transpose(A)
    ort, oct_, ovt = oracle.transpose(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    np.testing.assert_array_equal(rpt.cpu().numpy(), ort)
    np.testing.assert_array_equal(cit.cpu().numpy(), oct_)
    np.testing.assert_array_equal(vt.cpu().numpy(), ovt)


def test_transpose_rectangular_and_duplicates():
    g = csr_from_lists([(0, 4), (0, 4), (2, 1), (2, 4), (3, 0), (3, 0)], 5, 7, [1, 2, 3, 4, 5, 6])
    A = mat(g)
    rpt, cit, vt = sga.autosage_csr_transpose(A)
    ort, oct_, ovt = oracle.transpose(g.row_ptr, g.col_idx, g.vals, 7)
    np.testing.assert_array_equal(rpt.cpu().numpy(), ort)
    np.testing.assert_array_equal(cit.cpu().numpy(), oct_)
    np.testing.assert_array_equal(vt.cpu().numpy(), ovt)


# ---------------------------------------------------------------- planner and cache

def test_plan_probe_cache_replay(tmp_path, skew):
    g = skew
    A = mat(g)
    X = dev(synth.normal(g.n_cols, 32, 13, synth.STREAM_X))
    sga.autosage_cache_clear()
    plan = sga.autosage_plan(A, sga.OP_SPMM, 32, flags=sga.PLAN_PROBE | sga.PLAN_VERIFY)
    first = plan.schedule()
    assert first["probe_ms"] > 0
    Y1 = sga.autosage_spmm(A, X, plan=plan).clone()
    assert_close(to_np(Y1), oracle.spmm(g.row_ptr, g.col_idx, g.vals, X.cpu().numpy()), TOL_F32, "planned spmm")
    path = str(tmp_path / "plans.txt")
    sga.autosage_cache_save(path)
    sga.autosage_cache_clear()
    assert sga.autosage_cache_size() == 0
    sga.autosage_cache_load(path)
    assert sga.autosage_cache_size() >= 1
    replay = sga.autosage_plan(A, sga.OP_SPMM, 32, flags=sga.PLAN_PROBE)
    assert "cache=1" in replay.describe()
    again = replay.schedule()
    for k in ("kind", "lanes_f", "lanes_e", "split"):
        assert again[k] == first[k]
    assert torch.equal(sga.autosage_spmm(A, X, plan=replay), Y1)
