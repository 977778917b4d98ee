"""GPU parity of the CSR-attention backward (dQ, dK, dV) against the oracle's
chain-rule gradients, through the C ABI."""
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


def mat(g):
    return sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)


def run(g, H, D, scale, seed, use_plan=True, schedule=None):
    A = mat(g)
    W = H * D
    Q, dO = (synth.normal(g.n_rows, W, seed, st) for st in (synth.STREAM_Q, synth.STREAM_G))
    K, V = (synth.normal(g.n_cols, W, seed, st) for st in (synth.STREAM_K, synth.STREAM_V))
    plan = None
    if use_plan:
        if schedule is None:
            plan = sga.autosage_plan(A, sga.OP_ATTN_BACKWARD, D, heads=H)
        else:
            plan = sga.autosage_plan_with_schedule(A, sga.OP_ATTN_BACKWARD, D, heads=H, **schedule)
    d = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    dQ, dK, dV = sga.autosage_csr_attention_backward(A, d(Q), d(K), d(V), d(dO), H, scale, plan=plan)
    rQ, rK, rV = oracle.csr_attention_backward(g.row_ptr, g.col_idx, Q, K, V, dO, H, scale)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        assert_close(to_np(got), ref, TOL_F32, f"{name} H={H} D={D}")


def test_backward_tiny_er():
    run(synth.tiny_er(0), 1, 32, 1 / np.sqrt(32), 0)


@pytest.mark.parametrize("H,D", [(2, 16), (8, 8), (3, 32)])
@pytest.mark.parametrize("schedule", [None, dict(kind=sga.SCHED_ROWGROUP), dict(kind=sga.SCHED_SPLIT, split=16),
                                      dict(kind=sga.SCHED_BINNED, split=16)],
                         ids=["auto", "rowgroup", "split16", "binned16"])
def test_backward_skewed(H, D, schedule):
    run(synth.rmat_skew(13, seed=5), H, D, 1 / np.sqrt(D), 3, schedule=schedule)


def test_backward_without_plan_and_rectangular_with_empty_rows():
    g = csr_from_lists([(0, 1), (0, 4), (2, 4), (2, 0), (5, 3), (5, 4), (5, 1)], 7, 6, None)
    run(g, 2, 8, 0.5, 4, use_plan=False)


def test_backward_bf16_multihead():
    g = synth.rmat_skew(12, seed=2)
    A = mat(g)
    H, D = 8, 64
    W = H * D
    Qb, Q = bf16_tensor(synth.normal(g.n_rows, W, 1, synth.STREAM_Q))
    Kb, K = bf16_tensor(synth.normal(g.n_cols, W, 1, synth.STREAM_K))
    Vb, V = bf16_tensor(synth.normal(g.n_cols, W, 1, synth.STREAM_V))
    dOb, dO = bf16_tensor(synth.normal(g.n_rows, W, 1, synth.STREAM_G))
    plan = sga.autosage_plan(A, sga.OP_ATTN_BACKWARD, D, heads=H, dtype=torch.bfloat16)
    dQ, dK, dV = sga.autosage_csr_attention_backward(A, Qb, Kb, Vb, dOb, H, 0.125, plan=plan)
    rQ, rK, rV = oracle.csr_attention_backward(g.row_ptr, g.col_idx, Q, K, V, dO, H, 0.125)
    for name, got, ref in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        assert_close(to_np(got), ref, TOL_BF16, f"bf16 {name}")


def test_backward_repeat_is_bitwise_identical():
    g = synth.rmat_skew(12, seed=7)
    A = mat(g)
    H, D = 4, 16
    x = [torch.from_numpy(synth.normal(g.n_rows, H * D, 9, st)).cuda()
         for st in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_G)]
    plan = sga.autosage_plan(A, sga.OP_ATTN_BACKWARD, D, heads=H)
    first = [t.clone() for t in sga.autosage_csr_attention_backward(A, *x, H, 0.25, plan=plan)]
    for _ in range(2):
        again = sga.autosage_csr_attention_backward(A, *x, H, 0.25, plan=plan)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


# wide rows: 4 fragments a lane (dV and dK in one pass over A^T) and 8 (two passes)
@pytest.mark.parametrize("H,D", [(2, 256), (4, 256)])
@pytest.mark.parametrize("schedule", [None, dict(kind=sga.SCHED_SPLIT, split=16)], ids=["auto", "split16"])
def test_backward_wide_rows(H, D, schedule):
    run(synth.rmat_skew(10, seed=6), H, D, 1 / np.sqrt(D), 5, schedule=schedule)
