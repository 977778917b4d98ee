"""GPU parity of the multi-relation (typed) SpMM against the oracle, through the C ABI."""
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


def setup(R, F, seed=0, scale=13):
    g = synth.rmat_skew(scale, seed=seed)
    etype = synth.rng_for(seed, 9).integers(0, R, g.nnz).astype(np.int32)
    Z = synth.normal(R * g.n_cols, F, seed, synth.STREAM_X).reshape(R, g.n_cols, F)
    A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
    return g, etype, Z, A


@pytest.mark.parametrize("R,F", [(1, 16), (4, 64), (7, 33), (3, 256)])
@pytest.mark.parametrize("probe", [False, True])
def test_typed_spmm_planned(R, F, probe):
    g, etype, Z, A = setup(R, F)
    et = torch.from_numpy(etype).cuda()
    plan = sga.autosage_plan_typed(A, et, R, F, flags=(sga.PLAN_PROBE | sga.PLAN_VERIFY) if probe else 0)
    Y = sga.autosage_spmm_typed(A, et, torch.from_numpy(Z).cuda(), plan=plan)
    assert_close(to_np(Y), oracle.spmm_typed(g.row_ptr, g.col_idx, etype, g.vals, Z), TOL_F32, f"typed R={R} F={F}")


def test_typed_spmm_without_plan_and_bf16():
    g, etype, Z, A = setup(5, 64, seed=2, scale=12)
    et = torch.from_numpy(etype).cuda()
    Zb, Z32 = bf16_tensor(Z.reshape(-1, 64))
    Y = sga.autosage_spmm_typed(A, et, Zb.reshape(5, g.n_cols, 64))
    assert Y.dtype == torch.bfloat16
    assert_close(to_np(Y), oracle.spmm_typed(g.row_ptr, g.col_idx, etype, g.vals, Z32.reshape(5, g.n_cols, 64)),
                 TOL_BF16, "typed bf16")


def test_typed_spmm_rejects_bad_types_and_mismatched_plans():
    g, etype, Z, A = setup(3, 8, seed=3, scale=10)
    bad = etype.copy()
    bad[7] = 3
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_plan_typed(A, torch.from_numpy(bad).cuda(), 3, 8)
    assert e.value.status == sga.ERR_INVALID_ARG
    et = torch.from_numpy(etype).cuda()
    plan = sga.autosage_plan_typed(A, et, 3, 8)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_spmm_typed(A, et, torch.zeros((4, g.n_cols, 8), device="cuda"), plan=plan)
    assert e.value.status == sga.ERR_PLAN_MISMATCH
