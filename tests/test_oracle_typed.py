"""Pins for the oracle's multi-relation (typed) SpMM (no GPU): it equals the
sum over relations of the pinned single-relation SpMM on each relation's
edges, and dense brute force sum_r A_r Z_r."""
import numpy as np
import pytest

import oracle


def test_typed_spmm_is_sum_of_relations():
    rng = np.random.default_rng(3)
    n, m, R, F = 20, 15, 3, 5
    rows, cols = np.nonzero(rng.random((n, m)) < 0.3)
    row_ptr = np.zeros(n + 1, np.int32)
    np.cumsum(np.bincount(rows, minlength=n), out=row_ptr[1:])
    col_idx = cols.astype(np.int32)
    etype = rng.integers(0, R, col_idx.size).astype(np.int32)
    vals = rng.uniform(-1, 1, col_idx.size).astype(np.float32)
    Z = rng.standard_normal((R, m, F)).astype(np.float32)
    Y = oracle.spmm_typed(row_ptr, col_idx, etype, vals, Z)
    dense = np.zeros((n, F))
    per_rel = np.zeros((n, F))
    for r in range(R):
        A = np.zeros((n, m))
        sel = etype == r
        np.add.at(A, (rows[sel], cols[sel]), vals[sel].astype(np.float64))
        dense += A @ Z[r].astype(np.float64)
        # the same relation through the single-relation oracle (edges of other types get weight 0)
        per_rel += oracle.spmm(row_ptr, col_idx, np.where(sel, vals, 0).astype(np.float32), Z[r])
    np.testing.assert_allclose(Y, dense, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(Y, per_rel, rtol=1e-12, atol=1e-12)
    # one relation reduces to plain SpMM exactly
    np.testing.assert_array_equal(oracle.spmm_typed(row_ptr, col_idx, np.zeros_like(etype), vals, Z[:1]),
                                  oracle.spmm(row_ptr, col_idx, vals, Z[0]))


TYPED_MUTATIONS = [
    ("relation ignored", "const float *z = Z + ((int64_t)edge_type[p] * n_cols + col_idx[p]) * ldz;",
     "const float *z = Z + ((int64_t)col_idx[p]) * ldz;"),
    ("edge value dropped", "      const double w = vals ? (double)vals[p] : 1.0;\n      const float *z = Z",
     "      const double w = 1.0;\n      const float *z = Z"),
]



@pytest.mark.parametrize("desc,orig,bad", TYPED_MUTATIONS, ids=[m[0] for m in TYPED_MUTATIONS])
def test_planted_typed_mistake_is_caught(tmp_path, desc, orig, bad):
    import os
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert orig in src, f"mutation anchor missing: {orig!r}"
    c = tmp_path / "oracle_bad.c"
    c.write_text(src.replace(orig, bad))
    so = tmp_path / "liboracle_bad.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", str(c), "-o", str(so), "-lm"],
                   check=True)
    with oracle.use_library(str(so)):
        with pytest.raises(AssertionError):
            test_typed_spmm_is_sum_of_relations()
