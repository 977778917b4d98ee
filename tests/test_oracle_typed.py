"""Pins for the oracle's multi-relation (typed) SpMM (no GPU): it equals the
sum over relations of the pinned single-relation SpMM on each relation's
edges, and dense brute force sum_r A_r Z_r."""
import numpy as np

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
