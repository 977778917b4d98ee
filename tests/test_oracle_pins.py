"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: a hand-worked
example (tests/golden/tiny_hand.json), brute-force dense linear algebra on
tiny graphs (numpy matmul, scipy), closed forms and invariants that the
definitions fix (identity, linearity, adjointness, softmax normalisation
and shift invariance, constant scores reducing attention to a mean).
The last test plants plausible mistakes in a copy of oracle.c and checks
that these pins catch every one of them.

Definitions followed: AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN
Aggregation (SpMM/SDDMM) and CSR Attention", Abstract (SpMM, SDDMM, the
pipeline SDDMM -> row-softmax -> SpMM); benchmark page "fused sparse
attention-value aggregation", problem statement (rows are destinations,
col_idx are sources, max-subtracted softmax, empty rows give zeros).
"""
import json
import os
import shutil
import subprocess

import numpy as np
import pytest
import scipy.sparse as sp
from scipy.special import softmax as sp_softmax

import oracle
import synth


# ---------------------------------------------------------------- helpers

def random_csr(n_rows, n_cols, density, seed, dup=False, empty_rows=()):
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for i in range(n_rows):
        if i in empty_rows:
            continue
        c = np.flatnonzero(rng.random(n_cols) < density)
        if dup and c.size:
            c = np.sort(np.concatenate([c, c[: max(1, c.size // 3)]]))
        rows += [i] * c.size
        cols += list(c)
    rows = np.array(rows, dtype=np.int64)
    cols = np.array(cols, dtype=np.int32)
    row_ptr = np.zeros(n_rows + 1, dtype=np.int32)
    np.cumsum(np.bincount(rows, minlength=n_rows), out=row_ptr[1:])
    vals = rng.uniform(-1, 1, cols.size).astype(np.float32)
    return row_ptr, cols, vals


def dense_of(row_ptr, col_idx, vals, n_cols):
    n = row_ptr.size - 1
    A = np.zeros((n, n_cols))
    rows = np.repeat(np.arange(n), np.diff(row_ptr))
    np.add.at(A, (rows, col_idx), vals.astype(np.float64) if vals is not None else 1.0)
    return A


def mask_of(row_ptr, col_idx, n_cols):
    n = row_ptr.size - 1
    M = np.zeros((n, n_cols), dtype=bool)
    M[np.repeat(np.arange(n), np.diff(row_ptr)), col_idx] = True
    return M


def dense_attention(row_ptr, col_idx, Q, K, V, heads, scale):
    """Masked dense attention: softmax over each row's pattern entries, then @ V."""
    n = row_ptr.size - 1
    M = mask_of(row_ptr, col_idx, K.shape[0])
    D = Q.shape[1] // heads
    O = np.zeros((n, Q.shape[1]))
    for h in range(heads):
        sl = slice(h * D, (h + 1) * D)
        S = scale * (Q[:, sl].astype(np.float64) @ K[:, sl].astype(np.float64).T)
        S = np.where(M, S, -np.inf)
        has = M.any(axis=1)
        P = np.zeros_like(S)
        P[has] = sp_softmax(S[has], axis=1)
        O[:, sl] = P @ V[:, sl].astype(np.float64)
    return O


GRAPHS = [
    ("dense-ish", dict(n_rows=17, n_cols=23, density=0.4, seed=1)),
    ("sparse-empty", dict(n_rows=40, n_cols=40, density=0.05, seed=2, empty_rows=(0, 5, 39))),
    ("duplicates", dict(n_rows=12, n_cols=9, density=0.5, seed=3, dup=True)),
    ("one-row", dict(n_rows=1, n_cols=64, density=0.5, seed=4)),
]


# ---------------------------------------------------------------- golden

@pytest.fixture(scope="module")
def hand(golden_dir):
    with open(os.path.join(golden_dir, "tiny_hand.json")) as f:
        return json.load(f)


def _hand_graph(hand):
    g = hand["graph"]
    return (np.array(g["row_ptr"], np.int32), np.array(g["col_idx"], np.int32),
            np.array(g["vals"], np.float32), np.array(hand["X"], np.float32))


def test_golden_hand_spmm(hand):
    rp, ci, v, X = _hand_graph(hand)
    np.testing.assert_array_equal(oracle.spmm(rp, ci, v, X), np.array(hand["spmm"]["Y"]))


def test_golden_hand_sddmm_softmax(hand):
    rp, ci, _, X = _hand_graph(hand)
    S = oracle.sddmm(rp, ci, X, X, 1.0)
    np.testing.assert_array_equal(S[:, 0], np.array(hand["sddmm"]["S"]))
    W = oracle.row_softmax(rp, S)
    np.testing.assert_allclose(W[:, 0], hand["row_softmax"]["W"], rtol=1e-15, atol=1e-17)


def test_golden_hand_attention(hand):
    rp, ci, _, X = _hand_graph(hand)
    O = oracle.csr_attention(rp, ci, X, X, X, 1, hand["attention"]["scale"])
    np.testing.assert_allclose(O, np.array(hand["attention"]["O"]), rtol=1e-15, atol=0)
    O2 = oracle.csr_attention(rp, ci, X, X, X, 1, hand["attention_half_scale"]["scale"])
    w = hand["attention_half_scale"]["w"]
    np.testing.assert_allclose(O2[0], [3 + 2 * w[1], 4 + 2 * w[1]], rtol=1e-15)


def test_golden_hand_transpose(hand):
    rp, ci, v, _ = _hand_graph(hand)
    rpt, cit, vt = oracle.transpose(rp, ci, v, 3)
    t = hand["transpose"]
    np.testing.assert_array_equal(rpt, t["row_ptr"])
    np.testing.assert_array_equal(cit, t["col_idx"])
    np.testing.assert_array_equal(vt, np.array(t["vals"], np.float32))


# ---------------------------------------------------------------- SpMM

@pytest.mark.parametrize("name,kw", GRAPHS)
def test_spmm_matches_dense(name, kw):
    rp, ci, v = random_csr(**kw)
    X = np.random.default_rng(7).standard_normal((kw["n_cols"], 5)).astype(np.float32)
    Y = oracle.spmm(rp, ci, v, X)
    ref = dense_of(rp, ci, v, kw["n_cols"]) @ X.astype(np.float64)
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)
    # row subset, out of order and repeated, gives the same rows
    rows = np.array([kw["n_rows"] - 1, 0, kw["n_rows"] // 2, 0])
    np.testing.assert_array_equal(oracle.spmm(rp, ci, v, X, rows=rows), Y[rows])


def test_spmm_identity_is_exact():
    n, F = 33, 7
    rp = np.arange(n + 1, dtype=np.int32)
    ci = np.arange(n, dtype=np.int32)
    X = np.random.default_rng(0).standard_normal((n, F)).astype(np.float32)
    np.testing.assert_array_equal(oracle.spmm(rp, ci, np.ones(n, np.float32), X), X.astype(np.float64))
    np.testing.assert_array_equal(oracle.spmm(rp, ci, None, X), X.astype(np.float64))
    c = np.float32(-2.5)
    np.testing.assert_array_equal(oracle.spmm(rp, ci, np.full(n, c, np.float32), X),
                                  float(c) * X.astype(np.float64))


def test_spmm_ones_column_gives_row_sums_and_empty_rows_zero():
    rp, ci, v = random_csr(30, 30, 0.2, 5, empty_rows=(3, 4))
    Y = oracle.spmm(rp, ci, v, np.ones((30, 1), np.float32))
    sums = np.array([v[rp[i]:rp[i + 1]].astype(np.float64).sum() for i in range(30)])
    np.testing.assert_allclose(Y[:, 0], sums, rtol=1e-13, atol=1e-14)
    assert Y[3, 0] == 0.0 and Y[4, 0] == 0.0


def test_spmm_linearity_and_permutation():
    rp, ci, v = random_csr(25, 31, 0.3, 6)
    rng = np.random.default_rng(1)
    X1 = rng.standard_normal((31, 4)).astype(np.float32)
    X2 = rng.standard_normal((31, 4)).astype(np.float32)
    # A(X1 + X2) = A X1 + A X2 (X1 + X2 formed exactly: both halves are float32
    # multiples of a power of two small enough that the float32 sum is exact)
    X1 = np.round(X1 * 256) / 256
    X2 = np.round(X2 * 256) / 256
    lhs = oracle.spmm(rp, ci, v, X1 + X2)
    np.testing.assert_allclose(lhs, oracle.spmm(rp, ci, v, X1) + oracle.spmm(rp, ci, v, X2),
                               rtol=1e-13, atol=1e-13)
    # reversing the edges inside each row changes nothing beyond rounding
    ci2, v2 = ci.copy(), v.copy()
    for i in range(25):
        ci2[rp[i]:rp[i + 1]] = ci[rp[i]:rp[i + 1]][::-1]
        v2[rp[i]:rp[i + 1]] = v[rp[i]:rp[i + 1]][::-1]
    np.testing.assert_allclose(oracle.spmm(rp, ci2, v2, X1), oracle.spmm(rp, ci, v, X1), rtol=1e-14, atol=1e-15)


def test_spmm_multihead_matches_per_head_dense():
    rp, ci, v = random_csr(20, 20, 0.3, 8)
    H, D = 3, 4
    rng = np.random.default_rng(2)
    W = rng.uniform(0, 1, (ci.size, H)).astype(np.float32)
    X = rng.standard_normal((20, H * D)).astype(np.float32)
    Y = oracle.spmm(rp, ci, W, X, heads=H)
    for h in range(H):
        ref = dense_of(rp, ci, W[:, h], 20) @ X[:, h * D:(h + 1) * D].astype(np.float64)
        np.testing.assert_allclose(Y[:, h * D:(h + 1) * D], ref, rtol=1e-12, atol=1e-12)


def test_spmm_ld_larger_than_f():
    rp, ci, v = random_csr(10, 12, 0.4, 9)
    big = np.random.default_rng(3).standard_normal((12, 9)).astype(np.float32)
    X = big[:, :5]  # row stride 9 floats
    np.testing.assert_array_equal(oracle.spmm(rp, ci, v, X), oracle.spmm(rp, ci, v, np.ascontiguousarray(X)))


# ---------------------------------------------------------------- transpose / SpMM-T

@pytest.mark.parametrize("name,kw", GRAPHS)
def test_transpose_matches_scipy(name, kw):
    rp, ci, v = random_csr(**kw)
    rpt, cit, vt = oracle.transpose(rp, ci, v, kw["n_cols"])
    A = sp.csr_matrix((v, ci, rp), shape=(kw["n_rows"], kw["n_cols"]))
    T = A.T.tocsr()  # scipy keeps duplicates; entries within a row ordered by original row
    T.has_sorted_indices = False
    T.sort_indices()
    np.testing.assert_array_equal(rpt, T.indptr)
    # within a column, duplicates share a row; compare (row, value) multisets per row of A^T
    for j in range(kw["n_cols"]):
        a = sorted(zip(cit[rpt[j]:rpt[j + 1]], vt[rpt[j]:rpt[j + 1]]))
        b = sorted(zip(T.indices[T.indptr[j]:T.indptr[j + 1]], T.data[T.indptr[j]:T.indptr[j + 1]]))
        assert a == b
        assert np.all(np.diff(cit[rpt[j]:rpt[j + 1]]) >= 0), "rows of A^T must keep increasing order"
    # transposing twice gives A back
    rp2, ci2, v2 = oracle.transpose(rpt, cit, vt, kw["n_rows"])
    np.testing.assert_array_equal(rp2, rp)
    np.testing.assert_array_equal(ci2, ci)
    np.testing.assert_array_equal(v2, v)


@pytest.mark.parametrize("name,kw", GRAPHS)
def test_spmm_t_adjoint_and_scatter_route(name, kw):
    rp, ci, v = random_csr(**kw)
    rng = np.random.default_rng(11)
    G = rng.standard_normal((kw["n_rows"], 3)).astype(np.float32)
    X = rng.standard_normal((kw["n_cols"], 3)).astype(np.float32)
    GX = oracle.spmm_t(rp, ci, v, G, kw["n_cols"])
    np.testing.assert_allclose(GX, oracle.spmm_t_scatter(rp, ci, v, G, kw["n_cols"]), rtol=1e-13, atol=1e-13)
    lhs = np.sum(G.astype(np.float64) * oracle.spmm(rp, ci, v, X))
    rhs = np.sum(GX * X.astype(np.float64))
    assert abs(lhs - rhs) <= 1e-12 * (1 + abs(lhs))
    np.testing.assert_allclose(GX, dense_of(rp, ci, v, kw["n_cols"]).T @ G.astype(np.float64),
                               rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- SDDMM

@pytest.mark.parametrize("name,kw", GRAPHS)
@pytest.mark.parametrize("heads", [1, 2])
def test_sddmm_matches_dense_masked(name, kw, heads):
    rp, ci, _ = random_csr(**kw)
    rng = np.random.default_rng(12)
    D = 3
    Q = rng.standard_normal((kw["n_rows"], heads * D)).astype(np.float32)
    K = rng.standard_normal((kw["n_cols"], heads * D)).astype(np.float32)
    S = oracle.sddmm(rp, ci, Q, K, 0.75, heads=heads)
    rows = np.repeat(np.arange(kw["n_rows"]), np.diff(rp))
    for h in range(heads):
        sl = slice(h * D, (h + 1) * D)
        dense = 0.75 * (Q[:, sl].astype(np.float64) @ K[:, sl].astype(np.float64).T)
        np.testing.assert_allclose(S[:, h], dense[rows, ci], rtol=1e-13, atol=1e-14)
    sub = np.array([kw["n_rows"] - 1, 0])
    s_sub = oracle.sddmm(rp, ci, Q, K, 0.75, heads=heads, rows=sub)
    want = np.concatenate([S[rp[i]:rp[i + 1]] for i in sub])
    np.testing.assert_array_equal(s_sub, want.reshape(s_sub.shape))


# ---------------------------------------------------------------- softmax

def test_softmax_normalised_shift_invariant_and_stable():
    rp, ci, _ = random_csr(30, 30, 0.3, 13, empty_rows=(7,))
    rng = np.random.default_rng(4)
    S = rng.standard_normal((ci.size, 2)) * 3
    W = oracle.row_softmax(rp, S)
    assert np.all(W >= 0)
    for i in range(30):
        b, e = rp[i], rp[i + 1]
        if e > b:
            np.testing.assert_allclose(W[b:e].sum(axis=0), 1.0, rtol=0, atol=1e-12)
            np.testing.assert_allclose(W[b:e], sp_softmax(S[b:e], axis=0), rtol=1e-13, atol=1e-16)
    shift = np.repeat(rng.uniform(-50, 50, 30), np.diff(rp))[:, None]
    np.testing.assert_allclose(oracle.row_softmax(rp, S + shift), W, rtol=1e-12, atol=1e-15)
    big = oracle.row_softmax(rp, S * 1e3 / 9)
    assert np.all(np.isfinite(big))


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("name,kw", GRAPHS)
@pytest.mark.parametrize("heads", [1, 2])
def test_attention_matches_dense_masked(name, kw, heads):
    if kw.get("dup"):
        pytest.skip("a dense mask cannot hold a repeated edge; each CSR entry is its own softmax term")
    rp, ci, _ = random_csr(**kw)
    n_src = kw["n_cols"]
    rng = np.random.default_rng(14)
    D = 4
    Q = rng.standard_normal((kw["n_rows"], heads * D)).astype(np.float32)
    K = rng.standard_normal((n_src, heads * D)).astype(np.float32)
    V = rng.standard_normal((n_src, heads * D)).astype(np.float32)
    O = oracle.csr_attention(rp, ci, Q, K, V, heads, 0.5)
    np.testing.assert_allclose(O, dense_attention(rp, ci, Q, K, V, heads, 0.5), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("heads", [1, 2])
def test_attention_duplicate_edges_are_separate_terms(heads):
    # Reading of the CSR with repeated entries: each entry is its own term of
    # the row's softmax and sum (a repeated edge counts twice). Expanding the
    # columns so that entry p of the CSR is key/value column p turns the
    # pattern into one without repeats, where dense masked attention applies.
    rp, ci, _ = random_csr(n_rows=12, n_cols=9, density=0.5, seed=3, dup=True)
    assert any(np.unique(ci[rp[i]:rp[i + 1]]).size < rp[i + 1] - rp[i] for i in range(12)), "no repeated entry"
    rng = np.random.default_rng(15)
    D = 4
    Q = rng.standard_normal((12, heads * D)).astype(np.float32)
    K = rng.standard_normal((9, heads * D)).astype(np.float32)
    V = rng.standard_normal((9, heads * D)).astype(np.float32)
    O = oracle.csr_attention(rp, ci, Q, K, V, heads, 0.5)
    expanded = np.arange(ci.size, dtype=np.int32)
    want = dense_attention(rp, expanded, Q, K[ci], V[ci], heads, 0.5)
    np.testing.assert_allclose(O, want, rtol=1e-12, atol=1e-13)


def test_attention_constant_scores_is_mean_aggregation():
    g = synth.erdos_renyi(64, 6.0, seed=3)
    rng = np.random.default_rng(5)
    K = rng.standard_normal((64, 8)).astype(np.float32)
    V = rng.standard_normal((64, 8)).astype(np.float32)
    mean = oracle.spmm(g.row_ptr, g.col_idx, synth.mean_vals(g), V)
    O = oracle.csr_attention(g.row_ptr, g.col_idx, np.zeros((64, 8), np.float32), K, V, 2, 0.3)
    np.testing.assert_allclose(O, mean, rtol=1e-6, atol=1e-7)  # mean_vals are float32 1/deg
    O0 = oracle.csr_attention(g.row_ptr, g.col_idx, K, K, V, 1, 0.0)
    np.testing.assert_allclose(O0, mean, rtol=1e-6, atol=1e-7)
    deg = g.degrees()
    # exact against a double-precision mean
    exact = np.zeros_like(O)
    for i in range(64):
        if deg[i]:
            exact[i] = V[g.col_idx[g.row_ptr[i]:g.row_ptr[i + 1]]].astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(O, exact, rtol=1e-13, atol=1e-14)
    assert np.all(O[deg == 0] == 0.0)


def test_attention_one_edge_row_copies_value():
    rp = np.array([0, 1, 1, 2], np.int32)
    ci = np.array([2, 0], np.int32)
    rng = np.random.default_rng(6)
    Q, K, V = (rng.standard_normal((3, 6)).astype(np.float32) for _ in range(3))
    O = oracle.csr_attention(rp, ci, Q, K, V, 3, 1.7)
    np.testing.assert_array_equal(O[0], V[2].astype(np.float64))
    np.testing.assert_array_equal(O[1], 0.0)
    np.testing.assert_array_equal(O[2], V[0].astype(np.float64))


def test_edge_softmax_aggregate_matches_dense():
    g = synth.attention_benchmark_shape(seed=1)
    rng = np.random.default_rng(8)
    scores = rng.standard_normal(g.nnz).astype(np.float32)
    V = rng.standard_normal((g.n_rows, 16)).astype(np.float32)
    out = oracle.edge_softmax_aggregate(g.row_ptr, g.col_idx, scores, V)
    M = mask_of(g.row_ptr, g.col_idx, g.n_cols)
    S = np.full((g.n_rows, g.n_cols), -np.inf)
    S[np.repeat(np.arange(g.n_rows), g.degrees()), g.col_idx] = scores
    P = np.zeros_like(S)
    has = M.any(axis=1)
    P[has] = sp_softmax(S[has], axis=1)
    np.testing.assert_allclose(out, P @ V.astype(np.float64), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- planner statistics, fingerprint

def test_row_stats_brute_force():
    rp, _, _ = random_csr(200, 300, 0.05, 21, empty_rows=(1, 2, 3))
    ints, reals = oracle.row_stats(rp, long_threshold=18)
    d = np.diff(rp).astype(np.int64)
    assert ints[0] == 200 and ints[1] == d.sum() and ints[2] == d.max() and ints[3] == d.min()
    assert ints[4] == np.count_nonzero(d == 0) and ints[5] == (d * d).sum()
    assert ints[6] == np.count_nonzero(d > 18) and ints[7] == d[d > 18].sum()
    buckets = np.zeros(32, np.int64)
    for x in d:
        buckets[0 if x == 0 else int(x).bit_length()] += 1
    np.testing.assert_array_equal(ints[8:], buckets)
    assert reals[0] == pytest.approx(d.mean(), rel=1e-15)
    assert reals[1] == pytest.approx(d.std() / d.mean(), rel=1e-12)


def _py_fingerprint(row_ptr, col_idx):
    M = (1 << 64) - 1

    def mix(z):
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M
        return z ^ (z >> 31)

    n = len(row_ptr) - 1
    h = mix(n)
    for i, r in enumerate(row_ptr):
        h = (h + mix(0x9E3779B97F4A7C15 ^ (i << 32) ^ (int(r) & 0xFFFFFFFF))) & M
    for p, c in enumerate(col_idx):
        h = (h + mix(0xD1B54A32D192ED03 ^ (p << 32) ^ (int(c) & 0xFFFFFFFF))) & M
    return h


def test_fingerprint_brute_force_and_sensitivity():
    rp, ci, _ = random_csr(50, 50, 0.1, 22)
    f = oracle.fingerprint(rp, ci)
    assert f == _py_fingerprint(rp, ci)
    ci2 = ci.copy()
    ci2[len(ci2) // 2] ^= 1
    assert oracle.fingerprint(rp, ci2) != f


# ---------------------------------------------------------------- named workloads

def test_generators_are_deterministic_and_well_formed():
    a, b = synth.tiny_er(0), synth.tiny_er(0)
    np.testing.assert_array_equal(a.row_ptr, b.row_ptr)
    np.testing.assert_array_equal(a.col_idx, b.col_idx)
    np.testing.assert_array_equal(a.vals, b.vals)
    assert a.n_rows == 4096 and 60000 < a.nnz < 71000
    for g in (a, synth.rmat(10, 16, seed=1), synth.products_like(scale=1e-3), synth.reddit_like(scale=2e-3)):
        assert g.row_ptr[0] == 0 and np.all(np.diff(g.row_ptr) >= 0)
        assert g.col_idx.min() >= 0 and g.col_idx.max() < g.n_cols
        for i in range(0, g.n_rows, max(1, g.n_rows // 50)):
            seg = g.col_idx[g.row_ptr[i]:g.row_ptr[i + 1]]
            assert np.all(np.diff(seg) > 0), "columns sorted and distinct inside a row"
    bits = synth.bf16_bits(np.array([1.0, 1.00390625, 1.01171875, -2.0, 3.0e38], np.float32))
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties go to even (1.0)
    np.testing.assert_array_equal(synth.bf16_to_f32(bits)[:4], [1.0, 1.0, 1.015625, -2.0])


# ---------------------------------------------------------------- planted mistakes

MUTATIONS = [
    # (description, original text, planted mistake)
    ("SpMM gathers the destination row instead of the source",
     "const float *x = X + (int64_t)col_idx[p] * ldx;", "const float *x = X + i * ldx;"),
    ("SpMM drops the edge value", "const double w = vals ? (double)vals[p * H + h] : 1.0;",
     "const double w = 1.0;"),
    ("SDDMM uses the destination's K row", "const float *kk = K + (int64_t)col_idx[p] * ldk;\n      for (int64_t h = 0; h < H; ++h) {\n        double s",
     "const float *kk = K + i * ldk;\n      for (int64_t h = 0; h < H; ++h) {\n        double s"),
    ("softmax forgets to normalise", "W[p * H + h] = exp(S[p * H + h] - m) / sum;",
     "W[p * H + h] = exp(S[p * H + h] - m);"),
    ("attention drops the scale", "s[p - b] = scale * acc;", "s[p - b] = acc;"),
    ("attention aggregates K instead of V", "const float *v = V + (int64_t)col_idx[p] * ldv;",
     "const float *v = K + (int64_t)col_idx[p] * ldk;"),
    ("transpose is not stable", "const int64_t dst = next[col_idx[p]]++;",
     "const int64_t dst = (i % 2) ? next[col_idx[p]]++ : next[col_idx[p]]++ ;"),
    ("transpose loses the values", "if (vals && vals_t) vals_t[dst] = vals[p];",
     "if (vals && vals_t) vals_t[dst] = 1.0f;"),
]

PIN_TESTS = [
    lambda: test_spmm_matches_dense("dense-ish", GRAPHS[0][1]),
    lambda: test_spmm_identity_is_exact(),
    lambda: test_sddmm_matches_dense_masked("dense-ish", GRAPHS[0][1], 2),
    lambda: test_softmax_normalised_shift_invariant_and_stable(),
    lambda: test_attention_matches_dense_masked("sparse-empty", GRAPHS[1][1], 2),
    lambda: test_attention_one_edge_row_copies_value(),
    lambda: test_transpose_matches_scipy("duplicates", GRAPHS[2][1]),
    lambda: test_spmm_t_adjoint_and_scatter_route("dense-ish", GRAPHS[0][1]),
]


def _caught(lib_path):
    with oracle.use_library(lib_path):
        for t in PIN_TESTS:
            try:
                t()
            except AssertionError:
                return True
    return False


@pytest.mark.parametrize("desc,orig,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, desc, orig, bad):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert orig in src, f"mutation anchor missing: {orig!r}"
    if desc == "transpose is not stable":
        # reverse the order inside each column instead of keeping row order
        bad_src = src.replace("for (int64_t i = 0; i < n_rows; ++i) {\n    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {\n      const int64_t dst",
                              "for (int64_t i = n_rows - 1; i >= 0; --i) {\n    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {\n      const int64_t dst")
        assert bad_src != src
    else:
        bad_src = src.replace(orig, bad)
    c = tmp_path / "oracle_bad.c"
    c.write_text(bad_src)
    so = tmp_path / "liboracle_bad.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", str(c), "-o", str(so), "-lm"], check=True)
    assert _caught(str(so)), f"planted mistake not caught: {desc}"
