"""Pins for the oracle's CSR-attention backward (no GPU).

The backward is checked against things other than itself: central finite
differences of the oracle's own forward (the definition of a derivative),
torch autograd through a dense masked attention in float64 on the CPU, and
two column-sum identities that follow from the softmax."""
import numpy as np
import pytest

import oracle
import synth


def small_graph(seed=0, n=9, m=7, p=0.5):
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for i in range(n):
        if i == 3:
            continue  # one empty row
        c = np.flatnonzero(rng.random(m) < p)
        if c.size == 0:
            c = np.array([i % m])
        rows += [i] * c.size
        cols += list(c)
    row_ptr = np.zeros(n + 1, np.int32)
    np.cumsum(np.bincount(np.array(rows), minlength=n), out=row_ptr[1:])
    return row_ptr, np.array(cols, np.int32)


def loss(row_ptr, col_idx, Q, K, V, dO, H, scale):
    return float(np.sum(oracle.csr_attention(row_ptr, col_idx, Q, K, V, H, scale) * dO))


@pytest.mark.parametrize("H,D", [(1, 3), (2, 2)])
def test_backward_matches_finite_differences(H, D):
    rp, ci = small_graph()
    n, m, F = rp.size - 1, 7, H * D
    rng = np.random.default_rng(1)
    # values exactly representable in float32 with room for +-eps steps in double
    Q, K, V, dO = (rng.standard_normal((r, F)).astype(np.float32) for r in (n, m, m, n))
    scale = 0.7
    dQ, dK, dV = oracle.csr_attention_backward(rp, ci, Q, K, V, dO, H, scale)
    eps = 1e-3
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        for idx in [(0, 0), (2, F - 1), (X.shape[0] - 1, 1 % F)]:
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += np.float32(eps)
            Xm[idx] -= np.float32(eps)
            step = float(Xp[idx]) - float(Xm[idx])
            args = {"Q": Q, "K": K, "V": V}
            args[name] = Xp
            lp = loss(rp, ci, args["Q"], args["K"], args["V"], dO, H, scale)
            args[name] = Xm
            lm = loss(rp, ci, args["Q"], args["K"], args["V"], dO, H, scale)
            fd = (lp - lm) / step
            assert abs(fd - G[idx]) <= 2e-5 * (1 + abs(G[idx])), (name, idx, fd, G[idx])


def test_backward_matches_torch_autograd_dense():
    torch = pytest.importorskip("torch")
    rp, ci = small_graph(seed=4, n=11, m=11, p=0.4)
    n = rp.size - 1
    H, D = 2, 3
    rng = np.random.default_rng(2)
    Q, K, V, dO = (rng.standard_normal((n, H * D)).astype(np.float32) for _ in range(4))
    scale = 0.5
    dQ, dK, dV = oracle.csr_attention_backward(rp, ci, Q, K, V, dO, H, scale)
    mask = np.zeros((n, n), bool)
    mask[np.repeat(np.arange(n), np.diff(rp)), ci] = True
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    out = []
    for h in range(H):
        sl = slice(h * D, (h + 1) * D)
        s = scale * tq[:, sl] @ tk[:, sl].T
        s = s.masked_fill(~torch.from_numpy(mask), float("-inf"))
        has = torch.from_numpy(mask.any(axis=1))
        w = torch.where(has[:, None], torch.softmax(s, dim=1), torch.zeros_like(s))
        w = torch.nan_to_num(w)
        out.append(w @ tv[:, sl])
    o = torch.cat(out, dim=1)
    (o * torch.from_numpy(dO.astype(np.float64))).sum().backward()
    np.testing.assert_allclose(dQ, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dK, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dV, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_backward_column_sum_identities():
    # each row's softmax weights sum to 1 and its score gradients to 0, so
    # sum_j dV_j = sum of dO over non-empty rows and sum_j dK_j = 0 (per head)
    g = synth.rmat_skew(10, seed=4)
    H, D = 2, 8
    Q, dO = (synth.normal(g.n_rows, H * D, 5, st) for st in (synth.STREAM_Q, synth.STREAM_G))
    K, V = (synth.normal(g.n_cols, H * D, 5, st) for st in (synth.STREAM_K, synth.STREAM_V))
    dQ, dK, dV = oracle.csr_attention_backward(g.row_ptr, g.col_idx, Q, K, V, dO, H, 0.3)
    nonempty = np.diff(g.row_ptr) > 0
    assert (~nonempty).any()  # the identity must hold with empty rows present
    np.testing.assert_allclose(dV.sum(0), dO.astype(np.float64)[nonempty].sum(0), rtol=1e-12, atol=1e-10)
    np.testing.assert_allclose(dK.sum(0), 0.0, atol=1e-10)


BACKWARD_MUTATIONS = [
    # (description, original text, planted mistake)
    ("dS drops the row sum D", "const double ds = w[p - b] * (dw[p - b] - Di);",
     "const double ds = w[p - b] * dw[p - b];"),
    ("dK gathers K instead of Q", "dK[j * F + h * D + d] += scale * ds * (double)q[d];",
     "dK[j * F + h * D + d] += scale * ds * (double)k[d];"),
    ("dQ without the score scale", "dQ[i * F + h * D + d] += scale * ds * (double)k[d];",
     "dQ[i * F + h * D + d] += ds * (double)k[d];"),
    ("dV weighted by dW instead of w", "dV[j * F + h * D + d] += w[p - b] * (double)go[d];",
     "dV[j * F + h * D + d] += dw[p - b] * (double)go[d];"),
]


def _backward_pins_fail() -> bool:
    pins = [lambda: test_backward_matches_finite_differences(1, 3),
            lambda: test_backward_matches_finite_differences(2, 2),
            test_backward_column_sum_identities]
    for pin in pins:
        try:
            pin()
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("desc,orig,bad", BACKWARD_MUTATIONS, ids=[m[0] for m in BACKWARD_MUTATIONS])
def test_planted_backward_mistake_is_caught(tmp_path, desc, orig, bad):
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
        assert _backward_pins_fail(), f"planted mistake not caught: {desc}"
