"""Shared helpers for the GPU parity tests (inputs from synth, references from oracle)."""
import numpy as np

import synth

TOL_F32 = 1e-4   # |gpu - oracle| <= TOL * (1 + |oracle|)
TOL_BF16 = 2e-2


def assert_close(gpu, ref, tol, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    err = np.abs(gpu - ref)
    bound = tol * (1.0 + np.abs(ref))
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / bound, 0)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu={gpu[i]!r} oracle={ref[i]!r}")


def to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def bf16_tensor(x32, device="cuda"):
    """float32 array -> (torch bf16 tensor, exact float32 values of it) via synth's RNE rounding."""
    import torch
    bits = synth.bf16_bits(x32)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return t, synth.bf16_to_f32(bits).reshape(x32.shape)


def csr_from_lists(rows_cols, n_rows, n_cols, vals=None):
    """Build CSR arrays from a list of (row, col) pairs, keeping the given order per row."""
    counts = np.zeros(n_rows, dtype=np.int64)
    for r, _ in rows_cols:
        counts[r] += 1
    row_ptr = np.zeros(n_rows + 1, dtype=np.int32)
    np.cumsum(counts, out=row_ptr[1:])
    order = sorted(range(len(rows_cols)), key=lambda k: (rows_cols[k][0], k))
    col_idx = np.array([rows_cols[k][1] for k in order], dtype=np.int32)
    v = None if vals is None else np.asarray(vals, dtype=np.float32)[order]
    return synth.Csr(n_rows, n_cols, row_ptr, col_idx, v)
