"""Seeded synthetic inputs for CSR sparse aggregation.

This module only draws graphs and feature matrices. It holds none of the
aggregation method's arithmetic (no SpMM, SDDMM, softmax or attention), so
the CPU oracle and the CUDA path can both take their inputs from here
without sharing any of the computation they are compared on.

Conventions (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN
Aggregation (SpMM/SDDMM) and CSR Attention", Abstract; and the benchmark
page "fused sparse attention-value aggregation", problem statement):
rows are destination nodes, ``col_idx`` holds the source node of each edge,
``row_ptr`` has ``n_rows + 1`` int32 entries, edge values are float32.
Generated graphs have duplicate edges merged and ``col_idx`` sorted
ascending inside every row.

Every draw uses numpy's PCG64 seeded from ``SeedSequence([seed, stream])``,
so a (seed, stream) pair gives the same numbers on every machine.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Streams: one independent substream per drawn object.
STREAM_GRAPH = 0
STREAM_VALS = 1
STREAM_X = 2
STREAM_Q = 3
STREAM_K = 4
STREAM_V = 5
STREAM_G = 6


def rng_for(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


@dataclasses.dataclass
class Csr:
    """A CSR matrix: rows are destinations, columns are sources."""

    n_rows: int
    n_cols: int
    row_ptr: np.ndarray  # int32 [n_rows + 1]
    col_idx: np.ndarray  # int32 [nnz]
    vals: np.ndarray | None = None  # float32 [nnz] or None (= all ones)

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    def degrees(self) -> np.ndarray:
        return np.diff(self.row_ptr.astype(np.int64))

    def with_vals(self, vals: np.ndarray | None) -> "Csr":
        return Csr(self.n_rows, self.n_cols, self.row_ptr, self.col_idx, vals)


def _csr_from_sorted_keys(keys: np.ndarray, n_rows: int, n_cols: int) -> Csr:
    """Build CSR from globally sorted, duplicate-free keys row * n_cols + col."""
    rows = keys // n_cols
    cols = (keys - rows * n_cols).astype(np.int32)
    counts = np.bincount(rows, minlength=n_rows).astype(np.int64)
    row_ptr = np.zeros(n_rows + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    if row_ptr[-1] > np.iinfo(np.int32).max:
        raise ValueError("nnz does not fit int32")
    return Csr(n_rows, n_cols, row_ptr.astype(np.int32), cols)


def csr_from_degrees(deg: np.ndarray, n_cols: int, rng: np.random.Generator,
                     draw=None) -> Csr:
    """Rows with the given degrees; each row gets distinct sorted columns.

    ``draw(rows, rng)`` returns one candidate column per entry of ``rows``
    (default: uniform over ``[0, n_cols)``). Duplicates inside a row are
    redrawn uniformly over all columns until none remain, so every row keeps
    its exact degree (a degree must not exceed ``n_cols``).
    """
    deg = np.asarray(deg, dtype=np.int64)
    n_rows = deg.shape[0]
    if deg.size and int(deg.max()) > n_cols:
        raise ValueError("degree larger than the number of columns")
    rows = np.repeat(np.arange(n_rows, dtype=np.int64), deg)
    cols = draw(rows, rng) if draw is not None else rng.integers(0, n_cols, rows.shape[0], dtype=np.int64)
    keys = rows * n_cols + cols.astype(np.int64)
    del rows, cols
    keys.sort()
    while True:
        dup = np.flatnonzero(keys[1:] == keys[:-1]) + 1
        if dup.size == 0:
            break
        r = keys[dup] // n_cols
        keys[dup] = r * n_cols + rng.integers(0, n_cols, dup.size, dtype=np.int64)
        keys.sort()
    return _csr_from_sorted_keys(keys, n_rows, n_cols)


def erdos_renyi(n: int, avg_degree: float, seed: int = 0) -> Csr:
    """G(n, p) with p = avg_degree / n over all n*n ordered pairs (self-loops allowed)."""
    rng = rng_for(seed, STREAM_GRAPH)
    p = float(avg_degree) / float(n)
    rows_all, cols_all = [], []
    block = max(1, (1 << 22) // max(n, 1))
    for r0 in range(0, n, block):
        r1 = min(n, r0 + block)
        mask = rng.random((r1 - r0, n)) < p
        r, c = np.nonzero(mask)
        rows_all.append(r.astype(np.int64) + r0)
        cols_all.append(c.astype(np.int64))
    rows = np.concatenate(rows_all) if rows_all else np.zeros(0, np.int64)
    cols = np.concatenate(cols_all) if cols_all else np.zeros(0, np.int64)
    return _csr_from_sorted_keys(rows * n + cols, n, n)


def rmat(scale: int, edge_factor: int = 16, a: float = 0.57, b: float = 0.19,
         c: float = 0.19, seed: int = 0) -> Csr:
    """R-MAT graph: 2**scale nodes, edge_factor * 2**scale drawn (u, v) pairs.

    Each pair picks one quadrant per bit level with probabilities a, b, c and
    d = 1 - a - b - c (no noise, no vertex permutation). Row = u. Duplicate
    pairs are merged; self-loops are kept.
    """
    rng = rng_for(seed, STREAM_GRAPH)
    n = 1 << scale
    m = edge_factor * n
    u = np.zeros(m, dtype=np.int64)
    v = np.zeros(m, dtype=np.int64)
    ab, abc = np.float32(a + b), np.float32(a + b + c)
    fa = np.float32(a)
    block = 1 << 18  # edges per block: keeps the per-level temporaries in cache
    for s0 in range(0, m, block):
        s1 = min(m, s0 + block)
        r = rng.random((scale, s1 - s0), dtype=np.float32)  # one row of draws per bit level
        ub = np.zeros(s1 - s0, dtype=np.int64)
        vb = np.zeros(s1 - s0, dtype=np.int64)
        for level in range(scale):
            rl = r[level]
            # quadrant: [0,a) -> (0,0); [a,a+b) -> (0,1); [a+b,a+b+c) -> (1,0); else (1,1)
            ub <<= 1
            vb <<= 1
            ub |= rl >= ab
            vb |= ((rl >= fa) & (rl < ab)) | (rl >= abc)
        u[s0:s1] = ub
        v[s0:s1] = vb
    keys = u * n + v
    keys.sort()
    keep = np.ones(keys.shape[0], dtype=bool)
    keep[1:] = keys[1:] != keys[:-1]
    return _csr_from_sorted_keys(keys[keep], n, n)


def uniform_degree(n: int, nnz: int, seed: int = 0) -> Csr:
    """Control graph: every row gets floor(nnz/n) or ceil(nnz/n) distinct uniform columns."""
    rng = rng_for(seed, STREAM_GRAPH)
    base, extra = divmod(int(nnz), int(n))
    deg = np.full(n, base, dtype=np.int64)
    deg[rng.permutation(n)[:extra]] += 1
    return csr_from_degrees(deg, n, rng)


def _rescale_degrees(deg: np.ndarray, target: int, max_deg: int, rng) -> np.ndarray:
    """Scale real degrees so they sum to ``target`` with every degree in [1, max_deg]."""
    deg = np.clip(deg, 1.0, float(max_deg))
    for _ in range(20):
        s = deg.sum()
        deg = np.clip(deg * (target / s), 1.0, float(max_deg))
    d = np.floor(deg).astype(np.int64)
    # distribute the rounding remainder to random rows that still have room
    short = int(target - d.sum())
    if short > 0:
        room = np.flatnonzero(d < max_deg)
        pick = rng.choice(room, size=min(short, room.size), replace=False)
        d[pick] += 1
    return d


def lognormal_powerlaw(n: int = 2_449_029, nnz: int = 123_700_000, sigma: float = 1.3,
                       max_deg: int = 17_000, seed: int = 0) -> Csr:
    """Degrees ~ LogNormal(mu, sigma) with mu = ln(nnz/n) - sigma^2/2, clipped to
    [1, max_deg] and rescaled to sum to ``nnz``; distinct uniform sorted sources."""
    rng = rng_for(seed, STREAM_GRAPH)
    mean = nnz / n
    mu = math.log(mean) - sigma * sigma / 2.0
    deg = rng.lognormal(mu, sigma, n)
    d = _rescale_degrees(deg, nnz, max_deg, rng)
    return csr_from_degrees(d, n, rng)


def community_powerlaw(n: int = 232_965, nnz: int = 114_600_000, n_comm: int = 50,
                       p_in: float = 0.8, alpha: float = 2.0, max_deg: int = 21_000,
                       seed: int = 0) -> Csr:
    """Planted communities with power-law degrees.

    Nodes get a community uniformly at random. Degrees ~ Pareto(alpha) scaled
    to sum to ``nnz`` and clipped at ``max_deg``. Each edge of row i picks,
    with probability ``p_in``, a uniform node of i's community, else a
    uniform node of the whole graph. Duplicates are redrawn uniformly over
    all nodes, which lowers the intra-community share of rows whose degree
    approaches their community's size.
    """
    rng = rng_for(seed, STREAM_GRAPH)
    comm = rng.integers(0, n_comm, n, dtype=np.int64)
    members = np.argsort(comm, kind="stable")
    sizes = np.bincount(comm, minlength=n_comm)
    starts = np.zeros(n_comm + 1, dtype=np.int64)
    np.cumsum(sizes, out=starts[1:])
    deg = (rng.pareto(alpha, n) + 1.0)
    d = _rescale_degrees(deg, nnz, max_deg, rng)

    def draw(rows, g):
        inside = g.random(rows.shape[0]) < p_in
        cr = comm[rows]
        pick = starts[cr] + (g.random(rows.shape[0]) * sizes[cr]).astype(np.int64)
        pick = np.minimum(pick, starts[cr + 1] - 1)
        return np.where(inside, members[pick], g.integers(0, n, rows.shape[0], dtype=np.int64))

    return csr_from_degrees(d, n, rng, draw)


def uniform_vals(csr: Csr, seed: int = 0) -> np.ndarray:
    """Edge values U[-1, 1] in float32."""
    rng = rng_for(seed, STREAM_VALS)
    return rng.uniform(-1.0, 1.0, csr.nnz).astype(np.float32)


def mean_vals(csr: Csr) -> np.ndarray:
    """Edge values 1/deg(dst) (mean aggregation), float32."""
    deg = csr.degrees()
    inv = np.zeros_like(deg, dtype=np.float64)
    nz = deg > 0
    inv[nz] = 1.0 / deg[nz]
    return np.repeat(inv, deg).astype(np.float32)


def normal(n: int, f: int, seed: int = 0, stream: int = STREAM_X) -> np.ndarray:
    """An n x f float32 matrix with N(0, 1) entries."""
    rng = rng_for(seed, stream)
    return rng.standard_normal((n, f), dtype=np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even); returns the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    out = ((b + rounding) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --- Named workloads -------------------------------------------------------

def tiny_er(seed: int = 0) -> Csr:
    """Erdos-Renyi, 4,096 nodes, average degree 16, edge values U[-1, 1]."""
    g = erdos_renyi(4096, 16.0, seed)
    return g.with_vals(uniform_vals(g, seed))


def attention_benchmark_shape(seed: int = 0) -> Csr:
    """The fused attention-aggregation benchmark shape: 384 nodes, average degree 18."""
    return erdos_renyi(384, 18.0, seed)


def rmat_skew(scale: int = 20, seed: int = 0) -> Csr:
    """R-MAT skew stress graph (a, b, c, d = 0.57, 0.19, 0.19, 0.05), edge values U[-1, 1]."""
    g = rmat(scale, 16, 0.57, 0.19, 0.19, seed)
    return g.with_vals(uniform_vals(g, seed))


def uniform_control(like: Csr, seed: int = 0) -> Csr:
    """Uniform-degree control graph with the same node and edge counts as ``like``."""
    g = uniform_degree(like.n_rows, like.nnz, seed)
    return g.with_vals(uniform_vals(g, seed))


def products_like(seed: int = 0, scale: float = 1.0) -> Csr:
    """Lognormal power-law graph shaped like OGBN-Products (mean aggregation)."""
    n = max(64, int(round(2_449_029 * scale)))
    g = lognormal_powerlaw(n, int(round(123_700_000 * scale)), 1.3,
                           max(64, int(round(17_000 * min(1.0, scale ** 0.5)))), seed)
    return g.with_vals(mean_vals(g))


def reddit_like(seed: int = 0, scale: float = 1.0) -> Csr:
    """Power-law graph with 50 planted communities shaped like Reddit, edge values U[-1, 1]."""
    n = max(256, int(round(232_965 * scale)))
    g = community_powerlaw(n, int(round(114_600_000 * scale)), 50, 0.8, 2.0,
                           max(64, min(n, int(round(21_000 * scale ** 0.5)))), seed)
    return g.with_vals(uniform_vals(g, seed))
