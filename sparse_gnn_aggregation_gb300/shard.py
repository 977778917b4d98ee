"""Row-sharded aggregation over several GPUs, one process per GPU.

Every operation of the library is defined per destination row (AutoSAGE,
"Input-Aware CUDA Scheduling for Sparse GNN Aggregation (SpMM/SDDMM) and CSR
Attention", Abstract; benchmark page "fused sparse attention-value
aggregation", problem statement: an output row per destination node from its
incoming edges), so contiguous row ranges are independent units:

* partition: rank r takes rows ``bounds[r]:bounds[r+1]``, ranges of about
  equal edge count (``autosage_partition_rows``, host side, once per graph);
* ownership: the feature rows of the input matrix are split by the same
  kind of bounds (node i's features live with the process that owns row i
  of the matrix whose rows they are);
* halo: the distinct columns a shard's edges reference, and the shard's CSR
  renumbered to address them by position (``autosage_shard_halo``);
* exchange: the one data-path step -- an all-gather of the owned row blocks
  (``torch.distributed``; NCCL between GPUs, gloo on the CPU), after which the
  halo rows are packed into a dense matrix on the GPU (``autosage_gather_rows``);
* compute: the unchanged ops on the shard's CSR; the outputs are the shard's
  own rows, so nothing is reduced afterwards.

SpMM with A^T shards the rows of A^T (A's columns), built once from A. This
module only arranges data and calls the library's C ABI; every step of the
aggregation runs in the library's kernels.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import CsrMatrix, autosage_gather_rows, autosage_partition_rows, autosage_shard_halo


@dataclasses.dataclass
class Shard:
    """One process's part of a CSR graph (host arrays)."""

    rank: int
    world: int
    bounds: np.ndarray     # int64 [world + 1]: rank k owns rows bounds[k]:bounds[k+1]
    row_ptr: np.ndarray    # int32 [rows + 1], rebased to start at 0
    local_col: np.ndarray  # int32 [shard nnz]: position of each edge's column in halo
    vals: np.ndarray | None
    halo: np.ndarray       # int32: the referenced global columns, increasing
    n_cols: int            # columns of the whole graph

    @property
    def row_begin(self) -> int:
        return int(self.bounds[self.rank])

    @property
    def row_end(self) -> int:
        return int(self.bounds[self.rank + 1])

    @property
    def n_rows(self) -> int:
        return self.row_end - self.row_begin

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    def csr(self, device="cuda") -> CsrMatrix:
        """The shard's CSR on the device: its rows, columns renumbered into the halo."""
        return CsrMatrix.from_numpy(self.row_ptr, self.local_col, self.vals, max(int(self.halo.size), 0), device)


def make_shard(row_ptr, col_idx, vals, n_cols: int, rank: int, world: int, bounds=None) -> Shard:
    """Rank ``rank``'s shard of a HOST CSR split into ``world`` equal-nnz row ranges."""
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int32)
    if bounds is None:
        bounds = autosage_partition_rows(row_ptr, world)
    b, e = int(bounds[rank]), int(bounds[rank + 1])
    halo, local = autosage_shard_halo(row_ptr, col_idx, n_cols, b, e)
    rp = (row_ptr[b:e + 1] - row_ptr[b]).astype(np.int32)
    v = None if vals is None else np.ascontiguousarray(vals[row_ptr[b]:row_ptr[e]], dtype=np.float32)
    return Shard(rank, world, np.asarray(bounds, dtype=np.int64), rp, local, v, halo, int(n_cols))


def exchange_rows(X_owned, bounds, group=None):
    """All-gather of the row blocks the ranks own: rank k holds rows
    ``bounds[k]:bounds[k+1]`` of a matrix; returns the whole matrix on every
    rank (on X_owned's device). Blocks are padded to the largest one for the
    collective and trimmed afterwards."""
    import torch
    import torch.distributed as dist

    world = len(bounds) - 1
    sizes = [int(bounds[k + 1] - bounds[k]) for k in range(world)]
    width = max(sizes) if sizes else 0
    F = int(X_owned.shape[1])
    pad = torch.zeros((width, F), dtype=X_owned.dtype, device=X_owned.device)
    pad[:X_owned.shape[0]] = X_owned
    blocks = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(blocks, pad, group=group)
    return torch.cat([blk[:n] for blk, n in zip(blocks, sizes)], dim=0)


def halo_rows(X_full, halo_idx, out=None):
    """Pack the halo rows X_full[halo] into a dense matrix on the GPU."""
    return autosage_gather_rows(X_full, halo_idx, out)


def transpose_host(row_ptr, col_idx, vals, n_cols: int, device="cuda"):
    """CSR of A^T, built by the library on the GPU and brought back to the host
    (the shards of SpMM with A^T are row ranges of A^T)."""
    from . import autosage_csr_transpose

    A = CsrMatrix.from_numpy(row_ptr, col_idx, vals, n_cols, device)
    rpt, cit, vt = autosage_csr_transpose(A)
    return (rpt.cpu().numpy(), cit.cpu().numpy(), None if vt is None else vt.cpu().numpy())
