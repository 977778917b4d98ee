"""Row sharding on the CPU with two gloo ranks (no GPU).

Each rank takes an equal-nnz row range of the graph (the library's host-side
partition), computes its halo (the library's host-side halo and column
renumbering), receives the feature rows it needs through the one exchange
step (an all-gather of the row blocks the ranks own), and computes its rows;
the shard outputs are gathered and concatenated. The per-shard arithmetic
here is the oracle's (the library's kernels need a GPU; the GPU test runs
them on each shard), so the concatenation must equal the whole-graph oracle
bit for bit: the shards keep every row's edges in order. SpMM with A^T is
sharded over the rows of A^T. The partition and halo are also checked
against their definitions.
"""
import os
import shutil
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from sparse_gnn_aggregation_gb300 import build
    build.build()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _graph():
    import synth
    g = synth.rmat_skew(10, seed=5)
    return g.with_vals(synth.uniform_vals(g, 5))


def _gather_rows_to_all(Y, world):
    sizes = torch.tensor([Y.shape[0]], dtype=torch.int64)
    all_sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(all_sizes, sizes)
    width = int(max(s.item() for s in all_sizes))
    pad = torch.zeros((width,) + tuple(Y.shape[1:]), dtype=Y.dtype)
    pad[:Y.shape[0]] = Y
    blocks = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(blocks, pad)
    return torch.cat([b[:int(n.item())] for b, n in zip(blocks, all_sizes)])


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    from sparse_gnn_aggregation_gb300 import shard as sh

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        g = _graph()
        F, H, D = 6, 2, 4
        X = synth.normal(g.n_cols, F, 5, synth.STREAM_X)
        Q = synth.normal(g.n_rows, H * D, 5, synth.STREAM_Q)
        K = synth.normal(g.n_cols, H * D, 5, synth.STREAM_K)
        V = synth.normal(g.n_cols, H * D, 5, synth.STREAM_V)
        s = sh.make_shard(g.row_ptr, g.col_idx, g.vals, g.n_cols, rank, world)
        b, e = s.row_begin, s.row_end
        # the exchange: every rank contributes the node rows it owns
        Xf = sh.exchange_rows(torch.from_numpy(X[b:e]), s.bounds).numpy()
        Kf = sh.exchange_rows(torch.from_numpy(K[b:e]), s.bounds).numpy()
        Vf = sh.exchange_rows(torch.from_numpy(V[b:e]), s.bounds).numpy()
        exchanged = bool(np.array_equal(Xf, X) and np.array_equal(Kf, K) and np.array_equal(Vf, V))
        # the shard's rows from its halo rows only
        Y = oracle.spmm(s.row_ptr, s.local_col, s.vals, Xf[s.halo])
        S = oracle.sddmm(s.row_ptr, s.local_col, Q[b:e], Kf[s.halo], 0.7)
        O = oracle.csr_attention(s.row_ptr, s.local_col, Q[b:e], Kf[s.halo], Vf[s.halo], H, 0.5)
        # SpMM with A^T: shards of A^T's rows; the input rows are owned by A's row partition
        G = synth.normal(g.n_rows, F, 5, synth.STREAM_G)
        rpt, cit, vt = oracle.transpose(g.row_ptr, g.col_idx, g.vals, g.n_cols)
        st = sh.make_shard(rpt, cit, vt, g.n_rows, rank, world)
        Gf = sh.exchange_rows(torch.from_numpy(G[b:e]), s.bounds).numpy()
        GX = oracle.spmm(st.row_ptr, st.local_col, st.vals, Gf[st.halo])
        res = {
            "bounds": s.bounds.tolist(), "bounds_t": st.bounds.tolist(), "exchanged": exchanged,
            "halo_ok": bool(np.array_equal(s.halo, np.unique(g.col_idx[g.row_ptr[b]:g.row_ptr[e]]))
                            and np.array_equal(s.halo[s.local_col], g.col_idx[g.row_ptr[b]:g.row_ptr[e]])),
            "Y": _gather_rows_to_all(torch.from_numpy(Y), world).numpy(),
            "S": _gather_rows_to_all(torch.from_numpy(S), world).numpy(),
            "O": _gather_rows_to_all(torch.from_numpy(O), world).numpy(),
            "GX": _gather_rows_to_all(torch.from_numpy(GX), world).numpy(),
        }
        if rank == 0:
            out.update(res)
        else:
            out[f"halo_ok_{rank}"] = res["halo_ok"]
            out[f"exchanged_{rank}"] = res["exchanged"]
    finally:
        dist.destroy_process_group()


def test_two_rank_shards_concatenate_to_the_whole_graph():
    import oracle
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    g = _graph()
    import synth
    F, H, D = 6, 2, 4
    X = synth.normal(g.n_cols, F, 5, synth.STREAM_X)
    Q = synth.normal(g.n_rows, H * D, 5, synth.STREAM_Q)
    K = synth.normal(g.n_cols, H * D, 5, synth.STREAM_K)
    V = synth.normal(g.n_cols, H * D, 5, synth.STREAM_V)
    G = synth.normal(g.n_rows, F, 5, synth.STREAM_G)
    assert res["exchanged"] and res["exchanged_1"], "the all-gather did not rebuild the owned rows"
    assert res["halo_ok"] and res["halo_ok_1"], "halo is not the sorted set of referenced columns"
    np.testing.assert_array_equal(res["Y"], oracle.spmm(g.row_ptr, g.col_idx, g.vals, X))
    np.testing.assert_array_equal(res["S"], oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 0.7))
    np.testing.assert_array_equal(res["O"], oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, H, 0.5))
    np.testing.assert_array_equal(res["GX"], oracle.spmm_t(g.row_ptr, g.col_idx, g.vals, G, g.n_cols))
    for key in ("bounds", "bounds_t"):
        bnd = res[key]
        assert bnd[0] == 0 and bnd[-1] == (g.n_rows if key == "bounds" else g.n_cols)
        assert all(a <= c for a, c in zip(bnd, bnd[1:]))


def test_partition_balances_edges_and_covers_rows():
    import synth
    import sparse_gnn_aggregation_gb300 as sga
    g = synth.rmat_skew(12, seed=2)
    deg = g.degrees()
    for parts in (1, 2, 3, 8, 64):
        bnd = sga.autosage_partition_rows(g.row_ptr, parts)
        assert bnd[0] == 0 and bnd[-1] == g.n_rows and np.all(np.diff(bnd) >= 0)
        per = np.array([g.row_ptr[bnd[k + 1]] - g.row_ptr[bnd[k]] for k in range(parts)])
        assert per.sum() == g.nnz
        # each cut lands at the first row starting at or past k/parts of the edges,
        # so a part exceeds its share by less than one row
        assert per.max() <= -(-g.nnz // parts) + deg.max()
    # an empty graph, more parts than rows, and a broken row_ptr
    assert list(sga.autosage_partition_rows(np.zeros(4, np.int32), 2)) == [0, 0, 3]
    assert list(sga.autosage_partition_rows(np.array([0, 5], np.int32), 3)) == [0, 1, 1, 1]
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_partition_rows(np.array([0, 3, 2], np.int32), 2)
    assert e.value.status == sga.ERR_INVALID_CSR


def test_halo_renumbers_edges_and_rejects_bad_columns():
    import sparse_gnn_aggregation_gb300 as sga
    rp = np.array([0, 2, 5, 6], np.int32)
    ci = np.array([7, 3, 3, 9, 1, 4], np.int32)
    halo, local = sga.autosage_shard_halo(rp, ci, 10, 1, 3)
    assert list(halo) == [1, 3, 4, 9]
    assert list(halo[local]) == [3, 9, 1, 4]
    halo, local = sga.autosage_shard_halo(rp, ci, 10, 1, 1)  # an empty shard
    assert halo.size == 0 and local.size == 0
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_shard_halo(rp, ci, 8, 0, 3)  # column 9 >= n_cols
    assert e.value.status == sga.ERR_INVALID_CSR
