"""bench.py pieces that run without a GPU: the reference (oracle) arm's JSON
line on a small graph, and the algorithmic byte formulas."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--scale", "11",
                          "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_algorithmic_bytes():
    # SpMM: row_ptr + col_idx + vals + gathered rows + output rows
    assert bench.spmm_bytes(10, 100, 4, 4) == 44 + 800 + 1600 + 160
    # SDDMM: row_ptr + col_idx + Q rows + gathered K rows + scores
    assert bench.sddmm_bytes(10, 100, 4, 4) == 44 + 400 + 160 + 1600 + 400
    fused = bench.attn_bytes(10, 100, 2, 8, 2, True)
    assert fused == 44 + 400 + 2 * 10 * 16 * 2 + 2 * 100 * 16 * 2
    assert bench.attn_bytes(10, 100, 2, 8, 2, False) == fused + 5 * 4 * 100 * 2
    ops = bench.op_list({"rmat": None, "uniform": None})
    assert len(ops) == 2 * 2 * len(bench.FS) + 3
    assert [k for k, *_ in ops][-3:] == ["spmm_t/rmat/F64", "attn_fused/rmat/H8D64", "attn_unfused/rmat/H8D64"]


def test_cache_aware_bound():
    gp = {"l2_GBps": 20000.0, "dram_GBps": 8000.0}
    # DRAM side: 8 GB of DRAM bytes at 8 TB/s is 1 ms; 10 GB through L2 at 20 TB/s is 0.5 ms
    bound, frac = bench.cache_bound(10e9, 8e9, 2.0, gp)
    assert bound == 1.0 and frac == 0.5
    # L2 side: 40 GB through L2 at 20 TB/s is 2 ms, more than 1 ms of DRAM
    bound, frac = bench.cache_bound(40e9, 8e9, 4.0, gp)
    assert bound == 2.0 and frac == 0.5
    # no DRAM count or no measured rates: no bound
    assert bench.cache_bound(10e9, None, 2.0, gp) == (None, None)
    assert bench.cache_bound(10e9, 8e9, 2.0, None) == (None, None)


def test_roofline_entry_fields(monkeypatch):
    per_op = {"attn_fused/rmat/H8D64": {"ms": 2.0}}
    monkeypatch.setattr(bench, "traffic_for", lambda key: 4e9)
    gp = {"l2_GBps": 20000.0, "dram_GBps": 8000.0, "row_bytes": 2048}
    e = bench.roofline_entry("attn_fused/rmat/H8D64", per_op, 10000.0, 6746.6, "measured", gp)
    assert e["bound"] == "hbm" and e["unit"] == "GB/s" and e["peak"] == 6746.6
    assert e["frac"] == round(10000.0 / 6746.6, 4)
    assert e["traffic"] == 4e9 and e["traffic_GBps"] == 2000.0
    assert e["l2_frac"] == 0.5
    # 20 GB of algorithmic bytes: 1 ms through L2, 0.5 ms of DRAM -> bound 1 ms of 2 ms
    assert e["cache_aware_bound_ms"] == 1.0 and e["cache_aware_frac"] == 0.5
    assert "gather_peaks" not in bench.roofline_entry("attn_fused/rmat/H8D64", per_op, 10000.0, 6746.6, "measured")


def test_backward_bytes_count_the_transpose_structure_once():
    n, m, nnz, H, D, s = 10, 12, 100, 2, 8, 2
    W = H * D
    rows = 4 * (n + 1) + 4 * nnz + 3 * n * W * s + 2 * nnz * W * s + 16 * nnz * H + 4 * nnz + 8 * nnz * H
    # A^T's row_ptr and col_idx once; per product: weights, gathered rows, output rows
    want = rows + 4 * (m + 1) + 4 * nnz + 2 * (4 * nnz * H + nnz * W * s + m * W * s)
    assert bench.attn_backward_bytes(n, m, nnz, H, D, s) == want
