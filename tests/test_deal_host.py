"""The item deal's run table (host logic in csrc/common.cuh), checked on the
CPU: a host-only program compiled with nvcc replays the block -> item mapping
and checks that every item is dealt exactly once with the documented runs."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_gnn_aggregation_gb300", "csrc")


def test_deal_table_covers_every_item_once(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "deal_check"
    src = os.path.join(ROOT, "tests", "native", "deal_check.cu")
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, src, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip().endswith("OK"), out.stdout[-2000:]
