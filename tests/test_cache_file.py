"""Persistent plan cache file handling on the host (no GPU): round trip,
bad header, corrupt and truncated lines are skipped with a status, never a crash."""
import os

import pytest


@pytest.fixture(scope="module")
def sga():
    from sparse_gnn_aggregation_gb300 import build
    build.build()
    import sparse_gnn_aggregation_gb300 as m
    return m


HEADER = "# autosage plan cache v1\n"
GOOD = "NVIDIA_GB300|sm152|op0|dt0|F64|H1|n10|m10|nnz20|fp00000000000000ab\tsplit 16 2 512 0.123000\n"


def test_round_trip(tmp_path, sga):
    sga.autosage_cache_clear()
    p = tmp_path / "c.txt"
    p.write_text(HEADER + GOOD)
    sga.autosage_cache_load(str(p))
    assert sga.autosage_cache_size() == 1
    q = tmp_path / "d.txt"
    sga.autosage_cache_save(str(q))
    assert q.read_text() == HEADER + GOOD
    sga.autosage_cache_clear()
    assert sga.autosage_cache_size() == 0


def test_per_edge_marker_round_trip(tmp_path, sga):
    # an SDDMM entry with per-edge reductions carries the optional `edge` marker
    sga.autosage_cache_clear()
    line = "NVIDIA_GB300|sm152|op2|dt0|F64|H1|n10|m10|nnz20|fp00000000000000ab\trowgroup 16 1 0 0.250000 edge\n"
    p = tmp_path / "c.txt"
    p.write_text(HEADER + GOOD + line)
    sga.autosage_cache_load(str(p))
    assert sga.autosage_cache_size() == 2
    q = tmp_path / "d.txt"
    sga.autosage_cache_save(str(q))
    assert sorted(q.read_text().splitlines()[1:]) == sorted([GOOD.strip(), line.strip()])
    sga.autosage_cache_clear()


def test_hybrid_schedule_round_trip(tmp_path, sga):
    # the ELL + CSR schedule family is stored by name like the others
    sga.autosage_cache_clear()
    line = "NVIDIA_GB300|sm152|op0|dt0|F4|H1|n10|m10|nnz20|fp00000000000000ab\thybrid 1 4 512 0.050000\n"
    p = tmp_path / "c.txt"
    p.write_text(HEADER + line)
    sga.autosage_cache_load(str(p))
    assert sga.autosage_cache_size() == 1
    q = tmp_path / "d.txt"
    sga.autosage_cache_save(str(q))
    assert q.read_text() == HEADER + line
    sga.autosage_cache_clear()


def test_aggregation_lanes_marker_round_trip(tmp_path, sga):
    # unfused attention whose aggregation stage runs with its own feature lanes
    # carries the optional `agg=G` marker (alone or after `edge`)
    sga.autosage_cache_clear()
    line = "NVIDIA_GB300|sm152|op4|dt1|F64|H8|n10|m10|nnz20|fp00000000000000ab\tbinned 16 1 512 5.740000 agg=32\n"
    p = tmp_path / "c.txt"
    p.write_text(HEADER + line)
    sga.autosage_cache_load(str(p))
    assert sga.autosage_cache_size() == 1
    q = tmp_path / "d.txt"
    sga.autosage_cache_save(str(q))
    assert q.read_text() == HEADER + line
    sga.autosage_cache_clear()


def test_wrong_header_rejected(tmp_path, sga):
    sga.autosage_cache_clear()
    p = tmp_path / "c.txt"
    p.write_text("# autosage plan cache v0\n" + GOOD)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_cache_load(str(p))
    assert e.value.status == sga.ERR_CACHE_FORMAT
    assert sga.autosage_cache_size() == 0


@pytest.mark.parametrize("bad", [
    "no-tab-here split 16 2 512 0.1\n",
    "key\tsplit 16 2\n",                       # truncated
    "key\twarp 16 2 512 0.1\n",                # unknown schedule
    "key\tbinned 16 2 0 0.1\n",                # binned schedule without a chunk length
    "key\trowgroup 3 1 0 0.1\n",               # lanes not a power of two
    "key\tsplit 16 4 0 0.1\n",                 # split schedule without a chunk length
    "key\trowgroup 16 4 0 0.1 extra\n",        # trailing field
    "key\trowgroup 16 4 0 0.1 edge edge\n",    # marker twice
    "key\trowgroup 16 1 0 0.1 agg=24\n",       # aggregation lanes not a power of two
    "key\trowgroup 16 1 0 0.1 agg=64\n",       # more aggregation lanes than a warp
    "key\trowgroup 16 1 0 0.1 agg=16x\n",      # not a number
    "key\trowgroup 16 1 0 0.1 agg=16 agg=32\n",  # marker twice
    "\tsplit 16 2 512 0.1\n",                  # empty key
])
def test_corrupt_lines_are_skipped(tmp_path, sga, bad):
    sga.autosage_cache_clear()
    p = tmp_path / "c.txt"
    p.write_text(HEADER + bad + GOOD)
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_cache_load(str(p))
    assert e.value.status == sga.ERR_CACHE_FORMAT
    assert sga.autosage_cache_size() == 1  # the good line still loaded


def test_truncated_file_and_missing_file(tmp_path, sga):
    sga.autosage_cache_clear()
    p = tmp_path / "c.txt"
    p.write_text(HEADER + GOOD[: len(GOOD) // 2])
    with pytest.raises(sga.AutosageError):
        sga.autosage_cache_load(str(p))
    assert sga.autosage_cache_size() == 0
    with pytest.raises(sga.AutosageError) as e:
        sga.autosage_cache_load(str(tmp_path / "missing.txt"))
    assert e.value.status == sga.ERR_CACHE_IO


def test_save_is_atomic_replace(tmp_path, sga):
    sga.autosage_cache_clear()
    p = tmp_path / "c.txt"
    p.write_text(HEADER + GOOD)
    sga.autosage_cache_load(str(p))
    sga.autosage_cache_save(str(p))
    assert not os.path.exists(str(p) + ".tmp")
    assert p.read_text() == HEADER + GOOD
