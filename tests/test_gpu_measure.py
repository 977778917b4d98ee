"""The gather-rate measurement that bench.py uses for its cache-aware bound:
rows gathered from an L2-resident table come faster than from a table far
larger than L2, and both rates are plausible for one GPU."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

import sparse_gnn_aggregation_gb300 as sga  # noqa: E402


def test_l2_resident_gathers_beat_dram_gathers():
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    hot = sga.autosage_measure_gather(l2 // 3, 2048, 1 << 21, 3)
    cold = sga.autosage_measure_gather(16 * l2, 2048, 1 << 21, 3)
    print(f"gather rates: L2-resident {hot:.0f} GB/s, DRAM-sized {cold:.0f} GB/s")
    assert 500 < cold < 50_000 and 500 < hot < 100_000, (hot, cold)
    assert hot > 1.3 * cold, (hot, cold)


@pytest.mark.parametrize("row_bytes", [16, 48, 512, 4096])
def test_row_widths(row_bytes):
    assert sga.autosage_measure_gather(64 << 20, row_bytes, 1 << 18, 1) > 0
