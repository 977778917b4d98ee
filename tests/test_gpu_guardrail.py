"""The guardrail and the plan cache across processes (GPU). Failures are
injected on the host (AUTOSAGE_FAULT) in a child process; no GPU fault,
trap or hang is involved."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import oracle, synth
import sparse_gnn_aggregation_gb300 as sga
g = synth.rmat_skew(12, seed=4)
A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
X = torch.from_numpy(synth.normal(g.n_cols, 32, 4, synth.STREAM_X)).cuda()
mode = sys.argv[2]
if mode == "load":
    sga.autosage_cache_load(sys.argv[3])
plan = sga.autosage_plan(A, sga.OP_SPMM, 32, flags=sga.PLAN_PROBE | sga.PLAN_VERIFY, allow_probe_failure=True)
Y = sga.autosage_spmm(A, X, plan=plan)
ref = oracle.spmm(g.row_ptr, g.col_idx, g.vals, X.cpu().numpy())
err = float(np.max(np.abs(Y.cpu().numpy() - ref) / (1 + np.abs(ref))))
if mode == "save":
    sga.autosage_cache_save(sys.argv[3])
print(json.dumps({"schedule": plan.schedule(), "describe": plan.describe(), "err": err,
                  "checksum": float(Y.double().sum().item()),
                  "bits": Y.cpu().numpy().view(np.uint32).astype(np.uint64).sum().item()}))
"""


def child(mode, path="", env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    out = subprocess.run([sys.executable, "-c", CHILD, ROOT, mode, path], capture_output=True, text=True,
                         env=env, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return json.loads(out.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("fault", ["probe_fail", "verify_fail"])
def test_injected_failures_fall_back_to_the_default_schedule(fault):
    r = child("plain", env_extra={"AUTOSAGE_FAULT": fault})
    assert r["schedule"]["kind"] == 0 and r["schedule"]["lanes_f"] == 0  # the row-group default
    assert r["err"] <= 1e-4


def test_cache_replays_the_same_schedule_and_bits_in_a_new_process(tmp_path):
    path = str(tmp_path / "plans.txt")
    first = child("save", path)
    again = child("load", path)
    assert "cache=1" in again["describe"]
    for k in ("kind", "lanes_f", "lanes_e", "split"):
        assert again["schedule"][k] == first["schedule"][k]
    assert again["bits"] == first["bits"]
    assert first["err"] <= 1e-4
