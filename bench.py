"""Benchmark: SpMM / SDDMM / CSR attention on the R-MAT skew-stress workload.

One step is one pass over every hot-path operation on R-MAT scale 20
(1,048,576 nodes, edge factor 16, a,b,c,d = 0.57,0.19,0.19,0.05,
duplicates merged) and its uniform-degree control graph of equal nnz:
  SpMM and SDDMM at F in {4, 8, 16, 32, 64, 128, 256} on both graphs (fp32),
  SpMM with A^T at F = 64 (R-MAT), and CSR attention on R-MAT with 8 heads
  of width 64 in bf16, fused and unfused (SDDMM -> row softmax -> SpMM).
Schedules come from the planner (estimate + on-device probes), built
before the timed region. L2 is flushed (a 2x-L2 buffer is overwritten)
before every operation; each operation is timed with CUDA events on the
stream it runs on, so the flush is outside the timed spans.

value = algorithmic bytes of the step / summed operation time (GB/s).
Algorithmic bytes per operation (CSR arrays + gathered rows + outputs):
  SpMM:   4(N+1) + 8 nnz + nnz F s + N F s
  SDDMM:  4(N+1) + 4 nnz + N F s + nnz F s + 4 nnz
  fused attention: 4(N+1) + 4 nnz + 2 N H D s + 2 nnz H D s
  unfused attention: the fused bytes + 5 * 4 nnz H (scores written, read
                     twice and written by the softmax, read by the SpMM)

Cache-aware bound: the rates of random 2 KB row gathers from an L2-resident
table and from one 16x L2 are measured first (autosage_measure_gather). An
operation needs at least max(DRAM bytes / DRAM gather rate, algorithmic
bytes / L2 gather rate), with its DRAM bytes from profiles/traffic.txt (an
ncu count); per_op and roofline report that bound and its fraction of the
measured time (cache_aware_frac), beside the plain fraction of the HBM peak.

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
row sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

FS = [4, 8, 16, 32, 64, 128, 256]
HEADS, HEAD_DIM = 8, 64
METRIC = "SpMM/SDDMM/CSR-attn achieved HBM GB/s (% of ~8 TB/s) and nnz·F/s on 1 GB300"
WORKLOAD = "R-MAT s20 ef16 + uniform control: SpMM/SDDMM F4-256 f32, SpMM^T F64, bf16 attn H8 D64"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


KERNEL_FILES = {
    "spmm": ["spmm.cu", "common.cuh"],
    "spmm_t": ["spmm.cu", "graph.cu", "common.cuh"],
    "sddmm": ["sddmm.cu", "common.cuh"],
    "attn_fused": ["attention.cu", "common.cuh"],
    "attn_unfused": ["sddmm.cu", "softmax.cu", "spmm.cu", "common.cuh"],
}


def source_hash(files=None) -> str:
    """Hash of kernel sources (all of csrc/, or the listed files)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_gnn_aggregation_gb300", "csrc")
    for f in sorted(files or os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def kernel_hash(op_key: str) -> str:
    """Hash of the sources that define the kernels of an operation key like 'attn_fused/rmat/H8D64'."""
    return source_hash(KERNEL_FILES.get(op_key.split("/")[0]))


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_for(op_key: str):
    """DRAM bytes per launch from profiles/traffic.txt (null when the kernels changed since)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_hash(op_key)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and parts[0] == op_key and parts[2] == cur:
                return float(parts[1])
    return None


def gather_peaks(dev):
    """Measured read rates of random row gathers on this GPU (the library's
    autosage_measure_gather): from an L2-resident table (a third of L2), the rate
    at which L2 serves hot gathered rows, and from a table of 16x L2, the DRAM
    rate of the same access pattern. Rows of 2 KB (one warp each): the
    fastest row size measured (1 KB rows: 15.6 and 6.1 TB/s, 2 KB: 19.4 and
    7.2 TB/s on a GB300), so the rates are ceilings for the 1 KB rows of the
    widest operations."""
    import torch
    import sparse_gnn_aggregation_gb300 as sga
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    return {"l2_GBps": round(sga.autosage_measure_gather(l2 // 3, 2048, 1 << 23, 5), 1),
            "dram_GBps": round(sga.autosage_measure_gather(16 * l2, 2048, 1 << 23, 5), 1),
            "row_bytes": 2048, "table_bytes": [l2 // 3, 16 * l2]}


def cache_bound(op_bytes_, traffic, ms, gp):
    """Cache-aware bound of one operation: every algorithmic byte passes through
    L2 (at most the L2 gather rate) and the DRAM bytes ncu counted come from HBM
    (at most the DRAM gather rate), so the operation needs at least the larger
    of the two times. Returns (bound_ms, bound_ms / ms), or Nones without the
    DRAM count."""
    if not traffic or not gp:
        return None, None
    t = max(traffic / (gp["dram_GBps"] * 1e6), op_bytes_ / (gp["l2_GBps"] * 1e6))
    return round(t, 4), round(t / ms, 4)


def roofline_entry(dom_key, per_op, achieved, peak, peak_src, gp=None):
    """The dominant operation against the measured HBM peak: `achieved` counts
    algorithmic bytes (L2 hits included); `traffic` is the DRAM bytes of one
    launch from profiles/traffic.txt (null once its kernels changed), and
    traffic_GBps / traffic_frac the DRAM rate those bytes give at the bench's
    time: what the launch really asks of HBM. With the measured gather rates
    (gp): l2_frac = achieved / the L2 gather rate, and cache_aware_frac = the
    cache-aware bound (cache_bound) / the measured time."""
    if not dom_key:
        return {"bound": "hbm", "kernel": None, "achieved": None, "peak": peak, "unit": "GB/s", "frac": None,
                "traffic": None}
    traffic = traffic_for(dom_key)
    e = {"bound": "hbm", "kernel": dom_key, "achieved": achieved, "peak": peak,
         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)",
         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic}
    if traffic:
        gbs = traffic / per_op[dom_key]["ms"] / 1e6
        e["traffic_GBps"] = round(gbs, 1)
        e["traffic_frac"] = round(gbs / peak, 4)
    if gp:
        e["gather_peaks"] = gp
        e["l2_frac"] = round(achieved / gp["l2_GBps"], 4)
        ms = per_op[dom_key]["ms"]
        e["cache_aware_bound_ms"], e["cache_aware_frac"] = cache_bound(achieved * ms * 1e6, traffic, ms, gp)
    return e


# ---------------------------------------------------------------- workload

def build_graphs(scale: int = 20):
    rm = synth.rmat_skew(scale, seed=0)
    un = synth.uniform_control(rm, seed=0)
    return {"rmat": rm, "uniform": un}


def spmm_bytes(n, nnz, F, s):
    return 4 * (n + 1) + 8 * nnz + nnz * F * s + n * F * s


def sddmm_bytes(n, nnz, F, s):
    return 4 * (n + 1) + 4 * nnz + n * F * s + nnz * F * s + 4 * nnz


def attn_bytes(n, nnz, H, D, s, fused):
    b = 4 * (n + 1) + 4 * nnz + 2 * n * H * D * s + 2 * nnz * H * D * s
    if not fused:
        b += 5 * 4 * nnz * H
    return b


def attn_backward_bytes(n, m, nnz, H, D, s):
    """Algorithmic bytes of one CSR-attention backward: the one pass over the
    rows of A (CSR arrays, Q and dO rows once per row, K and V rows gathered
    per edge, dQ written, scores and dW written and read back per edge and
    head, the A^T position of each edge read, w and dS written in A^T order)
    and the two SpMMs over A^T for dV and dK (A^T's CSR arrays once, then for
    each product its per-head weights, its gathered dO or Q rows and its
    output)."""
    W = H * D
    rows = 4 * (n + 1) + 4 * nnz + 3 * n * W * s + 2 * nnz * W * s + 4 * 4 * nnz * H + 4 * nnz + 2 * 4 * nnz * H
    csr_t = 4 * (m + 1) + 4 * nnz
    product = 4 * nnz * H + nnz * W * s + m * W * s
    return rows + csr_t + 2 * product


def workload_config(graphs, world):
    """The `config` object of both arms' lines (identical keys and values)."""
    rm, un = graphs["rmat"], graphs["uniform"]
    return {"workload": WORKLOAD, "nodes": rm.n_rows, "nnz_rmat": rm.nnz, "nnz_uniform": un.nnz,
            "max_degree_rmat": int(rm.degrees().max()),
            "l2": "GPU arm: a 2x-L2 buffer is overwritten before every operation, outside the timed spans",
            "parallelism": f"replicas x{world}"}


def op_list(graphs, only=None):
    """(key, kind, graph, F) in execution order; graphs alternate so the other
    graph's data sits between two uses of one CSR. `only` keeps keys containing it."""
    ops = []
    for F in FS:
        for gname in ("rmat", "uniform"):
            ops.append((f"spmm/{gname}/F{F}", "spmm", gname, F))
        for gname in ("rmat", "uniform"):
            ops.append((f"sddmm/{gname}/F{F}", "sddmm", gname, F))
    ops.append(("spmm_t/rmat/F64", "spmm_t", "rmat", 64))
    ops.append(("attn_fused/rmat/H8D64", "attn_fused", "rmat", HEAD_DIM))
    ops.append(("attn_unfused/rmat/H8D64", "attn_unfused", "rmat", HEAD_DIM))
    if only:
        ops = [o for o in ops if any(w in o[0] for w in only.split(","))]
    return ops


def op_bytes(kind, g, F):
    n, nnz = g.n_rows, g.nnz
    if kind in ("spmm", "spmm_t"):
        return spmm_bytes(n, nnz, F, 4), 2 * nnz * F
    if kind == "sddmm":
        return sddmm_bytes(n, nnz, F, 4), 2 * nnz * F
    fused = kind == "attn_fused"
    return attn_bytes(n, nnz, HEADS, HEAD_DIM, 2, fused), 2 * nnz * HEADS * HEAD_DIM


# ---------------------------------------------------------------- the two largest configs

def large_config_rows(dev, flush, stream, steps, warmup, oracle_frac=0.05):
    """Throughput on the products-like and Reddit-like graphs, measured like
    the step (L2 flushed before every launch, CUDA events on the launching
    stream, algorithmic bytes), with the oracle timed beside each operation
    on a seeded uniform sample of the rows (fraction ``oracle_frac``):
      products-like (2,449,029 nodes, 123.7M edges, mean aggregation):
        SpMM at F = 32 and 100, SpMM with A^T at F = 32 and 100 (fixed edge
        values, kept in A^T order by the plan) and at F = 32 with the values
        read per call (spmm_t_vpc), and the A^T build (once per plan) on its own;
      Reddit-like (232,965 nodes, 114.6M edges, 50 communities):
        SpMM at F = 128 and 602, SDDMM at F = 128."""
    import ctypes

    import torch

    import oracle
    import sparse_gnn_aggregation_gb300 as sga

    oracle.build()
    peak, _ = measured_peak()
    out = {}

    def timed(fn):
        for _ in range(warmup):
            flush.fill_(1.0)
            fn()
        evs = []
        for _ in range(steps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    def oracle_rate(kind, g, F, X, gt=None):
        rng = np.random.default_rng(54321)
        src = gt if kind.startswith("spmm_t") else g
        k = max(1, int(round(src.n_rows * oracle_frac)))
        rows = np.sort(rng.choice(src.n_rows, size=k, replace=False)).astype(np.int64)
        enn = int((src.row_ptr[rows + 1] - src.row_ptr[rows]).sum())
        t0 = time.perf_counter()
        if kind == "sddmm":
            oracle.sddmm(src.row_ptr, src.col_idx, X, X, 1.0, rows=rows)
            b = sddmm_bytes(rows.size, enn, F, 4)
        else:
            oracle.spmm(src.row_ptr, src.col_idx, src.vals, X, rows=rows)
            b = spmm_bytes(rows.size, enn, F, 4)
        dt = time.perf_counter() - t0
        return {"GBps": round(b / dt / 1e9, 3), "rows_sampled": int(rows.size), "s": round(dt, 3),
                "cores": oracle.threads()}

    flags = sga.PLAN_PROBE | sga.PLAN_VERIFY
    for gname, gen, ops in (("products", synth.products_like, [("spmm", 32), ("spmm", 100), ("spmm_t", 32),
                                                               ("spmm_t", 100), ("spmm_t_vpc", 32)]),
                            ("reddit", synth.reddit_like, [("spmm", 128), ("spmm", 602), ("sddmm", 128)])):
        g = gen(seed=0)
        A = sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols)
        gt = None
        if any(k.startswith("spmm_t") for k, _ in ops):
            rpt, cit, vt = oracle.transpose(g.row_ptr, g.col_idx, g.vals, g.n_cols)
            gt = synth.Csr(g.n_cols, g.n_rows, rpt, cit, vt)
            t_rp = torch.empty(g.n_cols + 1, dtype=torch.int32, device=dev)
            t_ci = torch.empty(g.nnz, dtype=torch.int32, device=dev)
            t_v = torch.empty(g.nnz, dtype=torch.float32, device=dev)
            lib = sga.library()
            ms = timed(lambda: lib.autosage_csr_transpose(A.c, ctypes.c_void_p(t_rp.data_ptr()),
                                                          ctypes.c_void_p(t_ci.data_ptr()),
                                                          ctypes.c_void_p(t_v.data_ptr()),
                                                          ctypes.c_void_p(stream.cuda_stream)))
            out[f"transpose_build/{gname}"] = {"ms": round(ms, 4), "note": "CSR of A^T (stable radix sort), "
                                               "built once per SpMM^T plan; not part of the SpMM^T rows"}
            del t_rp, t_ci, t_v
        for kind, F in ops:
            key = f"{kind}/{gname}/F{F}"
            if kind == "sddmm":
                Q = torch.randn(g.n_rows, F, device=dev)
                K = torch.randn(g.n_cols, F, device=dev)
                S = torch.empty(g.nnz, device=dev)
                plan = sga.autosage_plan(A, sga.OP_SDDMM, F, flags=flags)
                ms = timed(lambda: sga.autosage_sddmm(A, Q, K, 1.0, S, plan=plan))
                b = sddmm_bytes(g.n_rows, g.nnz, F, 4)
                del Q, K, S
            else:
                # mean aggregation's values are fixed: SpMM^T plans keep them in A^T order;
                # spmm_t_vpc reads them per call (gathered into A^T order at every call)
                tr = kind.startswith("spmm_t")
                X = torch.randn(g.n_rows if tr else g.n_cols, F, device=dev)
                Y = torch.empty(g.n_cols if tr else g.n_rows, F, device=dev)
                fl = flags | (sga.PLAN_FIXED_VALUES if kind == "spmm_t" else 0)
                plan = sga.autosage_plan(A, sga.OP_SPMM_T if tr else sga.OP_SPMM, F, flags=fl)
                ms = timed(lambda: sga.autosage_spmm(A, X, Y, transpose=tr, plan=plan))
                b = spmm_bytes(g.n_rows, g.nnz, F, 4)
                del X, Y
            Xh = np.random.default_rng(2).standard_normal((g.n_rows, F), dtype=np.float32)
            out[key] = {"ms": round(ms, 4), "GBps": round(b / ms / 1e6, 1),
                        "frac_of_hbm_peak": round(b / ms / 1e6 / peak, 4),
                        "nnzF_per_s": g.nnz * F / (ms * 1e-3), "bytes": int(b), "dtype": "f32",
                        "plan": plan.describe(), "oracle": oracle_rate(kind, g, F, Xh, gt)}
            del plan
        del A
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.idx = device_index
        self.out = os.path.join("/tmp", f"autosage_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        # nvidia-smi takes a moment to start: wait for its first sample so
        # that the samples cover the timed region that follows
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 3.0 and self.proc.poll() is None:
            if os.path.getsize(self.out) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for name, val in zip(names[1:], p[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.out)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- ranks

def aggregate_ranks(step_ms, step_bytes, world, device="cpu"):
    """Whole-job rate: every rank ran its own step (weak scaling, no data
    exchange); the job's step time is the slowest rank's, and the job moved
    world x step_bytes in it. Returns (max step ms, GB/s)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(step_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    return step_ms, (step_bytes * world / (step_ms * 1e-3) / 1e9 if step_ms > 0 else 0.0)


# ---------------------------------------------------------------- GPU arm

def run_ours(args):
    import torch

    import sparse_gnn_aggregation_gb300 as sga

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    graphs = build_graphs(args.scale)
    ops = op_list(graphs, args.only)
    stream = torch.cuda.current_stream()
    if args.cache and os.path.exists(args.cache):
        sga.autosage_cache_load(args.cache)
    mats = {k: sga.CsrMatrix.from_numpy(g.row_ptr, g.col_idx, g.vals, g.n_cols) for k, g in graphs.items()}
    # resident inputs (one per width so nothing is shared between operations)
    feats, host_feats = {}, {}
    for key, kind, gname, F in ops:
        g = graphs[gname]
        if kind in ("spmm", "spmm_t"):
            src = g.n_rows if kind == "spmm_t" else g.n_cols
            feats[key] = {"X": torch.randn(src, F, device=dev, generator=None)}
        elif kind == "sddmm":
            feats[key] = {"Q": torch.randn(g.n_rows, F, device=dev), "K": torch.randn(g.n_cols, F, device=dev)}
        else:
            W = HEADS * HEAD_DIM
            feats[key] = {t: torch.randn(g.n_rows, W, device=dev).to(torch.bfloat16) for t in ("Q", "K", "V")}
    outs = {}
    plans = {}
    flags = sga.PLAN_PROBE | sga.PLAN_VERIFY
    t_plan = time.perf_counter()
    for key, kind, gname, F in ops:
        A = mats[gname]
        if kind == "spmm":
            plans[key] = sga.autosage_plan(A, sga.OP_SPMM, F, flags=flags)
        elif kind == "spmm_t":
            # the step's edge values do not change: the plan keeps them in A^T order
            plans[key] = sga.autosage_plan(A, sga.OP_SPMM_T, F, flags=flags | sga.PLAN_FIXED_VALUES)
        elif kind == "sddmm":
            plans[key] = sga.autosage_plan(A, sga.OP_SDDMM, F, flags=flags)
        elif kind == "attn_fused":
            plans[key] = sga.autosage_plan(A, sga.OP_ATTN, F, heads=HEADS, dtype=torch.bfloat16, flags=flags)
        else:
            plans[key] = sga.autosage_plan(A, sga.OP_ATTN_UNFUSED, F, heads=HEADS, dtype=torch.bfloat16,
                                           flags=flags)
    plan_s = time.perf_counter() - t_plan
    if args.cache:
        sga.autosage_cache_save(args.cache)

    def run(key, kind, gname, F, f, out=None):
        A, P = mats[gname], plans[key]
        if kind == "spmm":
            return sga.autosage_spmm(A, f["X"], out, plan=P)
        if kind == "spmm_t":
            return sga.autosage_spmm(A, f["X"], out, transpose=True, plan=P)
        if kind == "sddmm":
            return sga.autosage_sddmm(A, f["Q"], f["K"], 1.0, out, plan=P)
        return sga.autosage_csr_attention(A, f["Q"], f["K"], f["V"], HEADS, 1.0 / 8.0,
                                          fused=(kind == "attn_fused"), out=out, plan=P)

    for key, kind, gname, F in ops:
        outs[key] = run(key, kind, gname, F, feats[key])
    torch.cuda.synchronize()

    # the gather-rate ceilings of this GPU (before the timed region)
    gpeaks = None if args.no_gather_peaks else gather_peaks(dev)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    ev = {key: [] for key, *_ in ops}

    def step(timed):
        for key, kind, gname, F in ops:
            flush.fill_(1.0)
            if timed:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                # an NVTX range per timed operation: a profiler can name the
                # operation's kernel launches by its key
                torch.cuda.nvtx.range_push(key)
            run(key, kind, gname, F, feats[key], outs[key])
            if timed:
                torch.cuda.nvtx.range_pop()
                e1.record(stream)
                ev[key].append((e0, e1))

    for _ in range(args.warmup):
        step(False)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for _ in range(args.steps):
        step(True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - w0
    clock_info = clocks.stop()

    # secondary figure: each operation again right after itself, L2 warm
    # (inputs that fit the 129 MB L2 stay there; not part of `value`)
    warm = {}
    for key, kind, gname, F in ops:
        run(key, kind, gname, F, feats[key], outs[key])
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run(key, kind, gname, F, feats[key], outs[key])
        e1.record(stream)
        warm[key] = (e0, e1)
    torch.cuda.synchronize()

    per_op = {}
    tot_ms, tot_bytes, tot_flops, tot_nnzF = 0.0, 0.0, 0.0, 0.0
    for key, kind, gname, F in ops:
        ms = [a.elapsed_time(b) for a, b in ev[key]]
        mean_ms = float(np.mean(ms))
        g = graphs[gname]
        b, fl = op_bytes(kind, g, F)
        width = F * (HEADS if kind.startswith("attn") else 1)
        warm_ms = warm[key][0].elapsed_time(warm[key][1])
        per_op[key] = {"ms": round(mean_ms, 5), "GBps": round(b / mean_ms / 1e6, 1),
                       "nnzF_per_s": g.nnz * width / (mean_ms * 1e-3),
                       "warm_l2_ms": round(warm_ms, 5), "plan": plans[key].describe()}
        tr = traffic_for(key)
        if tr:
            per_op[key]["dram_GBps"] = round(tr / mean_ms / 1e6, 1)
        if gpeaks:
            per_op[key]["l2_frac"] = round(b / mean_ms / 1e6 / gpeaks["l2_GBps"], 4)
            per_op[key]["cache_aware_bound_ms"], per_op[key]["cache_aware_frac"] = cache_bound(b, tr, mean_ms, gpeaks)
        tot_ms += mean_ms
        tot_bytes += b
        tot_flops += fl
        tot_nnzF += g.nnz * width
    step_ms, value = aggregate_ranks(tot_ms, tot_bytes, world, dev)

    # rows beyond the step: the CSR-attention backward on the same graph
    next_rows = {}
    if not args.no_next and (not args.only or "backward" in args.only.split(",")):
        g = graphs["rmat"]
        A = mats["rmat"]
        W = HEADS * HEAD_DIM
        bq, bk, bv, bo = (torch.randn(n, W, device=dev).to(torch.bfloat16)
                          for n in (g.n_rows, g.n_cols, g.n_cols, g.n_rows))
        bplan = sga.autosage_plan(A, sga.OP_ATTN_BACKWARD, HEAD_DIM, heads=HEADS, dtype=torch.bfloat16)
        outs_b = [torch.empty_like(bq), torch.empty_like(bk), torch.empty_like(bv)]
        for _ in range(args.warmup):
            flush.fill_(1.0)
            sga.autosage_csr_attention_backward(A, bq, bk, bv, bo, HEADS, 0.125, *outs_b, plan=bplan)
        times = []
        for _ in range(args.steps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            sga.autosage_csr_attention_backward(A, bq, bk, bv, bo, HEADS, 0.125, *outs_b, plan=bplan)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
        b = attn_backward_bytes(g.n_rows, g.n_cols, g.nnz, HEADS, HEAD_DIM, 2)
        peak_gbs, _ = measured_peak()
        next_rows["attn_backward/rmat/H8D64"] = {
            "ms": round(ms, 4), "GBps": round(b / ms / 1e6, 1), "frac_of_hbm_peak": round(b / ms / 1e6 / peak_gbs, 4),
            "bytes": int(b), "dtype": "bf16 in/out, f32 accumulate", "plan": bplan.describe()}
        del bq, bk, bv, bo, outs_b, bplan
    if not args.no_next and (not args.only or "typed" in args.only.split(",")):
        # multi-relation SpMM (RGCN-style): 4 relations, F = 64, fp32
        g = graphs["rmat"]
        A = mats["rmat"]
        R, F = 4, 64
        et = torch.from_numpy(synth.rng_for(0, 9).integers(0, R, g.nnz).astype(np.int32)).to(dev)
        Z = torch.randn(R, g.n_cols, F, device=dev)
        Yt = torch.empty(g.n_rows, F, device=dev)
        tplan = sga.autosage_plan_typed(A, et, R, F, flags=sga.PLAN_PROBE | sga.PLAN_VERIFY)
        for _ in range(args.warmup):
            flush.fill_(1.0)
            sga.autosage_spmm_typed(A, et, Z, Yt, plan=tplan)
        times = []
        for _ in range(args.steps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            sga.autosage_spmm_typed(A, et, Z, Yt, plan=tplan)
            e1.record(stream)
            times.append((e0, e1))
        torch.cuda.synchronize()
        ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
        b = spmm_bytes(g.n_rows, g.nnz, F, 4)
        peak_gbs, _ = measured_peak()
        next_rows["spmm_typed/rmat/R4F64"] = {
            "ms": round(ms, 4), "GBps": round(b / ms / 1e6, 1), "frac_of_hbm_peak": round(b / ms / 1e6 / peak_gbs, 4),
            "bytes": int(b), "dtype": "f32", "plan": tplan.describe()}
        del et, Z, Yt, tplan

    # the products-like and Reddit-like configs: throughput rows beside the step
    configs = {}
    if not args.no_configs and (not args.only or "configs" in args.only.split(",")):
        configs = large_config_rows(dev, flush, stream, args.steps, args.warmup)

    # dominant operation: the largest share of the step
    # (one main kernel per launch: the unfused pipeline is three kernels, so it is not a candidate)
    cands = [k for k in per_op if not k.startswith("attn_unfused")]
    dom_key = max(cands, key=lambda k: per_op[k]["ms"]) if cands else None
    peak, peak_src = measured_peak()
    achieved = per_op[dom_key]["GBps"] if dom_key else None

    # end to end through the public API with host buffers: H2D inputs, op, D2H output
    e2e = None
    if not args.skip_e2e:
        pinned_in = {k: {n: t.cpu().pin_memory() for n, t in f.items()} for k, f in feats.items()}
        pinned_out = {k: torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for k, o in outs.items()}
        dev_in = {k: {n: torch.empty_like(t) for n, t in f.items()} for k, f in feats.items()}
        h2d = sum(t.numel() * t.element_size() for f in pinned_in.values() for t in f.values())
        d2h = sum(t.numel() * t.element_size() for t in pinned_out.values())

        # three streams: host->device copies, the operations, device->host copies;
        # op k's inputs are copied while op k-1 runs and its output is read back
        # while op k+1 runs (every op has its own buffers, and events order the
        # reuse of those buffers from one step to the next)
        s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        n_ops = len(ops)
        ev_in = [torch.cuda.Event() for _ in range(n_ops)]
        ev_ran = [torch.cuda.Event() for _ in range(n_ops)]
        ev_read = [torch.cuda.Event() for _ in range(n_ops)]
        started = [False] * n_ops

        def e2e_step():
            for k, (key, kind, gname, F) in enumerate(ops):
                with torch.cuda.stream(s_in):
                    if started[k]:
                        s_in.wait_event(ev_ran[k])  # the previous step's op k has read its inputs
                    for n, t in pinned_in[key].items():
                        dev_in[key][n].copy_(t, non_blocking=True)
                    ev_in[k].record(s_in)
                with torch.cuda.stream(s_run):
                    s_run.wait_event(ev_in[k])
                    if started[k]:
                        s_run.wait_event(ev_read[k])  # the previous step's output has been read back
                    run(key, kind, gname, F, dev_in[key], outs[key])
                    ev_ran[k].record(s_run)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_ran[k])
                    pinned_out[key].copy_(outs[key], non_blocking=True)
                    ev_read[k].record(s_out)
                started[k] = True

        # warm-up as for the timed step: the first passes of the copy engines
        # over freshly pinned host buffers run slower than later ones (measured:
        # 192 ms per step over steps 2-3 against 124 ms over steps 4-5)
        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(1, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
        e2e = {"value": round(tot_bytes * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 3)}

    # launches inside the timed region (per step, our kernels only)
    def launches(key, kind):
        # SDDMM: one launch (every edge's score is finished in its own item);
        # SpMM: merge path + its fix-up, or the row kernel, a fix-up for cut rows
        # and (hybrid) the ELL slab's kernel; fused attention: the row kernel and
        # a fix-up for cut rows; unfused: SDDMM, the row softmax (with a merge and
        # a normalisation pass for cut rows) and the SpMM
        d = plans[key].describe()
        long_rows = int(d.split("long_rows=")[1].split()[0]) if "long_rows=" in d else 0
        cut = 1 if long_rows > 0 else 0
        if kind == "sddmm":
            return 1
        if "sched=mergepath" in d:
            spmm = 2
        else:
            spmm = 1 + cut + (1 if "sched=hybrid" in d else 0)
        if kind == "attn_fused":
            return 1 + cut
        if kind == "attn_unfused":
            return 1 + (1 + 2 * cut) + spmm
        return spmm

    n_launch = sum(launches(k, kind) for k, kind, *_ in ops) * args.steps

    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "wall_ms_per_step_incl_flush": round(wall * 1e3 / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 (F sweep, SpMM^T); bf16 in / f32 softmax+acc (attention)",
        "data": "synthetic",
        "config": workload_config(graphs, world),
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "nnzF_per_s": tot_nnzF * world / max(step_ms * 1e-3, 1e-12),
        "edges_per_s": sum(graphs[g].nnz for _, _, g, _ in ops) * world / max(step_ms * 1e-3, 1e-12),
        "roofline": roofline_entry(dom_key, per_op, achieved, peak, peak_src, gpeaks),
        "clocks": clock_info,
        "gpu_launches": n_launch,
        "plan_seconds": round(plan_s, 2),
        "per_op": per_op,
        "next": next_rows,
        "configs": configs,
        "source_hash": source_hash(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if args.scale != 20 or args.only:
        line["config"]["workload"] = f"PARTIAL (scale {args.scale}, only={args.only}); not the benchmark workload"
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(graphs, budget_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------- oracle arm

def cpu_baseline(graphs, budget_s=15.0, steps=1):
    """The oracle on the host cores over a row sample of the same operations.

    A seeded uniform sample of rows (fraction f of every graph) keeps the
    degree mix; f is chosen from a calibration pass so one pass takes about
    budget_s. Value = algorithmic bytes of the sampled rows / oracle time (GB/s).
    """
    import oracle

    oracle.build()
    ops = op_list(graphs)
    feats = {}
    samples = {}

    def sample(g, frac):
        key = (id(g), frac)
        if key not in samples:
            rng = np.random.default_rng(12345)
            k = max(1, min(g.n_rows, int(round(g.n_rows * frac))))
            rows = np.sort(rng.choice(g.n_rows, size=k, replace=False)).astype(np.int64)
            deg = (g.row_ptr[rows + 1] - g.row_ptr[rows]).astype(np.int64)
            samples[key] = (rows, int(deg.sum()))
        return samples[key]

    def one_pass(frac, per_op=None):
        tot_b, tot_t = 0.0, 0.0
        for key, kind, gname, F in ops:
            g = graphs[gname]
            rows, enn = sample(g, frac)
            if key not in feats:
                W = F * (HEADS if kind.startswith("attn") else 1)
                feats[key] = np.random.default_rng(1).standard_normal((g.n_cols, W), dtype=np.float32)
            X = feats[key]
            if kind == "spmm_t" and "T" not in feats:
                feats["T"] = oracle.transpose(g.row_ptr, g.col_idx, g.vals, g.n_cols)
            t0 = time.perf_counter()
            if kind == "spmm_t":
                rpt, cit, vt = feats["T"]
                oracle.spmm(rpt, cit, vt, X, rows=rows)
                b = 4 * (rows.size + 1) + 8 * enn + enn * F * 4 + rows.size * F * 4
            elif kind == "spmm":
                oracle.spmm(g.row_ptr, g.col_idx, g.vals, X, rows=rows)
                b = 4 * (rows.size + 1) + 8 * enn + enn * F * 4 + rows.size * F * 4
            elif kind == "sddmm":
                oracle.sddmm(g.row_ptr, g.col_idx, X, X, 1.0, rows=rows)
                b = 4 * (rows.size + 1) + 8 * enn + rows.size * F * 4 + enn * F * 4
            else:
                oracle.csr_attention(g.row_ptr, g.col_idx, X, X, X, HEADS, 0.125, rows=rows)
                b = attn_bytes(rows.size, enn, HEADS, HEAD_DIM, 2, kind == "attn_fused")
            dt = time.perf_counter() - t0
            if per_op is not None:
                per_op[key] = {"GBps": round(b / dt / 1e9, 3), "s": round(dt, 4)}
            tot_t += dt
            tot_b += b
        return tot_b, tot_t

    frac = 1.0 / 2048
    one_pass(frac)  # warm: features, transpose, thread pool
    per_op = {}
    b, t = one_pass(frac, per_op)
    # the time per row falls as the sample grows (fixed costs per call), so
    # rescale until a pass takes at least half the budget
    for _ in range(3):
        if t >= 0.5 * budget_s or frac >= 1.0:
            break
        frac = min(1.0, frac * budget_s / max(t, 1e-3))
        b, t = one_pass(frac, per_op)
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": oracle.threads(), "kind": "oracle",
            "sample": f"a seeded uniform {100 * frac:.2f}% of the rows of each graph for every operation of "
                      f"the step ({b / 1e9:.2f} GB algorithmic, {t:.1f} s)",
            "per_op": per_op, "single_core_ms": single_core_ms()}


def single_core_ms():
    """The oracle on one thread for the two small workloads: the tiny
    Erdos-Renyi graph (4,096 nodes, degree 16; SpMM, SDDMM, attention at
    F = 32) and the fused attention-aggregation benchmark shape (384 nodes,
    degree 18, edge-softmax aggregation with given scores at F = 64).
    Median of 3 runs, ms."""
    import oracle

    def med(fn):
        ts = []
        for _ in range(3):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        return round(1e3 * float(np.median(ts)), 3)

    oracle.set_threads(1)
    try:
        g = synth.tiny_er(0)
        X, Q, K, V = (synth.normal(g.n_rows, 32, 0, st) for st in
                      (synth.STREAM_X, synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
        p = synth.attention_benchmark_shape(0)
        S = synth.normal(p.nnz, 1, 0, synth.STREAM_Q)
        PV = synth.normal(p.n_rows, 64, 0, synth.STREAM_V)
        out = {
            "tiny_er/spmm/F32": med(lambda: oracle.spmm(g.row_ptr, g.col_idx, g.vals, X)),
            "tiny_er/sddmm/F32": med(lambda: oracle.sddmm(g.row_ptr, g.col_idx, Q, K, 1.0)),
            "tiny_er/attention/H1D32": med(lambda: oracle.csr_attention(g.row_ptr, g.col_idx, Q, K, V, 1,
                                                                        1.0 / np.sqrt(32))),
            "page_shape/edge_softmax_aggregate/F64": med(lambda: oracle.edge_softmax_aggregate(
                p.row_ptr, p.col_idx, S, PV)),
        }
    finally:
        oracle.set_threads(oracle.threads())
    return out


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    graphs = build_graphs(args.scale)
    budget = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(graphs, budget_s=budget)
    vals = []
    for _ in range(args.steps):
        vals.append(cpu_baseline(graphs, budget_s=budget))
    v = float(np.mean([x["value"] for x in vals]))
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": workload_config(graphs, world),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "kind": "oracle", "cores": vals[-1]["cores"],
                             "sample": vals[-1]["sample"]},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the rows measured beyond the step")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the products-like and Reddit-like throughput rows")
    ap.add_argument("--no-gather-peaks", action="store_true",
                    help="skip measuring the L2 and DRAM gather rates (the cache-aware bound)")
    ap.add_argument("--only", default=None, help="run only operations whose key contains one of these comma-separated texts "
                         "(backward, typed: the rows measured beyond the step)")
    ap.add_argument("--scale", type=int, default=20, help="R-MAT scale (20 is the benchmark workload)")
    ap.add_argument("--cache", default=None, help="plan cache file: loaded if present, saved after planning")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
