"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/autosage.h declares (no compute calls here)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "autosage.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(autosage_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    import shutil
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from sparse_gnn_aggregation_gb300 import build
    return build.build()


def test_header_declares_the_core_api():
    syms = declared_symbols()
    for name in ("autosage_spmm", "autosage_sddmm", "autosage_csr_attention", "autosage_plan",
                 "autosage_plan_destroy", "autosage_cache_load", "autosage_cache_save",
                 "autosage_status_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True)
    exported = {line.split()[-1] for line in out.stdout.splitlines() if line.strip()}
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, f"not exported: {missing}"


def test_binding_loads_and_names_match(lib_path):
    import sparse_gnn_aggregation_gb300 as sga
    assert sorted(sga.EXPORTS) == declared_symbols()
    for name in sga.EXPORTS:
        assert hasattr(sga.library(), name)
        if name not in ("autosage_status_string", "autosage_last_error", "autosage_version", "autosage_plan_destroy",
                        "autosage_cache_clear", "autosage_cache_size", "autosage_plan_describe",
                        "autosage_plan_schedule"):
            assert hasattr(sga, name), f"binding lacks {name}"
    assert sga.autosage_version().startswith("autosage-gb300")
    assert sga.library().autosage_status_string(sga.ERR_PROBE).decode().startswith("every probed")


def test_host_side_argument_checks_need_no_gpu(lib_path):
    """Calls rejected on the host return a status before touching the device."""
    import ctypes
    import sparse_gnn_aggregation_gb300 as sga
    lib = sga.library()
    assert lib.autosage_spmm(None, None, 0, None, 0, 4, 0, 0, None, None) == sga.ERR_INVALID_ARG
    assert b"A is NULL" in lib.autosage_last_error()
    c = sga._Csr(-1, 4, 0, 16, 0, 0)
    assert lib.autosage_sddmm(ctypes.byref(c), None, 0, None, 0, 4, 0, 1.0, None, None, None) == sga.ERR_INVALID_ARG
    c = sga._Csr(4, 4, 0, 16, 0, 0)  # row_ptr "pointer" 16, F = 0
    assert lib.autosage_spmm(ctypes.byref(c), None, 0, None, 0, 0, 0, 0, None, None) == sga.ERR_INVALID_ARG
    assert lib.autosage_cache_load(b"/nonexistent/dir/cache.txt") == sga.ERR_CACHE_IO
    sched = sga._Schedule(sga.SCHED_ROWGROUP, 3, 1, 0)  # lanes not a power of two
    h = ctypes.c_void_p()
    assert lib.autosage_plan_with_schedule(ctypes.byref(c), 0, 4, 1, 0, ctypes.byref(sched), ctypes.byref(h),
                                           None) == sga.ERR_INVALID_ARG


def test_no_alloc_entry_checks_its_csr_on_the_host(lib_path):
    """The allocation-free attention refuses a misaligned or over-large CSR with
    the same host-side checks as autosage_csr_attention, before it touches a
    device (this runs without a GPU: a refused call makes no CUDA call)."""
    import ctypes
    import sparse_gnn_aggregation_gb300 as sga
    lib = sga.library()
    P = ctypes.c_void_p
    feat = P(0x10000)  # stand-in device addresses: never dereferenced on a refused call
    misaligned = sga._Csr(4, 4, 4, 0x20000, 0x30002, 0)  # col_idx not 4-byte aligned
    st = lib.autosage_csr_attention_unfused_noalloc(ctypes.byref(misaligned), feat, feat, feat, 1, 4, sga.F32,
                                                    1.0, feat, None)
    assert st == sga.ERR_INVALID_ARG
    assert b"aligned" in lib.autosage_last_error()
    huge = sga._Csr(2 ** 31, 4, 4, 0x20000, 0x30000, 0)  # n_rows does not fit int32
    st = lib.autosage_csr_attention_unfused_noalloc(ctypes.byref(huge), feat, feat, feat, 1, 4, sga.F32,
                                                    1.0, feat, None)
    assert st == sga.ERR_UNSUPPORTED
    ok = sga._Csr(4, 4, 4, 0x20000, 0x30000, 0)
    st = lib.autosage_csr_attention_unfused_noalloc(ctypes.byref(ok), feat, feat, feat, 0, 4, sga.F32,
                                                    1.0, feat, None)
    assert st == sga.ERR_INVALID_ARG  # heads < 1
    assert lib.autosage_plan_rebind(None, ctypes.byref(ok), None) == sga.ERR_INVALID_ARG


def test_gather_rate_arguments_are_checked_on_the_host(lib_path):
    # bad sizes are refused before any device call (no GPU here)
    import ctypes
    import sparse_gnn_aggregation_gb300 as sga
    lib = sga.library()
    g = ctypes.c_double(-1.0)
    for table, row, n, reps in ((1 << 20, 8, 100, 1), (1 << 20, 4112, 10, 1), (1 << 20, 1000, 10, 1),
                                (100, 1024, 10, 1), (1 << 20, 1024, 0, 1), (1 << 20, 1024, 10, 0)):
        assert lib.autosage_measure_gather(table, row, n, reps, ctypes.byref(g), None) == sga.ERR_INVALID_ARG
        assert g.value == 0.0
    assert lib.autosage_measure_gather(1 << 20, 1024, 10, 1, None, None) == sga.ERR_INVALID_ARG


def test_aggregation_lanes_are_checked_on_the_host(lib_path):
    # lanes_f_agg belongs to unfused attention and must be a power of two that
    # fits a warp with the edge lanes; bad values are refused before the CSR
    # is touched (the addresses below are never dereferenced)
    import ctypes
    import sparse_gnn_aggregation_gb300 as sga
    lib = sga.library()
    A = sga._Csr(4, 4, 4, 0x20000, 0x30000, 0)
    out = ctypes.c_void_p()
    for op, agg, lanes_e in ((sga.OP_SPMM, 16, 1), (sga.OP_ATTN, 16, 1), (sga.OP_ATTN_UNFUSED, 24, 1),
                             (sga.OP_ATTN_UNFUSED, 32, 2), (sga.OP_ATTN_UNFUSED, 64, 1)):
        s = sga._Schedule(sga.SCHED_BINNED, 16, lanes_e, 512, 0, agg)
        st = lib.autosage_plan_with_schedule(ctypes.byref(A), op, 64, 8, sga.BF16, ctypes.byref(s),
                                             ctypes.byref(out), None)
        assert st == sga.ERR_INVALID_ARG, (op, agg, lanes_e)
        assert b"lanes_f_agg" in lib.autosage_last_error()
        assert out.value is None


def test_header_is_plain_c_and_a_c_program_links(lib_path, tmp_path):
    # the boundary is usable from C: the header compiles as C11 (no C++ or
    # torch types), and a C program links against the library and calls the
    # entry points that need no GPU
    import shutil
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "use.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "autosage.h"
int main(void) {
  autosage_schedule s;
  memset(&s, 0, sizeof s);
  s.kind = AUTOSAGE_SCHED_BINNED;
  s.per_edge = 1;
  const char *v = autosage_version();
  const char *e = autosage_status_string(AUTOSAGE_ERR_INVALID_CSR);
  /* a NULL CSR is an argument error, reported before any launch */
  autosage_status st = autosage_spmm(NULL, NULL, 0, NULL, 0, 4, AUTOSAGE_F32, 0, NULL, NULL);
  printf("%s|%s|%d|%d\n", v, e, (int)st, (int)(st == AUTOSAGE_ERR_INVALID_ARG));
  return st == AUTOSAGE_ERR_INVALID_ARG ? 0 : 1;
}
""")
    exe = tmp_path / "use"
    libdir = os.path.dirname(lib_path)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lautosage", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    version, err, _, ok = out.stdout.strip().split("|")
    assert version.startswith("autosage") and "CSR" in err and ok == "1"
