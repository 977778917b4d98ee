// Host runtime and C ABI: argument checks, feature geometry, plans and their
// workspace, the input-aware schedule picker (cost estimate from row
// statistics, checked by short timed runs on the device), and the persistent plan
// cache (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN Aggregation
// (SpMM/SDDMM) and CSR Attention", Abstract: the scheduler picks tiling and
// mapping for each input from a cheap cost estimate that short runs on the
// device refine, and keeps its choices in a persistent cache so that later
// runs replay them). The
// fallback ("guardrail") is this library's own default row-group schedule,
// never a vendor library or the CPU.
#include <algorithm>
#include <cinttypes>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <map>
#include <mutex>
#include <sstream>
#include <string>
#include <vector>

#include "../../include/autosage.h"
#include "internal.h"

using namespace autosage;

namespace {

thread_local std::string g_last_error;

autosage_status fail(autosage_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

autosage_status cuda_fail(cudaError_t e, const char *where) {
  return fail(AUTOSAGE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define CUDA_TRY(expr)                                     \
  do {                                                     \
    cudaError_t _e = (expr);                               \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr);    \
  } while (0)

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

int pow2ceil(int64_t x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// ---------------------------------------------------------------- validation

// Host-side checks of a CSR descriptor (sizes, NULL pointers, alignment);
// with AUTOSAGE_CHECK=1 and gpu_check, also the full structural validation
// on the GPU (synchronising; it allocates a stream-ordered flag).
autosage_status check_csr(const autosage_csr *A, bool gpu_check) {
  if (!A) return fail(AUTOSAGE_ERR_INVALID_ARG, "A is NULL");
  if (A->n_rows < 0 || A->n_cols < 0 || A->nnz < 0)
    return fail(AUTOSAGE_ERR_INVALID_ARG, "negative CSR size");
  if (A->n_rows >= INT32_MAX || A->n_cols >= INT32_MAX || A->nnz >= INT32_MAX)
    return fail(AUTOSAGE_ERR_UNSUPPORTED, "CSR sizes must fit int32");
  if (!A->row_ptr) return fail(AUTOSAGE_ERR_INVALID_ARG, "row_ptr is NULL");
  if (A->nnz > 0 && !A->col_idx) return fail(AUTOSAGE_ERR_INVALID_ARG, "col_idx is NULL");
  if (A->nnz > 0 && A->n_cols == 0) return fail(AUTOSAGE_ERR_INVALID_CSR, "edges but no columns");
  if ((reinterpret_cast<uintptr_t>(A->row_ptr) | reinterpret_cast<uintptr_t>(A->col_idx) |
       reinterpret_cast<uintptr_t>(A->vals)) & 3u)
    return fail(AUTOSAGE_ERR_INVALID_ARG, "CSR arrays must be 4-byte aligned");
  if (gpu_check && getenv("AUTOSAGE_CHECK") && atoi(getenv("AUTOSAGE_CHECK")) > 0) {
    // full structural check on the GPU (synchronising)
    autosage_status st = autosage_validate_csr(A, nullptr);
    if (st != AUTOSAGE_OK) return st;
  }
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- geometry

struct Mat {
  const void *p;
  int64_t ld;
};

// Pick the widest fragment (16, 8, 4 or 2 bytes) that every matrix's
// pointer, leading dimension and the head width allow; then lanes and slots.
autosage_status choose_geom(DType dt, int H, int64_t D, std::initializer_list<Mat> mats, int G_req,
                            int E_req, bool need_head_reduce, int nv_max, Geom &g) {
  const int s = dtype_size(dt);
  const int64_t F = (int64_t)H * D;
  int vb = 0;
  for (int cand : {16, 8, 4, 2}) {
    if (cand < s) continue;
    if ((D * s) % cand) continue;
    bool ok = true;
    for (const Mat &m : mats) {
      if ((reinterpret_cast<uintptr_t>(m.p) % cand) || ((m.ld * s) % cand)) ok = false;
    }
    if (ok) {
      vb = cand;
      break;
    }
  }
  if (vb == 0) return fail(AUTOSAGE_ERR_INVALID_ARG, "feature pointers must be aligned to the element size");
  g.dt = dt;
  g.H = H;
  g.D = D;
  g.es = H;
  g.VW = vb / s;
  g.nfrag = static_cast<int>(F / g.VW);
  g.cph = static_cast<int>(D / g.VW);
  g.G = G_req > 0 ? G_req : std::min(32, pow2ceil(g.nfrag));
  // an explicit edge-lane count with automatic feature lanes keeps the group within a warp
  if (G_req <= 0 && E_req > 0 && is_pow2(E_req) && E_req <= 32) g.G = std::min(g.G, 32 / E_req);
  if (!is_pow2(g.G) || g.G > 32) return fail(AUTOSAGE_ERR_INVALID_ARG, "lanes_f must be a power of two <= 32");
  const int64_t per_lane = (g.nfrag + g.G - 1) / g.G;
  g.NV = pow2ceil(per_lane);
  if (g.NV > nv_max)
    return fail(AUTOSAGE_ERR_UNSUPPORTED, "feature width %" PRId64 " too large for one pass", F);
  g.E = E_req > 0 ? E_req : std::max(1, std::min(32 / g.G, 8));
  if (!is_pow2(g.E) || g.G * g.E > 32) return fail(AUTOSAGE_ERR_INVALID_ARG, "lanes_f * lanes_e must be <= 32");
  // fragment-to-lane mapping and head reductions
  g.fs = 1;
  g.ks = g.G;
  g.one = true;
  g.R = g.G;
  g.batched = false;
  if (H == 1) {
    g.batched = g.G >= 4;  // batches of 4 (G = 4) or 8 edges
  } else if (!need_head_reduce) {
    // per-head weights only (SpMM): with four or more slots per lane,
    // consecutive fragments keep a lane in one head, so each edge needs one
    // weight per lane instead of one per slot (measured: faster at 4 slots,
    // slower at 2, where interleaved lanes coalesce better)
    if (g.NV >= 4 && g.NV <= g.cph && g.cph % g.NV == 0) {
      g.fs = g.NV;
      g.ks = 1;
    } else {
      g.one = false;
    }
  } else {
    if (!is_pow2(g.cph))
      return fail(AUTOSAGE_ERR_UNSUPPORTED, "multi-head reduction needs D/VW a power of two");
    if (g.NV <= g.cph) {  // consecutive fragments per lane, all in one head
      g.fs = g.NV;
      g.ks = 1;
      g.R = g.cph / g.NV;
    } else if (g.cph <= g.G) {  // interleaved lanes, one head per slot
      g.one = false;
      g.R = g.cph;
    } else {
      return fail(AUTOSAGE_ERR_UNSUPPORTED, "head width does not fit the lane mapping");
    }
  }
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- device info

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  std::string name;
  double bw = 6.8e12;  // bytes/s used by the estimate
};

DeviceInfo device_info() {
  DeviceInfo d;
  cudaGetDevice(&d.device);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, d.device) == cudaSuccess) {
    d.sms = prop.multiProcessorCount;
    d.name = prop.name;
    for (char &c : d.name)
      if (c == ' ' || c == '|' || c == '\t') c = '_';
  }
  return d;
}

// ---------------------------------------------------------------- device buffers

struct DevBuf {
  void *p = nullptr;
  size_t bytes = 0;
  cudaError_t alloc(size_t n) {
    release();
    if (n == 0) return cudaSuccess;
    cudaError_t e = cudaMalloc(&p, n);
    if (e == cudaSuccess) bytes = n;
    else p = nullptr;
    return e;
  }
  void release() {
    if (p) cudaFree(p);
    p = nullptr;
    bytes = 0;
  }
  template <typename T> T *as() const { return static_cast<T *>(p); }
};

// ---------------------------------------------------------------- statistics

struct RowStats {
  int64_t ints[40];
  double mean = 0, cv = 0;
};

autosage_status gpu_row_stats(int64_t n_rows, const int32_t *row_ptr, int64_t thr, RowStats &out,
                              cudaStream_t s) {
  unsigned long long *d = nullptr;
  CUDA_TRY(cudaMallocAsync(&d, 40 * sizeof(unsigned long long), s));
  cudaError_t e = launch_row_stats(n_rows, row_ptr, thr, d, s);
  unsigned long long h[40] = {0};
  if (e == cudaSuccess) e = cudaMemcpyAsync(h, d, sizeof h, cudaMemcpyDeviceToHost, s);
  cudaFreeAsync(d, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "row statistics");
  for (int i = 0; i < 40; ++i) out.ints[i] = static_cast<int64_t>(h[i]);
  out.ints[0] = n_rows;
  if (n_rows == 0) out.ints[3] = 0;
  out.mean = n_rows > 0 ? (double)out.ints[1] / (double)n_rows : 0.0;
  const double var = n_rows > 0 ? (double)out.ints[5] / (double)n_rows - out.mean * out.mean : 0.0;
  out.cv = out.mean > 0.0 ? std::sqrt(var > 0.0 ? var : 0.0) / out.mean : 0.0;
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- plan

// Hybrid schedule: rows of 1..kEllMaxDegree edges (the degree buckets from
// key kEllFirstKey of the binned order on) are kept in an ELL slab of
// kEllSlots columns; every other row runs as in the binned schedule.
constexpr int kEllSlots = 8;
constexpr int kEllMaxDegree = 7;
constexpr int kEllFirstKey = 28;  // bit length 3: degrees 4..7

struct Sched {
  int kind = AUTOSAGE_SCHED_ROWGROUP;
  int G = 0, E = 0, split = 0;
  int pe = 0;  // SDDMM, one head: per-edge shuffle reductions instead of batched ones
  int G2 = 0;  // unfused attention: feature lanes of the aggregation stage (0: G)
};

}  // namespace

struct autosage_plan_s {
  autosage_op op;
  DType dt;
  int64_t F;  // feature width (attention: head dim D)
  int H;
  int64_t n_rows, n_cols, nnz;
  Sched sched;
  double probe_ms = -1;
  double est_ms = -1;
  bool from_cache = false;
  int64_t maxdeg = -1;  // longest row of the walked CSR (-1: not computed)
  bool comp = true;     // SpMM: compensated accumulation (serial sums longer than 512 edges)
  // The A the plan is bound to: calls must pass these structure arrays (the
  // edge values come from each call); a0 also serves the planning probes.
  // a_fp is the fingerprint of A's structure (autosage_plan_rebind checks it).
  autosage_csr a0{};
  uint64_t a_fp = 0;
  // AUTOSAGE_PLAN_FIXED_VALUES: the edge values are part of the plan (SPMM_T
  // keeps them in A^T order in t_vals); calls must pass this value array
  bool fixed_vals = false;
  const float *fixed_vals_ptr = nullptr;
  // the CSR the plan's workspace was built over (A, or A^T for SPMM_T)
  int64_t k_rows = 0;
  const int32_t *k_row_ptr = nullptr;
  const int32_t *k_col_idx = nullptr;
  // A^T when op == SPMM_T; t_vals receives the call's edge values in A^T order
  DevBuf t_row_ptr, t_col_idx, t_vals;
  // split workspace
  DevBuf long_rows, long_ptr, chunk_row, chunk_begin, partial, ml, row_ml, row_order;
  // hybrid schedule: the ELL slab of the short rows (positions [ell_pos0,
  // ell_pos0 + n_ell) of row_order)
  DevBuf ell_col, ell_start;
  int64_t n_ell = 0, ell_pos0 = 0;
  ChunkList cl;
  // merge-path workspace
  DevBuf mp_part, mp_carry_val, mp_carry_row, mp_head_val;
  int64_t mp_warps = 0;
  // unfused attention scores (backward: the softmax weights)
  DevBuf scores;
  // A^T position -> A edge (SPMM_T); backward: A edge -> A^T position, edge
  // buffers (dW scratch, w and dS in A^T order) and the A^T SpMM plan
  DevBuf t_perm, t_inv, grad_dw, grad_wt, grad_dst;
  autosage_plan_s *tplan = nullptr;
  // typed SpMM: number of relations (0: untyped), the combined gather index,
  // and the caller's column and edge-type arrays it was built from
  int typed = 0;
  int64_t base_cols = 0;
  DevBuf typed_idx;
  const int32_t *typed_col = nullptr;
  const int32_t *typed_type = nullptr;
  ~autosage_plan_s() {
    for (DevBuf *b : {&t_row_ptr, &t_col_idx, &t_vals, &long_rows, &long_ptr, &chunk_row,
                      &chunk_begin, &partial, &ml, &row_ml, &row_order, &mp_part, &mp_carry_val,
                      &mp_carry_row, &mp_head_val, &scores, &t_perm, &t_inv, &grad_dw, &grad_wt, &grad_dst,
                      &typed_idx, &ell_col, &ell_start})
      b->release();
    delete tplan;
  }
};

namespace {

// ---------------------------------------------------------------- cache

constexpr const char *kCacheHeader = "# autosage plan cache v1";

struct CacheEntry {
  Sched sched;
  double probe_ms = -1;
};

std::mutex g_cache_mu;
std::map<std::string, CacheEntry> g_cache;

std::string cache_key(const DeviceInfo &dev, autosage_op op, DType dt, int64_t F, int H,
                      int64_t n_rows, int64_t n_cols, int64_t nnz, uint64_t fp) {
  char buf[512];
  snprintf(buf, sizeof buf, "%s|sm%d|op%d|dt%d|F%" PRId64 "|H%d|n%" PRId64 "|m%" PRId64 "|nnz%" PRId64 "|fp%016" PRIx64,
           dev.name.c_str(), dev.sms, (int)op, (int)dt, F, H, n_rows, n_cols, nnz, fp);
  return buf;
}

const char *sched_name(int kind) {
  switch (kind) {
    case AUTOSAGE_SCHED_ROWGROUP: return "rowgroup";
    case AUTOSAGE_SCHED_SPLIT: return "split";
    case AUTOSAGE_SCHED_MERGEPATH: return "mergepath";
    case AUTOSAGE_SCHED_BINNED: return "binned";
    case AUTOSAGE_SCHED_HYBRID: return "hybrid";
  }
  return "?";
}

// ---------------------------------------------------------------- op geometry

struct OpShape {
  int H;
  int64_t D;       // width per head (F for H == 1)
  bool head_reduce;
  int nv_max;
};

OpShape op_shape(autosage_op op, int64_t F, int H) {
  switch (op) {
    case AUTOSAGE_OP_SPMM:
    case AUTOSAGE_OP_SPMM_T: return {1, F, false, 16};
    case AUTOSAGE_OP_SDDMM: return {1, F, true, 16};
    case AUTOSAGE_OP_ATTN: return {H, F, true, 8};
    case AUTOSAGE_OP_ATTN_UNFUSED: return {H, F, true, 16};
    case AUTOSAGE_OP_SOFTMAX: return {H, 1, false, 16};
    case AUTOSAGE_OP_ATTN_BACKWARD: return {H, F, true, 8};
  }
  return {1, F, false, 16};
}

// Default schedule (the guardrail): row groups with lanes from the width.
Sched default_sched() { return Sched{AUTOSAGE_SCHED_ROWGROUP, 0, 0, 0}; }

// ---------------------------------------------------------------- workspace

autosage_status build_split(autosage_plan_s *P, int split, cudaStream_t s) {
  P->cl = ChunkList{};
  if (split <= 0 || P->k_rows == 0) return AUTOSAGE_OK;
  DevBuf flags, scan_out, scan_tmp;
  CUDA_TRY(flags.alloc(sizeof(int32_t) * (size_t)(P->k_rows + 1)));
  CUDA_TRY(scan_out.alloc(sizeof(int32_t) * (size_t)(P->k_rows + 1)));
  CUDA_TRY(scan_tmp.alloc(scan_tmp_bytes(P->k_rows)));
  CUDA_TRY(P->long_rows.alloc(sizeof(int32_t) * (size_t)(P->k_rows + 1)));
  CUDA_TRY(P->long_ptr.alloc(sizeof(int32_t) * (size_t)(P->k_rows + 1)));
  const int64_t max_chunks = P->nnz / split + P->k_rows + 1;
  // chunk arrays sized after counting: first pass counts, second fills
  int64_t n_long = 0, n_chunks = 0;
  {
    // temporary chunk arrays large enough for any graph would be wasteful; count first
    RowStats st;
    autosage_status rs = gpu_row_stats(P->k_rows, P->k_row_ptr, split, st, s);
    if (rs != AUTOSAGE_OK) return rs;
    n_chunks = (st.ints[7] + (int64_t)split - 1) / split + st.ints[6];  // upper bound
    n_chunks = std::min(n_chunks, max_chunks);
  }
  CUDA_TRY(P->chunk_row.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(n_chunks, 1)));
  CUDA_TRY(P->chunk_begin.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(n_chunks, 1)));
  int64_t got_chunks = 0;
  CUDA_TRY(build_chunk_lists(P->k_rows, P->k_row_ptr, split, flags.as<int32_t>(), scan_out.as<int32_t>(),
                             scan_tmp.p, P->long_rows.as<int32_t>(), P->long_ptr.as<int32_t>(),
                             P->chunk_row.as<int32_t>(), P->chunk_begin.as<int32_t>(), &n_long,
                             &got_chunks, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  if (got_chunks > n_chunks) return fail(AUTOSAGE_ERR_CUDA, "chunk count exceeded its bound");
  P->cl.chunk_row = P->chunk_row.as<int32_t>();
  P->cl.chunk_begin = P->chunk_begin.as<int32_t>();
  P->cl.long_rows = P->long_rows.as<int32_t>();
  P->cl.long_ptr = P->long_ptr.as<int32_t>();
  P->cl.n_long = static_cast<int>(n_long);
  P->cl.n_chunks = static_cast<int>(got_chunks);
  P->cl.split = split;
  // partial buffers for every consumer of the chunk list
  const int64_t C = got_chunks;
  const bool heads_op = P->op == AUTOSAGE_OP_ATTN || P->op == AUTOSAGE_OP_ATTN_UNFUSED ||
                        P->op == AUTOSAGE_OP_ATTN_BACKWARD;
  const int64_t width = P->F * (heads_op ? P->H : 1);
  if (P->op == AUTOSAGE_OP_ATTN_BACKWARD) {
    // per chunk: the (A, B) feature sums, (m, l, sum e dW) per head and the cut row's index
    CUDA_TRY(P->partial.alloc(sizeof(float) * (size_t)std::max<int64_t>(C * (2 * width + 3 * P->H + 1), 1)));
    CUDA_TRY(P->row_ml.alloc(sizeof(float) * (size_t)std::max<int64_t>(n_long * P->H * 3, 1)));
    return AUTOSAGE_OK;
  }
  if (P->op != AUTOSAGE_OP_SDDMM && P->op != AUTOSAGE_OP_SOFTMAX)
    CUDA_TRY(P->partial.alloc(sizeof(float) * (size_t)std::max<int64_t>(C * width, 1)));
  const int Hs = (P->op == AUTOSAGE_OP_SOFTMAX || heads_op) ? P->H : 1;
  CUDA_TRY(P->ml.alloc(sizeof(float) * (size_t)std::max<int64_t>(C * Hs * 2 + C, 1)));
  CUDA_TRY(P->row_ml.alloc(sizeof(float) * (size_t)std::max<int64_t>(n_long * Hs * 2, 1)));
  return AUTOSAGE_OK;
}

autosage_status build_mergepath(autosage_plan_s *P, int items, int64_t width, cudaStream_t s) {
  const int64_t total = P->k_rows + P->nnz;
  P->mp_warps = (total + items - 1) / items;
  CUDA_TRY(P->mp_part.alloc(sizeof(int2) * (size_t)(P->mp_warps + 1)));
  CUDA_TRY(P->mp_carry_val.alloc(sizeof(float) * (size_t)std::max<int64_t>(P->mp_warps * width, 1)));
  CUDA_TRY(P->mp_carry_row.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(P->mp_warps, 1)));
  CUDA_TRY(P->mp_head_val.alloc(sizeof(float) * (size_t)std::max<int64_t>(P->mp_warps * width, 1)));
  CUDA_TRY(launch_mergepath_partition(P->k_rows, P->nnz, P->k_row_ptr, items, P->mp_warps,
                                      P->mp_part.as<int2>(), s));
  return AUTOSAGE_OK;
}

// Build the workspace of a schedule for plan P (P->sched set).
autosage_status build_workspace(autosage_plan_s *P, cudaStream_t s) {
  for (DevBuf *b : {&P->long_rows, &P->long_ptr, &P->chunk_row, &P->chunk_begin, &P->partial,
                    &P->ml, &P->row_ml, &P->row_order, &P->mp_part, &P->mp_carry_val, &P->mp_carry_row,
                    &P->mp_head_val, &P->ell_col, &P->ell_start})
    b->release();
  P->cl = ChunkList{};
  P->n_ell = 0;
  P->mp_warps = 0;
  autosage_status st = AUTOSAGE_OK;
  if (P->op == AUTOSAGE_OP_SPMM || P->op == AUTOSAGE_OP_SPMM_T || P->op == AUTOSAGE_OP_ATTN_BACKWARD) {
    if (P->maxdeg < 0) {
      RowStats rs;
      st = gpu_row_stats(P->k_rows, P->k_row_ptr, 1024, rs, s);
      if (st != AUTOSAGE_OK) return st;
      P->maxdeg = rs.ints[2];
    }
    // longest run of edges one lane sums serially (edge lanes taken as 1 when automatic)
    const int64_t lanes_e = P->sched.E > 0 ? P->sched.E : 1;
    int64_t run = P->maxdeg;
    if (P->sched.kind == AUTOSAGE_SCHED_SPLIT || P->sched.kind == AUTOSAGE_SCHED_BINNED ||
        P->sched.kind == AUTOSAGE_SCHED_HYBRID)
      run = std::min<int64_t>(run, P->sched.split);
    if (P->sched.kind == AUTOSAGE_SCHED_MERGEPATH) run = std::min<int64_t>(run, P->sched.split);
    P->comp = run / lanes_e > 512;
  }
  const bool hybrid = P->sched.kind == AUTOSAGE_SCHED_HYBRID;
  if (hybrid && P->op != AUTOSAGE_OP_SPMM && P->op != AUTOSAGE_OP_SPMM_T)
    return fail(AUTOSAGE_ERR_UNSUPPORTED, "hybrid (ELL + CSR) schedule is SpMM only");
  if (hybrid && P->sched.split < kEllMaxDegree)
    return fail(AUTOSAGE_ERR_INVALID_ARG, "hybrid schedule needs a chunk length of at least %d", kEllMaxDegree);
  if (P->sched.kind == AUTOSAGE_SCHED_SPLIT || P->sched.kind == AUTOSAGE_SCHED_BINNED || hybrid) {
    st = build_split(P, P->sched.split, s);
    if (st == AUTOSAGE_OK && P->sched.kind != AUTOSAGE_SCHED_SPLIT && P->k_rows > 0) {
      CUDA_TRY(P->row_order.alloc(sizeof(int32_t) * (size_t)P->k_rows));
      CUDA_TRY(build_row_order(P->k_rows, P->k_row_ptr, P->sched.split, P->row_order.as<int32_t>(),
                               P->cl.bucket_start, s));
      P->cl.row_order = P->row_order.as<int32_t>();
    }
    if (st == AUTOSAGE_OK && hybrid && P->k_rows > 0) {
      // the degree buckets of 1..7 edges (keys 28, 29, 30 of the binned order) go to an ELL slab
      P->cl.ell_from = kEllFirstKey;
      P->cl.ell_to = 31;
      P->ell_pos0 = P->cl.bucket_start[kEllFirstKey];
      P->n_ell = (int64_t)P->cl.bucket_start[31] - P->ell_pos0;
      CUDA_TRY(P->ell_col.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(P->n_ell * kEllSlots, 1)));
      CUDA_TRY(P->ell_start.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(P->n_ell, 1)));
      CUDA_TRY(build_ell(P->n_ell, kEllSlots, P->row_order.as<int32_t>(), P->ell_pos0, P->k_row_ptr, P->k_col_idx,
                         P->ell_col.as<int32_t>(), P->ell_start.as<int32_t>(), s));
    }
  } else if (P->sched.kind == AUTOSAGE_SCHED_MERGEPATH) {
    if (P->op != AUTOSAGE_OP_SPMM && P->op != AUTOSAGE_OP_SPMM_T && P->op != AUTOSAGE_OP_SDDMM)
      return fail(AUTOSAGE_ERR_UNSUPPORTED, "merge-path schedule is SpMM and SDDMM only");
    // SDDMM writes one value per edge: its merge path needs partitions but no carries
    st = build_mergepath(P, P->sched.split, P->op == AUTOSAGE_OP_SDDMM ? 0 : P->F, s);
  }
  if (st != AUTOSAGE_OK) return st;
  if ((P->op == AUTOSAGE_OP_ATTN_UNFUSED || P->op == AUTOSAGE_OP_ATTN_BACKWARD) && !P->scores.p)
    CUDA_TRY(P->scores.alloc(sizeof(float) * (size_t)std::max<int64_t>(P->nnz * P->H, 1)));
  if (P->op == AUTOSAGE_OP_ATTN_BACKWARD && !P->grad_dw.p) {
    const size_t eb = sizeof(float) * (size_t)std::max<int64_t>(P->nnz * P->H, 1);
    CUDA_TRY(P->grad_dw.alloc(eb));
    CUDA_TRY(P->grad_wt.alloc(eb));
    CUDA_TRY(P->grad_dst.alloc(eb));
  }
  CUDA_TRY(cudaStreamSynchronize(s));
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- running ops

struct OpArgs {
  const void *X = nullptr;  // SpMM input / attention V
  int64_t ldx = 0;
  void *Y = nullptr;        // SpMM output / attention out
  int64_t ldy = 0;
  const void *Q = nullptr, *K = nullptr;
  int64_t ldq = 0, ldk = 0;
  float alpha = 1.f;
  float *S = nullptr;       // SDDMM output / softmax in-out
  const float *given = nullptr;  // given scores (edge-softmax aggregation)
  const void *dO = nullptr;      // backward: upstream gradient and outputs
  void *dQ = nullptr, *dK = nullptr, *dV = nullptr;
};

// The CSR one call walks: the caller's row_ptr, col_idx and edge values;
// for SPMM_T the plan's A^T, with the caller's edge values gathered into
// A^T's edge order through the stored permutation (so new values take
// effect without a new plan).
struct Walk {
  int64_t rows;
  const int32_t *row_ptr;
  const int32_t *col_idx;
  const float *vals;
};

cudaError_t walk_for(const autosage_plan_s *P, autosage_op op, const autosage_csr *A, cudaStream_t s, Walk &w) {
  if (op != AUTOSAGE_OP_SPMM_T) {
    w = Walk{A->n_rows, A->row_ptr, A->col_idx, A->vals};
    return cudaSuccess;
  }
  w = Walk{P->k_rows, P->k_row_ptr, P->k_col_idx, nullptr};
  if (!A->vals || A->nnz == 0) return cudaSuccess;
  w.vals = P->t_vals.as<float>();
  if (P->fixed_vals) return cudaSuccess;  // gathered once, when the values were fixed
  return launch_gather_vals(A->nnz, P->t_perm.as<int32_t>(), A->vals, P->t_vals.as<float>(), s);
}

// Fix the plan's edge values to A->vals (FIXED_VALUES plans): SPMM_T gathers
// them into A^T's edge order once, here, instead of at every call.
autosage_status fix_values(autosage_plan_s *P, const autosage_csr *A, cudaStream_t s) {
  P->fixed_vals = true;
  P->fixed_vals_ptr = A->vals;
  if (P->op == AUTOSAGE_OP_SPMM_T && A->vals && A->nnz > 0) {
    CUDA_TRY(launch_gather_vals(A->nnz, P->t_perm.as<int32_t>(), A->vals, P->t_vals.as<float>(), s));
    CUDA_TRY(cudaStreamSynchronize(s));
  }
  return AUTOSAGE_OK;
}

// Run `op` over the call's A with plan P's schedule (plan-free runs use a
// transient P with the default schedule and no workspace).
autosage_status run_op(const autosage_plan_s *P, autosage_op op, const autosage_csr *A, const OpArgs &a,
                       cudaStream_t s) {
  const ChunkList &cl = P->cl;
  Geom g;
  autosage_status st;
  Walk wk;
  cudaError_t e = walk_for(P, op, A, s, wk);
  if (e != cudaSuccess) return cuda_fail(e, "edge values in A^T order");
  switch (op) {
    case AUTOSAGE_OP_SPMM:
    case AUTOSAGE_OP_SPMM_T: {
      const bool mp = P->sched.kind == AUTOSAGE_SCHED_MERGEPATH;
      const int E_req = mp ? 0 : P->sched.E;
      // lanes and fragment width for the full row; rows wider than one pass
      // (NV > 16 fragments per lane) are cut into column tiles of 8 * G * VW,
      // run one after another: eight fragments a lane keep two edges in
      // flight (measured on the Reddit-like graph at F = 602: the probes then
      // choose merge path G = 16, E = 2 at 48.7 ms, against 62.6 ms with
      // tiles of 16 fragments)
      st = choose_geom(P->dt, 1, P->F, {{a.X, a.ldx}, {a.Y, a.ldy}}, P->sched.G, E_req, false, 1 << 20, g);
      if (st != AUTOSAGE_OK) return st;
      const int64_t tile = (int64_t)(g.NV > 16 ? 8 : 16) * g.G * g.VW;
      const size_t es = dtype_size(P->dt);
      for (int64_t off = 0; off < P->F && e == cudaSuccess; off += tile) {
        const int64_t w = std::min<int64_t>(tile, P->F - off);
        const char *x = static_cast<const char *>(a.X) + off * es;
        char *y = static_cast<char *>(a.Y) + off * es;
        Geom gt;
        st = choose_geom(P->dt, 1, w, {{x, a.ldx}, {y, a.ldy}}, P->sched.G, E_req, false, 16, gt);
        if (st != AUTOSAGE_OK) return st;
        gt.comp = P->comp;
        if (mp) {
          gt.E = 32 / gt.G;
          e = launch_spmm_mergepath(gt, wk.rows, wk.row_ptr, wk.col_idx, wk.vals, x, a.ldx, y,
                                    a.ldy, P->mp_part.as<int2>(), P->mp_warps, P->sched.split, P->mp_carry_val.as<float>(),
                                    P->mp_carry_row.as<int32_t>(), P->mp_head_val.as<float>(), s);
        } else {
          e = launch_spmm(gt, wk.rows, wk.row_ptr, wk.col_idx, wk.vals, x, a.ldx, y, a.ldy, cl,
                          P->partial.as<float>(), s);
          if (e == cudaSuccess && P->n_ell > 0)
            e = launch_spmm_ell(gt, P->n_ell, P->row_order.as<int32_t>() + P->ell_pos0, P->ell_col.as<int32_t>(),
                                P->ell_start.as<int32_t>(), wk.vals, x, a.ldx, y, a.ldy, s);
        }
      }
      break;
    }
    case AUTOSAGE_OP_SDDMM: {
      st = choose_geom(P->dt, 1, P->F, {{a.Q, a.ldq}, {a.K, a.ldk}}, P->sched.G, P->sched.E, true, 16, g);
      if (st != AUTOSAGE_OK) return st;
      if (P->sched.pe) g.batched = false;
      const bool mp = P->sched.kind == AUTOSAGE_SCHED_MERGEPATH;
      e = launch_sddmm(g, wk.rows, wk.row_ptr, wk.col_idx, a.Q, a.ldq, a.K, a.ldk, a.alpha, a.S, cl,
                       mp ? P->mp_part.as<int2>() : nullptr, mp ? P->mp_warps : 0, s);
      break;
    }
    case AUTOSAGE_OP_SOFTMAX: {
      e = launch_row_softmax(wk.rows, wk.row_ptr, P->H, a.S, cl, P->ml.as<float>(),
                             P->row_ml.as<float>(), s);
      break;
    }
    case AUTOSAGE_OP_ATTN: {
      const int64_t ld = P->H * P->F;
      if (a.given) {
        st = choose_geom(P->dt, P->H, P->F, {{a.X, ld}, {a.Y, ld}}, P->sched.G, P->sched.E, true, 8, g);
      } else {
        st = choose_geom(P->dt, P->H, P->F, {{a.Q, ld}, {a.K, ld}, {a.X, ld}, {a.Y, ld}}, P->sched.G,
                         P->sched.E, true, 8, g);
      }
      if (st == AUTOSAGE_OK) {
        e = launch_attention(g, wk.rows, wk.row_ptr, wk.col_idx, a.Q, a.K, a.given, a.X, ld, a.alpha,
                             a.Y, cl, P->partial.as<float>(), P->ml.as<float>(), s);
        break;
      }
      if (st != AUTOSAGE_ERR_UNSUPPORTED || P->H == 1) return st;
      // heads whose fragments cannot share an aligned lane segment: one launch per head
      const size_t es = dtype_size(P->dt);
      for (int h = 0; h < P->H && e == cudaSuccess; ++h) {
        const int64_t off = (int64_t)h * P->F;
        auto at = [&](const void *p) { return p ? static_cast<const char *>(p) + off * es : nullptr; };
        st = choose_geom(P->dt, 1, P->F, {{at(a.Q), ld}, {at(a.K), ld}, {at(a.X), ld}, {at(a.Y), ld}},
                         P->sched.G, P->sched.E, true, 8, g);
        if (st != AUTOSAGE_OK) return st;
        g.es = P->H;
        e = launch_attention(g, wk.rows, wk.row_ptr, wk.col_idx, at(a.Q), at(a.K),
                             a.given ? a.given + h : nullptr, at(a.X), ld, a.alpha,
                             const_cast<char *>(at(a.Y)), cl, P->partial.as<float>(), P->ml.as<float>(), s);
      }
      break;
    }
    case AUTOSAGE_OP_ATTN_UNFUSED: {
      const int64_t ld = P->H * P->F;
      float *S = a.S;
      st = choose_geom(P->dt, P->H, P->F, {{a.Q, ld}, {a.K, ld}}, P->sched.G, P->sched.E, true, 16, g);
      if (st == AUTOSAGE_OK) {
        e = launch_sddmm(g, wk.rows, wk.row_ptr, wk.col_idx, a.Q, ld, a.K, ld, a.alpha, S, cl, nullptr, 0, s);
      } else if (st == AUTOSAGE_ERR_UNSUPPORTED && P->H > 1) {
        const size_t es = dtype_size(P->dt);
        for (int h = 0; h < P->H && e == cudaSuccess; ++h) {
          const char *q = static_cast<const char *>(a.Q) + (int64_t)h * P->F * es;
          const char *k = static_cast<const char *>(a.K) + (int64_t)h * P->F * es;
          st = choose_geom(P->dt, 1, P->F, {{q, ld}, {k, ld}}, P->sched.G, P->sched.E, true, 16, g);
          if (st != AUTOSAGE_OK) return st;
          g.es = P->H;
          e = launch_sddmm(g, wk.rows, wk.row_ptr, wk.col_idx, q, ld, k, ld, a.alpha, S + h, cl, nullptr, 0, s);
        }
      } else {
        return st;
      }
      if (e != cudaSuccess) break;
      e = launch_row_softmax(wk.rows, wk.row_ptr, P->H, S, cl, P->ml.as<float>(), P->row_ml.as<float>(), s);
      if (e != cudaSuccess) break;
      Geom g2;
      // the aggregation stage has its own feature lanes (measured on R-MAT scale 20,
      // bf16, H = 8, D = 64: scores at 16 lanes and aggregation at 32 ran 5.74 ms,
      // both at 16 6.37 ms)
      const int G_agg = P->sched.G2 > 0 ? P->sched.G2 : P->sched.G;
      st = choose_geom(P->dt, P->H, P->F, {{a.X, ld}, {a.Y, ld}}, G_agg, P->sched.E, false, 16, g2);
      if (st != AUTOSAGE_OK) return st;
      e = launch_spmm(g2, wk.rows, wk.row_ptr, wk.col_idx, S, a.X, ld, a.Y, ld, cl,
                      P->partial.as<float>(), s);
      break;
    }
    case AUTOSAGE_OP_ATTN_BACKWARD: {
      const autosage_plan_s *T = P->tplan;
      if (!T) return fail(AUTOSAGE_ERR_INVALID_ARG, "backward plan lacks its A^T part");
      const int64_t ld = P->H * P->F;
      // scores, softmax, dW, D and dQ in one pass over the rows of A; w and
      // scale * dS land in the edge order of A^T
      st = choose_geom(P->dt, P->H, P->F, {{a.Q, ld}, {a.K, ld}, {a.X, ld}, {a.dO, ld}, {a.dQ, ld}},
                       P->sched.G, P->sched.E, true, 8, g);
      if (st != AUTOSAGE_OK) return st;
      e = launch_attention_backward(g, wk.rows, wk.row_ptr, wk.col_idx, a.Q, a.K, a.X, a.dO, ld, P->H,
                                    a.alpha, a.dQ, P->scores.as<float>(), P->grad_dw.as<float>(),
                                    P->t_inv.as<int32_t>(), P->grad_wt.as<float>(), P->grad_dst.as<float>(), cl,
                                    P->partial.as<float>(), P->row_ml.as<float>(), s);
      // dV = SpMM(A^T; w, dO) and dK = SpMM(A^T; scale * dS, Q) in one pass over A^T
      if (e == cudaSuccess) {
        st = choose_geom(P->dt, P->H, P->F, {{a.dO, ld}, {a.dV, ld}, {a.Q, ld}, {a.dK, ld}}, T->sched.G,
                         T->sched.E, false, 16, g);
        if (st != AUTOSAGE_OK) return st;
        g.comp = T->comp;
        if (g.NV <= 4) {
          e = launch_spmm2(g, T->k_rows, T->k_row_ptr, T->k_col_idx, P->grad_wt.as<float>(),
                           P->grad_dst.as<float>(), a.dO, a.Q, ld, a.dV, a.dK, ld, T->cl, T->partial.as<float>(), s);
        } else {  // rows of more than 4 fragments a lane: two products spill, so two passes
          e = launch_spmm(g, T->k_rows, T->k_row_ptr, T->k_col_idx, P->grad_wt.as<float>(), a.dO, ld, a.dV, ld,
                          T->cl, T->partial.as<float>(), s);
          if (e == cudaSuccess)
            e = launch_spmm(g, T->k_rows, T->k_row_ptr, T->k_col_idx, P->grad_dst.as<float>(), a.Q, ld, a.dK, ld,
                            T->cl, T->partial.as<float>(), s);
        }
      }
      break;
    }
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- estimate

// Estimated time (seconds) of a schedule from row statistics: the larger of
// the HBM time for the algorithmic bytes (gathers rounded up to 32-byte
// sectors) and the issue/latency time of all group steps, plus the critical
// path of the longest work item and a per-launch overhead.
double estimate(const DeviceInfo &dev, const RowStats &st, autosage_op op, DType dt, int64_t F, int H,
                const Sched &sc, const Geom &g) {
  const double n = (double)st.ints[0], nnz = (double)st.ints[1];
  const int s = dtype_size(dt);
  const double row_bytes = (double)F * H * s;
  const double sector = 32.0 * std::ceil(row_bytes / 32.0);
  double per_edge = 4.0, per_row = 4.0;
  switch (op) {
    case AUTOSAGE_OP_SPMM:
    case AUTOSAGE_OP_SPMM_T: per_edge += 4.0 + sector; per_row += row_bytes; break;
    case AUTOSAGE_OP_SDDMM: per_edge += 4.0 * H + sector; per_row += row_bytes; break;
    case AUTOSAGE_OP_ATTN: per_edge += 2.0 * sector; per_row += 2.0 * row_bytes; break;
    case AUTOSAGE_OP_ATTN_UNFUSED: per_edge += 3.0 * sector + 5.0 * 4.0 * H; per_row += 2.0 * row_bytes; break;
    case AUTOSAGE_OP_SOFTMAX: per_edge = 3.0 * 4.0 * H; per_row = 4.0; break;
  }
  const double bw = dev.bw > 0 ? dev.bw : 6.8e12;
  const double t_bw = (nnz * per_edge + n * per_row) / bw;
  // group steps: each edge lane handles U edges per step
  const int U = g.NV * g.VW <= 8 ? 4 : (g.NV * g.VW <= 16 ? 2 : 1);
  const double lanes_per_item = (double)g.G * g.E;
  const double groups = (double)std::max(1, dev.sms) * 48.0 * (32.0 / lanes_per_item);
  const double lat = 1.2e-6;  // one dependent gather round trip
  double steps = 0, longest = 0;
  int64_t split = (sc.kind == AUTOSAGE_SCHED_SPLIT || sc.kind == AUTOSAGE_SCHED_BINNED ||
                   sc.kind == AUTOSAGE_SCHED_HYBRID) ? sc.split : 0;
  for (int b = 0; b < 32; ++b) {
    const double cnt = (double)st.ints[8 + b];
    if (cnt == 0) continue;
    const double d = b == 0 ? 0.0 : 1.5 * std::pow(2.0, b - 1);
    double dd = d;
    double items = 1;
    if (split > 0 && d > split) {
      items = std::ceil(d / split);
      dd = (double)split;
    }
    steps += cnt * items * (1.0 + std::ceil(dd / (g.E * U)));
  }
  const double maxd = (double)st.ints[2];
  double par = groups;
  if (sc.kind == AUTOSAGE_SCHED_MERGEPATH) {
    // one group per warp walks its rows one after another
    const double items = (double)sc.split;
    par = (double)std::max(1, dev.sms) * 48.0;
    steps += (n + nnz) / items * 4.0;
    longest = items / (g.E * U) + items / 4.0;
  } else {
    const double lmax = split > 0 && maxd > split ? (double)split : maxd;
    longest = 1.0 + std::ceil(lmax / (g.E * U));
  }
  const double t_lat = steps * lat / par;
  const double t_tail = longest * lat;
  double launches = 1;
  if ((sc.kind == AUTOSAGE_SCHED_SPLIT || sc.kind == AUTOSAGE_SCHED_BINNED || sc.kind == AUTOSAGE_SCHED_HYBRID) &&
      st.ints[6] > 0)
    launches += (op == AUTOSAGE_OP_SOFTMAX ? 3 : 1);
  if (sc.kind == AUTOSAGE_SCHED_MERGEPATH) launches += 1;
  if (op == AUTOSAGE_OP_ATTN_UNFUSED) launches += 2;
  return std::max(t_bw, t_lat) + t_tail + launches * 3e-6;
}

// ---------------------------------------------------------------- plan creation

autosage_status make_plan_shell(const autosage_csr *A, autosage_op op, int64_t F, int heads,
                                autosage_dtype dt, autosage_plan_s **out, cudaStream_t s) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (F < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "F must be >= 1");
  if (heads < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "heads must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  if (op < AUTOSAGE_OP_SPMM || op > AUTOSAGE_OP_ATTN_BACKWARD) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad op");
  auto *P = new autosage_plan_s();
  P->op = op;
  P->dt = static_cast<DType>(dt);
  P->F = (op == AUTOSAGE_OP_SOFTMAX) ? 1 : F;
  P->H = (op == AUTOSAGE_OP_ATTN || op == AUTOSAGE_OP_ATTN_UNFUSED || op == AUTOSAGE_OP_SOFTMAX ||
          op == AUTOSAGE_OP_ATTN_BACKWARD) ? heads : 1;
  P->n_rows = A->n_rows;
  P->n_cols = A->n_cols;
  P->nnz = A->nnz;
  P->a0 = *A;
  st = autosage_fingerprint(A, &P->a_fp, s);
  if (st != AUTOSAGE_OK) {
    delete P;
    return st;
  }
  P->k_rows = A->n_rows;
  P->k_row_ptr = A->row_ptr;
  P->k_col_idx = A->col_idx;
  if (op == AUTOSAGE_OP_SPMM_T) {
    // the structure of A^T and the permutation that carries each call's
    // edge values into A^T's order
    cudaError_t e = P->t_row_ptr.alloc(sizeof(int32_t) * (size_t)(A->n_cols + 1));
    if (e == cudaSuccess) e = P->t_col_idx.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(A->nnz, 1));
    if (e == cudaSuccess) e = P->t_vals.alloc(sizeof(float) * (size_t)std::max<int64_t>(A->nnz, 1));
    if (e == cudaSuccess) e = P->t_perm.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(A->nnz, 1));
    if (e == cudaSuccess)
      e = csr_transpose(A->n_rows, A->n_cols, A->nnz, A->row_ptr, A->col_idx, nullptr,
                        P->t_row_ptr.as<int32_t>(), P->t_col_idx.as<int32_t>(), nullptr,
                        P->t_perm.as<int32_t>(), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
      delete P;
      return cuda_fail(e, "building A^T");
    }
    P->k_rows = A->n_cols;
    P->k_row_ptr = P->t_row_ptr.as<int32_t>();
    P->k_col_idx = P->t_col_idx.as<int32_t>();
  }
  *out = P;
  return AUTOSAGE_OK;
}

// Probe buffers shaped like the op's real arguments (never the caller's data).
struct ProbeBufs {
  DevBuf X, Y, Y2, Q, K, S, flush;
  OpArgs a;
  int64_t out_elems = 0;
  bool out_is_S = false;
};

autosage_status make_probe_bufs(const autosage_plan_s *P, ProbeBufs &pb, cudaStream_t s) {
  const int es = dtype_size(P->dt);
  const int64_t F = P->F, H = P->H, W = F * H;
  const int64_t src_rows = (P->op == AUTOSAGE_OP_SPMM_T) ? P->n_rows : P->n_cols;
  const int64_t dst_rows = P->k_rows;
  auto alloc_fill = [&](DevBuf &b, int64_t elems, DType dt, uint64_t seed) -> cudaError_t {
    cudaError_t e = b.alloc((size_t)std::max<int64_t>(elems, 1) * (dt == DType::F32 ? 4 : 2));
    if (e == cudaSuccess) e = fill_probe(b.p, elems, dt, seed, s);
    return e;
  };
  cudaError_t e = cudaSuccess;
  switch (P->op) {
    case AUTOSAGE_OP_SPMM:
    case AUTOSAGE_OP_SPMM_T:
      e = alloc_fill(pb.X, src_rows * F, P->dt, 1);
      if (e == cudaSuccess) e = pb.Y.alloc((size_t)std::max<int64_t>(dst_rows * F, 1) * es);
      if (e == cudaSuccess) e = pb.Y2.alloc((size_t)std::max<int64_t>(dst_rows * F, 1) * es);
      pb.a.X = pb.X.p; pb.a.ldx = F; pb.a.Y = pb.Y.p; pb.a.ldy = F;
      pb.out_elems = dst_rows * F;
      break;
    case AUTOSAGE_OP_SDDMM:
      e = alloc_fill(pb.Q, P->n_rows * F, P->dt, 2);
      if (e == cudaSuccess) e = alloc_fill(pb.K, P->n_cols * F, P->dt, 3);
      if (e == cudaSuccess) e = pb.Y.alloc((size_t)std::max<int64_t>(P->nnz, 1) * 4);
      if (e == cudaSuccess) e = pb.Y2.alloc((size_t)std::max<int64_t>(P->nnz, 1) * 4);
      pb.a.Q = pb.Q.p; pb.a.ldq = F; pb.a.K = pb.K.p; pb.a.ldk = F; pb.a.S = pb.Y.as<float>();
      pb.out_elems = P->nnz;
      pb.out_is_S = true;
      break;
    case AUTOSAGE_OP_SOFTMAX:
      e = alloc_fill(pb.S, P->nnz * H, DType::F32, 4);
      if (e == cudaSuccess) e = pb.Y.alloc((size_t)std::max<int64_t>(P->nnz * H, 1) * 4);
      if (e == cudaSuccess) e = pb.Y2.alloc((size_t)std::max<int64_t>(P->nnz * H, 1) * 4);
      pb.a.S = pb.Y.as<float>();
      pb.out_elems = P->nnz * H;
      pb.out_is_S = true;
      break;
    case AUTOSAGE_OP_ATTN:
    case AUTOSAGE_OP_ATTN_UNFUSED:
      e = alloc_fill(pb.Q, P->n_rows * W, P->dt, 5);
      if (e == cudaSuccess) e = alloc_fill(pb.K, P->n_cols * W, P->dt, 6);
      if (e == cudaSuccess) e = alloc_fill(pb.X, P->n_cols * W, P->dt, 7);
      if (e == cudaSuccess) e = pb.Y.alloc((size_t)std::max<int64_t>(P->n_rows * W, 1) * es);
      if (e == cudaSuccess) e = pb.Y2.alloc((size_t)std::max<int64_t>(P->n_rows * W, 1) * es);
      pb.a.Q = pb.Q.p; pb.a.K = pb.K.p; pb.a.X = pb.X.p; pb.a.Y = pb.Y.p;
      pb.a.alpha = 1.f / std::sqrt((float)F);
      pb.out_elems = P->n_rows * W;
      break;
  }
  // a buffer twice the L2 size, overwritten before every timed run so probes
  // see the cold-cache behaviour the operations meet in a real step
  if (e == cudaSuccess) {
    int dev = 0, l2 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    e = pb.flush.alloc((size_t)std::max(l2, 1 << 20) * 2);
  }
  if (e != cudaSuccess) return cuda_fail(e, "probe buffers");
  return AUTOSAGE_OK;
}

// Host-side fault injection for tests of the guardrail (no GPU fault):
// AUTOSAGE_FAULT=probe_fail makes every probe report a failure,
// AUTOSAGE_FAULT=verify_fail makes every spot check report a mismatch.
bool fault(const char *name) {
  const char *f = getenv("AUTOSAGE_FAULT");
  return f && strcmp(f, name) == 0;
}

// Time one schedule: 1 warm-up, then `reps` timed runs, each after an
// overwrite of the L2-sized flush buffer, issued back to back (one host
// synchronisation at the end, as the operations of a step run); median in ms.
autosage_status probe_time(autosage_plan_s *P, ProbeBufs &pb, int reps, double &ms, cudaStream_t s) {
  if (fault("probe_fail")) return fail(AUTOSAGE_ERR_PROBE, "probe failure injected (AUTOSAGE_FAULT=probe_fail)");
  std::vector<cudaEvent_t> ev(2 * (size_t)(reps + 1), nullptr);
  autosage_status st = AUTOSAGE_OK;
  for (cudaEvent_t &e : ev)
    if (st == AUTOSAGE_OK && cudaEventCreate(&e) != cudaSuccess) st = fail(AUTOSAGE_ERR_CUDA, "probe events");
  OpArgs a = pb.a;
  if (P->op == AUTOSAGE_OP_ATTN_UNFUSED) a.S = P->scores.as<float>();
  for (int r = 0; r <= reps && st == AUTOSAGE_OK; ++r) {
    if (P->op == AUTOSAGE_OP_SOFTMAX)
      cudaMemcpyAsync(pb.Y.p, pb.S.p, (size_t)pb.out_elems * 4, cudaMemcpyDeviceToDevice, s);
    if (pb.flush.p) cudaMemsetAsync(pb.flush.p, r & 0xff, pb.flush.bytes, s);
    cudaEventRecord(ev[2 * r], s);
    st = run_op(P, P->op, &P->a0, a, s);
    cudaEventRecord(ev[2 * r + 1], s);
  }
  std::vector<float> t;
  if (st == AUTOSAGE_OK) {
    const cudaError_t e = cudaEventSynchronize(ev.back());
    if (e != cudaSuccess) st = cuda_fail(e, "probe");
    for (int r = 1; r <= reps && st == AUTOSAGE_OK; ++r) {
      float x = 0;
      cudaEventElapsedTime(&x, ev[2 * r], ev[2 * r + 1]);
      t.push_back(x);
    }
  } else {
    cudaStreamSynchronize(s);
  }
  for (cudaEvent_t e : ev)
    if (e) cudaEventDestroy(e);
  if (st != AUTOSAGE_OK) return st;
  std::sort(t.begin(), t.end());
  ms = t[t.size() / 2];
  return AUTOSAGE_OK;
}

bool same_sched(const Sched &a, const Sched &b) {
  return a.kind == b.kind && a.G == b.G && a.E == b.E && a.split == b.split && a.pe == b.pe && a.G2 == b.G2;
}

struct Candidate {
  Sched sc;
  double est;
};

// Geometry of G feature lanes x E edge lanes for the op's width, as the
// candidate list and the estimate see it (fragment width from the row size).
// False when a lane would need more fragment slots than the kernels have.
bool cand_geom(const autosage_plan_s *P, int G, int E, Geom &g) {
  const OpShape sh = op_shape(P->op, P->F, P->H);
  const int s = dtype_size(P->dt);
  int vb = 16;
  while (vb > s && (P->F * s) % vb) vb >>= 1;
  const int64_t nfrag = std::max<int64_t>(1, (P->F * sh.H * s) / vb);
  if (G < 1 || E < 1 || G * E > 32 || G > std::min<int64_t>(32, pow2ceil(nfrag))) return false;
  g = Geom{};
  g.dt = P->dt; g.H = sh.H; g.D = sh.D; g.VW = vb / s; g.nfrag = (int)nfrag; g.G = G; g.E = E;
  g.NV = pow2ceil((nfrag + G - 1) / G);
  // SpMM runs rows wider than 16 fragments per lane as column tiles of 8
  // fragments per lane, one launch after another: each launch is a candidate
  // of that geometry
  if ((P->op == AUTOSAGE_OP_SPMM || P->op == AUTOSAGE_OP_SPMM_T) && g.NV > 16) g.NV = 8;
  return g.NV <= sh.nv_max;
}

// Candidate schedules for the op and its statistics.
std::vector<Candidate> candidates(const DeviceInfo &dev, const autosage_plan_s *P, const RowStats &st) {
  std::vector<Candidate> out;
  const OpShape sh = op_shape(P->op, P->F, P->H);
  // lanes across features from the width (what choose_geom would pick)
  const int s = dtype_size(P->dt);
  int vb = 16;
  while (vb > s && (P->F * s) % vb) vb >>= 1;
  const int64_t nfrag = std::max<int64_t>(1, (P->F * sh.H * s) / vb);
  std::vector<int> Gs;
  const int G0 = std::min(32, pow2ceil(nfrag));
  Gs.push_back(G0);
  if (G0 > 1 && P->op != AUTOSAGE_OP_SOFTMAX) Gs.push_back(G0 / 2);
  // SDDMM with per-edge reductions ran fastest with four fragments a lane
  if (P->op == AUTOSAGE_OP_SDDMM && G0 >= 16) Gs.push_back(G0 / 4);
  const int64_t maxd = st.ints[2];
  for (int G : Gs) {
    if (P->op == AUTOSAGE_OP_SOFTMAX && G != G0) continue;
    for (int E = 1; G * E <= 32; E <<= 1) {
      if (P->op == AUTOSAGE_OP_SOFTMAX && E > 1) break;
      Geom g{};
      if (!cand_geom(P, G, E, g)) continue;
      Sched rg{AUTOSAGE_SCHED_ROWGROUP, G, E, 0};
      out.push_back({rg, estimate(dev, st, P->op, P->dt, P->F, sh.H, rg, g)});
      for (int split : {128, 512, 2048, 8192}) {
        if (maxd <= split) continue;
        Sched sp{AUTOSAGE_SCHED_SPLIT, G, E, split};
        out.push_back({sp, estimate(dev, st, P->op, P->dt, P->F, sh.H, sp, g)});
      }
      // degree-binned order pays off when lengths vary widely (coefficient of variation > 1)
      if (st.cv > 1.0 && P->op != AUTOSAGE_OP_SOFTMAX) {
        const int split = maxd > 128 ? 128 : (int)std::max<int64_t>(maxd, 1);
        Sched bn{AUTOSAGE_SCHED_BINNED, G, E, split};
        out.push_back({bn, estimate(dev, st, P->op, P->dt, P->F, sh.H, bn, g) * 0.97});
        // SpMM: the short rows (1..7 edges, degree buckets 1..3) in an ELL slab, when
        // they are at least a tenth of the rows and a row takes few lanes (small width)
        const int64_t short_rows = st.ints[9] + st.ints[10] + st.ints[11];
        if ((P->op == AUTOSAGE_OP_SPMM || P->op == AUTOSAGE_OP_SPMM_T) && G <= 8 && 10 * short_rows >= st.ints[0]) {
          Sched hy{AUTOSAGE_SCHED_HYBRID, G, E, std::max(split, kEllMaxDegree + 1)};
          out.push_back({hy, estimate(dev, st, P->op, P->dt, P->F, sh.H, hy, g) * 0.97});
        }
      }
      if (((P->op == AUTOSAGE_OP_SPMM || P->op == AUTOSAGE_OP_SPMM_T) && G * E == 32) || P->op == AUTOSAGE_OP_SDDMM) {
        for (int items : {256, 1024}) {
          Sched mp{AUTOSAGE_SCHED_MERGEPATH, G, E, items};
          out.push_back({mp, estimate(dev, st, P->op, P->dt, P->F, sh.H, mp, g)});
        }
      }
    }
  }
  // single-head SDDMM: every candidate with 4 or more feature lanes also with
  // per-edge reductions (measured: faster on uniform rows at F >= 64, slower
  // on skewed rows and at small F; the estimate does not tell them apart)
  if (P->op == AUTOSAGE_OP_SDDMM) {
    const size_t n = out.size();
    for (size_t i = 0; i < n; ++i) {
      if (out[i].sc.G < 4) continue;
      Candidate c = out[i];
      c.sc.pe = 1;
      out.push_back(c);
    }
  }
  std::stable_sort(out.begin(), out.end(), [](const Candidate &a, const Candidate &b) { return a.est < b.est; });
  return out;
}

// Neighbours of a schedule for the probes' local refinement: half or twice
// the edge lanes, half or twice the feature lanes, a quarter or four times
// the chunk length (merge path: the items per warp), the other chunked
// family (split <-> binned) with the same lanes and chunk length, for
// SDDMM the other reduction form (per edge <-> batched), and for unfused
// attention half or twice the aggregation stage's feature lanes. Automatic
// lanes (0) are first resolved the way the kernels resolve them.
std::vector<Candidate> neighbours(const DeviceInfo &dev, const autosage_plan_s *P, const RowStats &st,
                                  const Sched &b) {
  std::vector<Candidate> out;
  const OpShape sh = op_shape(P->op, P->F, P->H);
  const int64_t maxd = st.ints[2];
  const bool softmax = P->op == AUTOSAGE_OP_SOFTMAX;
  int G = b.G, E = b.E;
  if (G <= 0 || E <= 0) {
    const int s = dtype_size(P->dt);
    int vb = 16;
    while (vb > s && (P->F * s) % vb) vb >>= 1;
    const int64_t nfrag = std::max<int64_t>(1, (P->F * sh.H * s) / vb);
    if (G <= 0) G = std::min(32, pow2ceil(nfrag));
    if (E <= 0) E = std::max(1, std::min(32 / G, 8));
  }
  auto add = [&](Sched x) {
    Geom g{};
    if (!cand_geom(P, x.G, x.E, g)) return;
    if (P->op != AUTOSAGE_OP_SDDMM || x.G < 4) x.pe = 0;
    if (P->op != AUTOSAGE_OP_ATTN_UNFUSED || x.G2 == x.G) x.G2 = 0;
    Geom ga{};
    if (x.G2 > 0 && !cand_geom(P, x.G2, x.E, ga)) return;
    if (softmax && x.E != 1) return;
    if (x.kind == AUTOSAGE_SCHED_MERGEPATH) {
      const bool spmm = P->op == AUTOSAGE_OP_SPMM || P->op == AUTOSAGE_OP_SPMM_T;
      if ((spmm && x.G * x.E != 32) || (!spmm && P->op != AUTOSAGE_OP_SDDMM)) return;
      if (x.split < 64 || x.split > 16384) return;
    } else if (x.kind == AUTOSAGE_SCHED_SPLIT) {
      if (x.split < 16 || x.split >= maxd) return;
    } else if (x.kind == AUTOSAGE_SCHED_BINNED) {
      if (softmax || x.split < 16) return;
    } else if (x.kind == AUTOSAGE_SCHED_HYBRID) {
      if ((P->op != AUTOSAGE_OP_SPMM && P->op != AUTOSAGE_OP_SPMM_T) || x.split < 16) return;
    } else {
      x.split = 0;
    }
    for (const Candidate &c : out)
      if (same_sched(c.sc, x)) return;
    out.push_back({x, estimate(dev, st, P->op, P->dt, P->F, sh.H, x, g)});
  };
  for (int e2 : {E / 2, E * 2}) {
    if (e2 < 1 || e2 > 32) continue;
    // SpMM's merge path keeps whole warps: the feature lanes follow the edge lanes
    const bool whole = b.kind == AUTOSAGE_SCHED_MERGEPATH && P->op != AUTOSAGE_OP_SDDMM;
    add(Sched{b.kind, whole ? 32 / e2 : G, e2, b.split, b.pe, b.G2});
  }
  if ((b.kind != AUTOSAGE_SCHED_MERGEPATH || P->op == AUTOSAGE_OP_SDDMM) && !softmax)
    for (int g2 : {G / 2, G * 2})
      if (g2 >= 1) add(Sched{b.kind, g2, E, b.split, b.pe, b.G2});
  if (b.kind != AUTOSAGE_SCHED_ROWGROUP)
    for (int s2 : {b.split / 4, b.split * 4}) add(Sched{b.kind, G, E, s2, b.pe, b.G2});
  if (b.kind == AUTOSAGE_SCHED_SPLIT) add(Sched{AUTOSAGE_SCHED_BINNED, G, E, b.split, b.pe, b.G2});
  if (b.kind == AUTOSAGE_SCHED_BINNED) add(Sched{AUTOSAGE_SCHED_SPLIT, G, E, b.split, b.pe, b.G2});
  if (b.kind == AUTOSAGE_SCHED_BINNED) add(Sched{AUTOSAGE_SCHED_HYBRID, G, E, b.split, b.pe, b.G2});
  if (b.kind == AUTOSAGE_SCHED_HYBRID) add(Sched{AUTOSAGE_SCHED_BINNED, G, E, b.split, b.pe, b.G2});
  if (b.kind == AUTOSAGE_SCHED_ROWGROUP && maxd > 128) add(Sched{AUTOSAGE_SCHED_BINNED, G, E, 128, b.pe, b.G2});
  if (P->op == AUTOSAGE_OP_SDDMM) add(Sched{b.kind, G, E, b.split, 1 - b.pe, b.G2});
  // unfused attention: half or twice the aggregation stage's feature lanes
  if (P->op == AUTOSAGE_OP_ATTN_UNFUSED) {
    const int Ga = b.G2 > 0 ? b.G2 : G;
    for (int ga : {Ga / 2, Ga * 2})
      if (ga >= 1 && ga <= 32) add(Sched{b.kind, G, E, b.split, b.pe, ga});
  }
  return out;
}

void log_line(const char *fmt, ...) {
  const char *path = getenv("AUTOSAGE_LOG");
  if (!path || !*path) return;
  FILE *f = fopen(path, "a");
  if (!f) return;
  va_list ap;
  va_start(ap, fmt);
  vfprintf(f, fmt, ap);
  va_end(ap);
  fputc('\n', f);
  fclose(f);
}

// The backward plan: the forward-direction workspace (weights, dW/dS, chunk
// lists of A) plus an SpMM plan over A^T (transposed CSR, edge permutation,
// its own chunk lists). Rows longer than the chunk length are cut in both
// directions; shorter rows run whole, so one chunk length serves every graph.
autosage_status build_backward_plan(autosage_plan_s *P, const Sched &sc, cudaStream_t s) {
  P->sched = sc;
  if (P->sched.kind == AUTOSAGE_SCHED_MERGEPATH) P->sched = Sched{AUTOSAGE_SCHED_SPLIT, sc.G, sc.E, sc.split};
  autosage_status st = build_workspace(P, s);
  if (st != AUTOSAGE_OK) return st;
  autosage_plan_s *T = nullptr;
  st = make_plan_shell(&P->a0, AUTOSAGE_OP_SPMM_T, P->F * P->H, 1, static_cast<autosage_dtype>(P->dt), &T, s);
  if (st != AUTOSAGE_OK) return st;
  T->sched = Sched{P->sched.kind, 0, 0, P->sched.split};
  st = build_workspace(T, s);
  if (st != AUTOSAGE_OK) {
    delete T;
    return st;
  }
  // dV and dK run as one two-product pass: partials of both outputs for cut rows
  if (T->cl.n_chunks > 0) {
    const cudaError_t e = T->partial.alloc(sizeof(float) * (size_t)(2 * (int64_t)T->cl.n_chunks * T->F));
    if (e != cudaSuccess) {
      delete T;
      return cuda_fail(e, "backward partials");
    }
  }
  delete P->tplan;
  P->tplan = T;
  // where each edge of A sits in A^T: the backward writes w and dS there directly
  CUDA_TRY(P->t_inv.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(P->nnz, 1)));
  CUDA_TRY(launch_invert_perm(P->nnz, T->t_perm.as<int32_t>(), P->t_inv.as<int32_t>(), s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return AUTOSAGE_OK;
}

// The backward's schedule: rows in degree-binned order, rows longer than 512
// edges cut (measured on the R-MAT scale-20 graph, H = 8, D = 64, bf16: 15.4 ms
// against 16.8 ms for split rows of 128 in plain order).
Sched default_backward_sched() { return Sched{AUTOSAGE_SCHED_BINNED, 0, 0, 512}; }

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char *autosage_version(void) { return "autosage-gb300 0.1"; }

const char *autosage_status_string(autosage_status s) {
  switch (s) {
    case AUTOSAGE_OK: return "ok";
    case AUTOSAGE_ERR_INVALID_ARG: return "invalid argument";
    case AUTOSAGE_ERR_INVALID_CSR: return "invalid CSR structure";
    case AUTOSAGE_ERR_UNSUPPORTED: return "unsupported shape";
    case AUTOSAGE_ERR_CUDA: return "CUDA error";
    case AUTOSAGE_ERR_CACHE_IO: return "cache file I/O error";
    case AUTOSAGE_ERR_CACHE_FORMAT: return "cache file format error";
    case AUTOSAGE_ERR_PROBE: return "every probed schedule failed";
    case AUTOSAGE_ERR_PLAN_MISMATCH: return "plan does not match the call";
  }
  return "unknown status";
}

const char *autosage_last_error(void) { return g_last_error.c_str(); }

autosage_status autosage_plan_with_schedule(const autosage_csr *A, autosage_op op, int64_t F, int heads,
                                            autosage_dtype dt, const autosage_schedule *sched,
                                            autosage_plan_t *out, void *stream) {
  if (!out) return fail(AUTOSAGE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!sched) return fail(AUTOSAGE_ERR_INVALID_ARG, "sched is NULL");
  if (sched->kind < AUTOSAGE_SCHED_ROWGROUP || sched->kind > AUTOSAGE_SCHED_HYBRID)
    return fail(AUTOSAGE_ERR_INVALID_ARG, "bad schedule kind");
  if ((sched->lanes_f && !is_pow2(sched->lanes_f)) || (sched->lanes_e && !is_pow2(sched->lanes_e)) ||
      sched->lanes_f > 32 || sched->lanes_e > 32 || sched->lanes_f * std::max(1, sched->lanes_e) > 32)
    return fail(AUTOSAGE_ERR_INVALID_ARG, "lanes must be powers of two with lanes_f * lanes_e <= 32");
  if (sched->split < 0) return fail(AUTOSAGE_ERR_INVALID_ARG, "negative split");
  if (sched->lanes_f_agg && (op != AUTOSAGE_OP_ATTN_UNFUSED || !is_pow2(sched->lanes_f_agg) ||
                             sched->lanes_f_agg * std::max(1, sched->lanes_e) > 32))
    return fail(AUTOSAGE_ERR_INVALID_ARG,
                "lanes_f_agg: unfused attention only, a power of two with lanes_f_agg * lanes_e <= 32");
  cudaStream_t s = as_stream(stream);
  autosage_plan_s *P = nullptr;
  autosage_status st = make_plan_shell(A, op, F, heads, dt, &P, s);
  if (st != AUTOSAGE_OK) return st;
  P->sched = Sched{sched->kind, sched->lanes_f, sched->lanes_e, sched->split, sched->per_edge ? 1 : 0,
                   sched->lanes_f_agg == sched->lanes_f ? 0 : sched->lanes_f_agg};
  if ((P->sched.kind == AUTOSAGE_SCHED_SPLIT || P->sched.kind == AUTOSAGE_SCHED_BINNED ||
       P->sched.kind == AUTOSAGE_SCHED_HYBRID) && P->sched.split == 0)
    P->sched.split = 1024;
  if (P->sched.kind == AUTOSAGE_SCHED_MERGEPATH && P->sched.split == 0) P->sched.split = 512;
  if (P->sched.kind == AUTOSAGE_SCHED_ROWGROUP) P->sched.split = 0;
  if (op == AUTOSAGE_OP_ATTN_BACKWARD) {
    st = build_backward_plan(P, P->sched, s);
    if (st != AUTOSAGE_OK) {
      delete P;
      return st;
    }
    *out = P;
    return AUTOSAGE_OK;
  }
  st = build_workspace(P, s);
  if (st != AUTOSAGE_OK) {
    delete P;
    return st;
  }
  *out = P;
  return AUTOSAGE_OK;
}

autosage_status autosage_plan(const autosage_csr *A, autosage_op op, int64_t F, int heads,
                              autosage_dtype dt, unsigned flags, autosage_plan_t *out, void *stream) {
  if (!out) return fail(AUTOSAGE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  cudaStream_t s = as_stream(stream);
  autosage_plan_s *P = nullptr;
  autosage_status st = make_plan_shell(A, op, F, heads, dt, &P, s);
  if (st != AUTOSAGE_OK) return st;
  if ((flags & AUTOSAGE_PLAN_FIXED_VALUES) && (st = fix_values(P, A, s)) != AUTOSAGE_OK) {
    delete P;
    return st;
  }
  if (op == AUTOSAGE_OP_ATTN_BACKWARD) {  // fixed schedule (no probes)
    st = build_backward_plan(P, default_backward_sched(), s);
    if (st != AUTOSAGE_OK) {
      delete P;
      return st;
    }
    *out = P;
    return AUTOSAGE_OK;
  }
  const DeviceInfo dev = device_info();
  // structure statistics and fingerprint of the CSR the kernels walk
  RowStats rs;
  st = gpu_row_stats(P->k_rows, P->k_row_ptr, 1024, rs, s);
  if (st != AUTOSAGE_OK) {
    delete P;
    return st;
  }
  // the cache key holds the fingerprint of the walked CSR (A^T for SPMM_T)
  uint64_t fp = P->a_fp;
  if (op == AUTOSAGE_OP_SPMM_T) {
    autosage_csr K{P->k_rows, A->n_rows, P->nnz, P->k_row_ptr, P->k_col_idx, nullptr};
    st = autosage_fingerprint(&K, &fp, stream);
    if (st != AUTOSAGE_OK) {
      delete P;
      return st;
    }
  }
  const std::string key = cache_key(dev, op, P->dt, P->F, P->H, A->n_rows, A->n_cols, A->nnz, fp);
  const bool use_cache = !(flags & AUTOSAGE_PLAN_NO_CACHE);
  if (use_cache) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    auto it = g_cache.find(key);
    if (it != g_cache.end()) {
      P->sched = it->second.sched;
      P->probe_ms = it->second.probe_ms;
      P->from_cache = true;
    }
  }
  if (P->from_cache) {
    st = build_workspace(P, s);
    if (st == AUTOSAGE_OK) {
      log_line("plan key=%s cache-hit %s G=%d E=%d split=%d", key.c_str(), sched_name(P->sched.kind),
               P->sched.G, P->sched.E, P->sched.split);
      *out = P;
      return AUTOSAGE_OK;
    }
    // a stale entry falls through to a fresh choice
    P->from_cache = false;
  }
  std::vector<Candidate> cands = candidates(dev, P, rs);
  const bool probe = (flags & AUTOSAGE_PLAN_PROBE) != 0;
  const bool verify = (flags & AUTOSAGE_PLAN_VERIFY) != 0;
  Sched best = default_sched();
  double best_ms = -1, best_est = -1;
  autosage_status result = AUTOSAGE_OK;
  if (!probe) {
    if (!cands.empty()) {
      best = cands[0].sc;
      best_est = cands[0].est;
    }
  } else {
    // probes: the best-estimated candidate of each family and lane count, then
    // the next best overall up to ten, plus the guardrail default
    std::vector<Candidate> top;
    auto have = [&](const Sched &x) {
      for (const Candidate &t : top)
        if (same_sched(t.sc, x)) return true;
      return false;
    };
    // the estimate ranks lane counts poorly, so every (family, feature lanes)
    // pair sends its best candidate to the probes
    for (int kind : {AUTOSAGE_SCHED_ROWGROUP, AUTOSAGE_SCHED_SPLIT, AUTOSAGE_SCHED_MERGEPATH, AUTOSAGE_SCHED_BINNED,
                     AUTOSAGE_SCHED_HYBRID}) {
      std::vector<int> seen_g;
      for (const Candidate &c : cands) {
        const int gk = c.sc.G * 2 + c.sc.pe;
        if (c.sc.kind != kind || std::find(seen_g.begin(), seen_g.end(), gk) != seen_g.end()) continue;
        seen_g.push_back(gk);
        top.push_back(c);
      }
    }
    for (const Candidate &c : cands) {
      if ((int)top.size() >= 10) break;
      if (!have(c.sc)) top.push_back(c);
    }
    if (!have(default_sched())) top.push_back({default_sched(), -1});
    ProbeBufs pb;
    st = make_probe_bufs(P, pb, s);
    if (st != AUTOSAGE_OK) {
      delete P;
      return st;
    }
    // the guardrail's output for the spot check
    bool have_ref = false;
    if (verify) {
      P->sched = default_sched();
      if (build_workspace(P, s) == AUTOSAGE_OK) {
        OpArgs a = pb.a;
        if (op == AUTOSAGE_OP_ATTN_UNFUSED) a.S = P->scores.as<float>();
        if (op == AUTOSAGE_OP_SOFTMAX)
          cudaMemcpyAsync(pb.Y.p, pb.S.p, (size_t)pb.out_elems * 4, cudaMemcpyDeviceToDevice, s);
        if (run_op(P, op, &P->a0, a, s) == AUTOSAGE_OK && cudaStreamSynchronize(s) == cudaSuccess) {
          const size_t bytes = (size_t)pb.out_elems * (pb.out_is_S ? 4 : dtype_size(P->dt));
          have_ref = cudaMemcpyAsync(pb.Y2.p, pb.Y.p, bytes, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
        }
      }
    }
    int ok_count = 0;
    // every schedule that passed its probe, with its time (for the final round)
    std::vector<std::pair<double, Candidate>> passed;
    // fastest schedule of each reduction form (SDDMM: batched, per edge)
    double form_ms[2] = {-1, -1};
    Sched form_best[2];
    auto probe_one = [&](const Candidate &c) {
      P->sched = c.sc;
      if (build_workspace(P, s) != AUTOSAGE_OK) {
        log_line("plan key=%s skip %s G=%d E=%d split=%d workspace: %s", key.c_str(), sched_name(c.sc.kind),
                 c.sc.G, c.sc.E, c.sc.split, g_last_error.c_str());
        return;
      }
      double ms = 0;
      if (probe_time(P, pb, 5, ms, s) != AUTOSAGE_OK) {
        log_line("plan key=%s skip %s G=%d E=%d split=%d probe: %s", key.c_str(), sched_name(c.sc.kind),
                 c.sc.G, c.sc.E, c.sc.split, g_last_error.c_str());
        return;
      }
      if (verify && have_ref && !same_sched(c.sc, default_sched())) {
        unsigned long long *cnt = nullptr, h = 1;
        if (cudaMallocAsync(&cnt, sizeof *cnt, s) == cudaSuccess) {
          // two fp32 kernels summing in different orders differ by rounding only; a
          // broken schedule is off by O(1), so the spot check is looser than parity
          const DType cdt = pb.out_is_S ? DType::F32 : P->dt;
          const float rtol = cdt == DType::F32 ? 1e-3f : 5e-2f;
          launch_compare(pb.Y.p, pb.Y2.p, pb.out_elems, cdt, rtol, rtol, cnt, s);
          cudaMemcpyAsync(&h, cnt, sizeof h, cudaMemcpyDeviceToHost, s);
          cudaFreeAsync(cnt, s);
          cudaStreamSynchronize(s);
        }
        if (fault("verify_fail")) h = 1;
        if (h != 0) {
          log_line("plan key=%s reject %s G=%d E=%d split=%d mismatches=%llu", key.c_str(),
                   sched_name(c.sc.kind), c.sc.G, c.sc.E, c.sc.split, h);
          return;
        }
      }
      ++ok_count;
      passed.push_back({ms, c});
      log_line("plan key=%s probe %s G=%d E=%d split=%d pe=%d agg=%d est_ms=%.4f probe_ms=%.4f", key.c_str(),
               sched_name(c.sc.kind), c.sc.G, c.sc.E, c.sc.split, c.sc.pe, c.sc.G2, c.est * 1e3, ms);
      if (best_ms < 0 || ms < best_ms) {
        best_ms = ms;
        best = c.sc;
        best_est = c.est;
      }
      const int f = c.sc.pe ? 1 : 0;
      if (form_ms[f] < 0 || ms < form_ms[f]) {
        form_ms[f] = ms;
        form_best[f] = c.sc;
      }
    };
    for (const Candidate &c : top) probe_one(c);
    // local refinement: the estimate ranks edge lanes and chunk lengths
    // poorly, so the neighbours of the fastest schedules are probed too: each
    // round expands the three fastest schedules of a reduction form that were
    // not expanded yet (a beam, since the best schedule can be two steps away
    // through a slightly slower one), at most four rounds, stopping when a
    // round finds nothing faster (separately for each reduction form: their
    // best lane counts differ)
    std::vector<Sched> tried, expanded;
    auto seen = [](const std::vector<Sched> &v, const Sched &x) {
      return std::any_of(v.begin(), v.end(), [&](const Sched &t) { return same_sched(t, x); });
    };
    for (const Candidate &c : top) tried.push_back(c.sc);
    for (int f = 0; f < 2; ++f) {
      for (int round = 0; round < 4 && form_ms[f] >= 0; ++round) {
        const double before = form_ms[f];
        std::vector<std::pair<double, Sched>> beam;
        for (const auto &pc : passed)
          if ((pc.second.sc.pe ? 1 : 0) == f && !seen(expanded, pc.second.sc)) beam.push_back({pc.first, pc.second.sc});
        std::stable_sort(beam.begin(), beam.end(), [](const std::pair<double, Sched> &x,
                                                      const std::pair<double, Sched> &y) { return x.first < y.first; });
        if (beam.size() > 3) beam.resize(3);
        if (beam.empty()) break;
        for (const auto &centre : beam) {
          expanded.push_back(centre.second);
          for (const Candidate &c : neighbours(dev, P, rs, centre.second)) {
            if ((c.sc.pe ? 1 : 0) != f || seen(tried, c.sc)) continue;
            tried.push_back(c.sc);
            probe_one(c);
          }
        }
        if (!(form_ms[f] < before)) break;
      }
    }
    // final round: the three fastest schedules timed again with more runs, so
    // that one lucky (or unlucky) median of five does not decide the plan
    std::stable_sort(passed.begin(), passed.end(),
                     [](const std::pair<double, Candidate> &x, const std::pair<double, Candidate> &y) {
                       return x.first < y.first;
                     });
    if (passed.size() > 1) {
      double final_ms = -1;
      for (size_t i = 0; i < passed.size() && i < 3; ++i) {
        const Candidate &c = passed[i].second;
        P->sched = c.sc;
        double ms = 0;
        if (build_workspace(P, s) != AUTOSAGE_OK || probe_time(P, pb, 11, ms, s) != AUTOSAGE_OK) continue;
        log_line("plan key=%s final %s G=%d E=%d split=%d pe=%d agg=%d probe_ms=%.4f", key.c_str(),
                 sched_name(c.sc.kind), c.sc.G, c.sc.E, c.sc.split, c.sc.pe, c.sc.G2, ms);
        if (final_ms < 0 || ms < final_ms) {
          final_ms = ms;
          best = c.sc;
          best_est = c.est;
          best_ms = ms;
        }
      }
    }
    cudaGetLastError();  // a failed candidate must not poison later calls
    if (ok_count == 0) {
      best = default_sched();
      result = fail(AUTOSAGE_ERR_PROBE, "every probed schedule failed; using the default");
    }
  }
  P->sched = best;
  P->probe_ms = best_ms;
  P->est_ms = best_est >= 0 ? best_est * 1e3 : -1;
  st = build_workspace(P, s);
  if (st != AUTOSAGE_OK && !same_sched(best, default_sched())) {
    P->sched = default_sched();
    st = build_workspace(P, s);
  }
  if (st != AUTOSAGE_OK) {
    delete P;
    return st;
  }
  if (use_cache && (probe || !cands.empty())) {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    g_cache[key] = CacheEntry{P->sched, P->probe_ms};
  }
  log_line("plan key=%s choose %s G=%d E=%d split=%d est_ms=%.4f probe_ms=%.4f", key.c_str(),
           sched_name(P->sched.kind), P->sched.G, P->sched.E, P->sched.split, P->est_ms, P->probe_ms);
  *out = P;
  return result;
}

autosage_status autosage_plan_destroy(autosage_plan_t plan) {
  if (!plan) return AUTOSAGE_OK;
  cudaDeviceSynchronize();
  delete plan;
  return AUTOSAGE_OK;
}

autosage_status autosage_plan_describe(autosage_plan_t P, char *buf, size_t len) {
  if (!P || !buf || len == 0) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad describe arguments");
  snprintf(buf, len, "op=%d sched=%s G=%d E=%d split=%d chunks=%d long_rows=%d mp_warps=%" PRId64
           " probe_ms=%.4f est_ms=%.4f cache=%d per_edge=%d fixed_vals=%d agg_lanes=%d",
           (int)P->op, sched_name(P->sched.kind), P->sched.G, P->sched.E, P->sched.split, P->cl.n_chunks,
           P->cl.n_long, P->mp_warps, P->probe_ms, P->est_ms, P->from_cache ? 1 : 0, P->sched.pe,
           P->fixed_vals ? 1 : 0, P->sched.G2);
  return AUTOSAGE_OK;
}

autosage_status autosage_plan_schedule(autosage_plan_t P, autosage_schedule *sched, double *probe_ms) {
  if (!P) return fail(AUTOSAGE_ERR_INVALID_ARG, "plan is NULL");
  if (sched) {
    sched->kind = P->sched.kind;
    sched->lanes_f = P->sched.G;
    sched->lanes_e = P->sched.E;
    sched->split = P->sched.split;
    sched->per_edge = P->sched.pe;
    sched->lanes_f_agg = P->sched.G2;
  }
  if (probe_ms) *probe_ms = P->probe_ms;
  return AUTOSAGE_OK;
}

autosage_status autosage_plan_rebind(autosage_plan_t P, const autosage_csr *A, void *stream) {
  if (!P) return fail(AUTOSAGE_ERR_INVALID_ARG, "plan is NULL");
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (P->typed) return fail(AUTOSAGE_ERR_UNSUPPORTED, "typed plans cannot be rebound; build a new one");
  if (P->n_rows != A->n_rows || P->n_cols != A->n_cols || P->nnz != A->nnz)
    return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "plan built for a graph of another size");
  uint64_t fp = 0;
  if ((st = autosage_fingerprint(A, &fp, stream)) != AUTOSAGE_OK) return st;
  if (fp != P->a_fp) return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "A has another structure than the plan's graph");
  if (P->fixed_vals && (st = fix_values(P, A, as_stream(stream))) != AUTOSAGE_OK) return st;
  P->a0 = *A;
  if (P->op != AUTOSAGE_OP_SPMM_T) {
    P->k_row_ptr = A->row_ptr;
    P->k_col_idx = A->col_idx;
  }
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- ops

static bool check_mode() {
  const char *c = getenv("AUTOSAGE_CHECK");
  return c && atoi(c) > 0;
}

// A plan's workspace (chunk lists, row order, A^T, merge-path partitions) is
// derived from the structure of the A it was built for, so a call must pass
// the same row_ptr and col_idx arrays; the edge values are read from the call.
// In checked mode the structure's fingerprint is compared as well, which
// catches arrays that were overwritten in place with another graph.
static autosage_status plan_matches(const autosage_plan_s *P, const autosage_csr *A, autosage_op op,
                                    int64_t F, int H, autosage_dtype dt, void *stream) {
  if (P->op != op) return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "plan built for op %d, called as op %d", (int)P->op, (int)op);
  if (P->typed) return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "a typed plan runs only through autosage_spmm_typed");
  if (P->n_rows != A->n_rows || P->n_cols != A->n_cols || P->nnz != A->nnz)
    return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "plan built for another graph");
  if (P->F != F || P->H != H || (int)P->dt != (int)dt)
    return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "plan built for another width, head count or dtype");
  if (A->row_ptr != P->a0.row_ptr || (A->nnz > 0 && A->col_idx != P->a0.col_idx))
    return fail(AUTOSAGE_ERR_PLAN_MISMATCH,
                "row_ptr / col_idx are not the arrays the plan was built for (after moving or copying the "
                "structure, call autosage_plan_rebind)");
  if (P->fixed_vals && A->vals != P->fixed_vals_ptr)
    return fail(AUTOSAGE_ERR_PLAN_MISMATCH,
                "the plan holds fixed edge values (AUTOSAGE_PLAN_FIXED_VALUES) of another array; pass that "
                "array, or call autosage_plan_rebind with the new one");
  if (check_mode()) {
    uint64_t fp = 0;
    autosage_status st = autosage_fingerprint(A, &fp, stream);
    if (st != AUTOSAGE_OK) return st;
    if (fp != P->a_fp)
      return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "the structure arrays changed since the plan was built");
  }
  return AUTOSAGE_OK;
}

// A transient plan with the default schedule and no workspace.
static autosage_plan_s transient(const autosage_csr *A, autosage_op op, int64_t F, int H, autosage_dtype dt) {
  autosage_plan_s P;
  P.op = op;
  P.dt = static_cast<DType>(dt);
  P.F = F;
  P.H = H;
  P.n_rows = A->n_rows;
  P.n_cols = A->n_cols;
  P.nnz = A->nnz;
  P.a0 = *A;
  P.k_rows = A->n_rows;
  P.k_row_ptr = A->row_ptr;
  P.k_col_idx = A->col_idx;
  P.sched = default_sched();
  return P;
}

static autosage_status check_mat(const void *p, int64_t ld, int64_t width, int64_t rows, const char *name) {
  if (rows > 0 && !p) return fail(AUTOSAGE_ERR_INVALID_ARG, "%s is NULL", name);
  if (ld < width) return fail(AUTOSAGE_ERR_INVALID_ARG, "%s: leading dimension < width", name);
  return AUTOSAGE_OK;
}

autosage_status autosage_spmm(const autosage_csr *A, const void *X, int64_t ldx, void *Y, int64_t ldy,
                              int64_t F, autosage_dtype dt, int transpose, autosage_plan_t plan,
                              void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (F < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "F must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  const int64_t out_rows = transpose ? A->n_cols : A->n_rows;
  const int64_t in_rows = transpose ? A->n_rows : A->n_cols;
  if ((st = check_mat(X, ldx, F, in_rows, "X")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(Y, ldy, F, out_rows, "Y")) != AUTOSAGE_OK) return st;
  if (out_rows == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.X = X; a.ldx = ldx; a.Y = Y; a.ldy = ldy;
  const autosage_op op = transpose ? AUTOSAGE_OP_SPMM_T : AUTOSAGE_OP_SPMM;
  if (plan) {
    if ((st = plan_matches(plan, A, op, F, 1, dt, stream)) != AUTOSAGE_OK) return st;
    return run_op(plan, op, A, a, as_stream(stream));
  }
  if (transpose) return fail(AUTOSAGE_ERR_INVALID_ARG, "transpose needs a plan built for AUTOSAGE_OP_SPMM_T");
  autosage_plan_s P = transient(A, op, F, 1, dt);
  return run_op(&P, op, A, a, as_stream(stream));
}

autosage_status autosage_sddmm(const autosage_csr *A, const void *Q, int64_t ldq, const void *K, int64_t ldk,
                               int64_t F, autosage_dtype dt, float alpha, float *out, autosage_plan_t plan,
                               void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (F < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "F must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  if ((st = check_mat(Q, ldq, F, A->n_rows, "Q")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(K, ldk, F, A->n_cols, "K")) != AUTOSAGE_OK) return st;
  if (A->nnz > 0 && !out) return fail(AUTOSAGE_ERR_INVALID_ARG, "out is NULL");
  if (A->nnz == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.Q = Q; a.ldq = ldq; a.K = K; a.ldk = ldk; a.alpha = alpha; a.S = out;
  if (plan) {
    if ((st = plan_matches(plan, A, AUTOSAGE_OP_SDDMM, F, 1, dt, stream)) != AUTOSAGE_OK) return st;
    return run_op(plan, AUTOSAGE_OP_SDDMM, A, a, as_stream(stream));
  }
  autosage_plan_s P = transient(A, AUTOSAGE_OP_SDDMM, F, 1, dt);
  return run_op(&P, AUTOSAGE_OP_SDDMM, A, a, as_stream(stream));
}

autosage_status autosage_row_softmax(const autosage_csr *A, float *scores, int heads, autosage_plan_t plan,
                                     void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (heads < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "heads must be >= 1");
  if (A->nnz > 0 && !scores) return fail(AUTOSAGE_ERR_INVALID_ARG, "scores is NULL");
  if (A->nnz == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.S = scores;
  if (plan) {
    if ((st = plan_matches(plan, A, AUTOSAGE_OP_SOFTMAX, 1, heads, AUTOSAGE_F32, stream)) != AUTOSAGE_OK) return st;
    return run_op(plan, AUTOSAGE_OP_SOFTMAX, A, a, as_stream(stream));
  }
  autosage_plan_s P = transient(A, AUTOSAGE_OP_SOFTMAX, 1, heads, AUTOSAGE_F32);
  return run_op(&P, AUTOSAGE_OP_SOFTMAX, A, a, as_stream(stream));
}

autosage_status autosage_csr_attention(const autosage_csr *A, const void *Q, const void *K, const void *V,
                                       int heads, int64_t D, autosage_dtype dt, float scale, void *out,
                                       int fused, autosage_plan_t plan, void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (heads < 1 || D < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "heads and D must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  const int64_t W = (int64_t)heads * D;
  if ((st = check_mat(Q, W, W, A->n_rows, "Q")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(K, W, W, A->n_cols, "K")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(V, W, W, A->n_cols, "V")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(out, W, W, A->n_rows, "out")) != AUTOSAGE_OK) return st;
  if (A->n_rows == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.Q = Q; a.K = K; a.X = V; a.Y = out; a.alpha = scale;
  cudaStream_t s = as_stream(stream);
  const autosage_op op = fused ? AUTOSAGE_OP_ATTN : AUTOSAGE_OP_ATTN_UNFUSED;
  if (plan) {
    if ((st = plan_matches(plan, A, op, D, heads, dt, stream)) != AUTOSAGE_OK) return st;
    if (!fused) a.S = plan->scores.as<float>();
    return run_op(plan, op, A, a, s);
  }
  autosage_plan_s P = transient(A, op, D, heads, dt);
  if (fused) return run_op(&P, op, A, a, s);
  float *S = nullptr;
  cudaError_t e = cudaMallocAsync(&S, sizeof(float) * (size_t)std::max<int64_t>(A->nnz * heads, 1), s);
  if (e != cudaSuccess) return cuda_fail(e, "score buffer");
  a.S = S;
  st = run_op(&P, op, A, a, s);
  cudaFreeAsync(S, s);
  return st;
}

autosage_status autosage_edge_softmax_aggregate(const autosage_csr *A, const float *scores, const void *V,
                                                int heads, int64_t D, autosage_dtype dt, void *out,
                                                autosage_plan_t plan, void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (heads < 1 || D < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "heads and D must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  const int64_t W = (int64_t)heads * D;
  if (A->nnz > 0 && !scores) return fail(AUTOSAGE_ERR_INVALID_ARG, "scores is NULL");
  if ((st = check_mat(V, W, W, A->n_cols, "V")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(out, W, W, A->n_rows, "out")) != AUTOSAGE_OK) return st;
  if (A->n_rows == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.X = V; a.Y = out; a.given = scores;
  if (plan) {
    if ((st = plan_matches(plan, A, AUTOSAGE_OP_ATTN, D, heads, dt, stream)) != AUTOSAGE_OK) return st;
    return run_op(plan, AUTOSAGE_OP_ATTN, A, a, as_stream(stream));
  }
  autosage_plan_s P = transient(A, AUTOSAGE_OP_ATTN, D, heads, dt);
  return run_op(&P, AUTOSAGE_OP_ATTN, A, a, as_stream(stream));
}

autosage_status autosage_csr_attention_backward(const autosage_csr *A, const void *Q, const void *K,
                                                const void *V, const void *dO, int heads, int64_t D,
                                                autosage_dtype dt, float scale, void *dQ, void *dK,
                                                void *dV, autosage_plan_t plan, void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (heads < 1 || D < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "heads and D must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  const int64_t W = (int64_t)heads * D;
  if ((st = check_mat(Q, W, W, A->n_rows, "Q")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(dO, W, W, A->n_rows, "dO")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(dQ, W, W, A->n_rows, "dQ")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(K, W, W, A->n_cols, "K")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(V, W, W, A->n_cols, "V")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(dK, W, W, A->n_cols, "dK")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(dV, W, W, A->n_cols, "dV")) != AUTOSAGE_OK) return st;
  if (A->n_rows == 0 && A->n_cols == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.Q = Q; a.K = K; a.X = V; a.dO = dO; a.dQ = dQ; a.dK = dK; a.dV = dV; a.alpha = scale;
  cudaStream_t s = as_stream(stream);
  if (plan) {
    if ((st = plan_matches(plan, A, AUTOSAGE_OP_ATTN_BACKWARD, D, heads, dt, stream)) != AUTOSAGE_OK) return st;
    return run_op(plan, AUTOSAGE_OP_ATTN_BACKWARD, A, a, s);
  }
  autosage_plan_s *P = nullptr;
  st = make_plan_shell(A, AUTOSAGE_OP_ATTN_BACKWARD, D, heads, dt, &P, s);
  if (st != AUTOSAGE_OK) return st;
  st = build_backward_plan(P, default_backward_sched(), s);
  if (st == AUTOSAGE_OK) st = run_op(P, AUTOSAGE_OP_ATTN_BACKWARD, A, a, s);
  cudaError_t e = cudaStreamSynchronize(s);
  delete P;
  if (st == AUTOSAGE_OK && e != cudaSuccess) return cuda_fail(e, "attention backward");
  return st;
}

autosage_status autosage_plan_typed(const autosage_csr *A, const int32_t *edge_type, int num_types, int64_t F,
                                    autosage_dtype dt, unsigned flags, autosage_plan_t *out, void *stream) {
  if (!out) return fail(AUTOSAGE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (num_types < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "num_types must be >= 1");
  if (A->nnz > 0 && !edge_type) return fail(AUTOSAGE_ERR_INVALID_ARG, "edge_type is NULL");
  if ((int64_t)num_types * std::max<int64_t>(A->n_cols, 1) >= INT32_MAX)
    return fail(AUTOSAGE_ERR_UNSUPPORTED, "num_types * n_cols must fit int32");
  cudaStream_t s = as_stream(stream);
  DevBuf idx;
  CUDA_TRY(idx.alloc(sizeof(int32_t) * (size_t)std::max<int64_t>(A->nnz, 1)));
  int *derr = nullptr, herr = 0;
  CUDA_TRY(cudaMallocAsync(&derr, sizeof(int), s));
  cudaError_t e = launch_typed_index(A->nnz, A->n_cols, num_types, A->col_idx, edge_type, idx.as<int32_t>(), derr, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&herr, derr, sizeof(int), cudaMemcpyDeviceToHost, s);
  cudaFreeAsync(derr, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    idx.release();
    return cuda_fail(e, "typed index");
  }
  if (herr) {
    idx.release();
    return fail(AUTOSAGE_ERR_INVALID_ARG, "edge_type outside [0, num_types)");
  }
  // an ordinary SpMM plan over the stacked blocks: A' has num_types * n_cols columns
  autosage_csr Ap{A->n_rows, (int64_t)num_types * A->n_cols, A->nnz, A->row_ptr, idx.as<int32_t>(), A->vals};
  autosage_plan_t P = nullptr;
  st = autosage_plan(&Ap, AUTOSAGE_OP_SPMM, F, 1, dt, flags, &P, stream);
  if (!P) {
    idx.release();
    return st;
  }
  P->typed = num_types;
  P->base_cols = A->n_cols;
  P->typed_idx = idx;  // the plan owns the index from here on
  idx.p = nullptr;
  idx.bytes = 0;
  P->typed_col = A->col_idx;
  P->typed_type = edge_type;
  *out = P;
  return st;
}

autosage_status autosage_spmm_typed(const autosage_csr *A, const int32_t *edge_type, int num_types, const void *Z,
                                    int64_t ldz, void *Y, int64_t ldy, int64_t F, autosage_dtype dt,
                                    autosage_plan_t plan, void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (F < 1 || num_types < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "F and num_types must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  if ((st = check_mat(Z, ldz, F, (int64_t)num_types * A->n_cols, "Z")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(Y, ldy, F, A->n_rows, "Y")) != AUTOSAGE_OK) return st;
  if (A->n_rows == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.X = Z; a.ldx = ldz; a.Y = Y; a.ldy = ldy;
  cudaStream_t s = as_stream(stream);
  if (plan) {
    if (plan->typed != num_types || plan->base_cols != A->n_cols || plan->n_rows != A->n_rows ||
        plan->nnz != A->nnz || plan->F != F || (int)plan->dt != (int)dt || plan->op != AUTOSAGE_OP_SPMM)
      return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "plan not built by autosage_plan_typed for this call");
    // the combined gather index was built from these arrays: they are structure
    if (A->row_ptr != plan->a0.row_ptr || (A->nnz > 0 && (A->col_idx != plan->typed_col || edge_type != plan->typed_type)))
      return fail(AUTOSAGE_ERR_PLAN_MISMATCH,
                  "row_ptr / col_idx / edge_type are not the arrays the typed plan was built from");
    // the stacked relation blocks as one CSR: the plan's combined index, the call's values
    const autosage_csr Ap{A->n_rows, (int64_t)num_types * A->n_cols, A->nnz, A->row_ptr,
                          plan->typed_idx.as<int32_t>(), A->vals};
    if (check_mode()) {
      uint64_t fp = 0;
      if ((st = autosage_fingerprint(&Ap, &fp, stream)) != AUTOSAGE_OK) return st;
      if (fp != plan->a_fp) return fail(AUTOSAGE_ERR_PLAN_MISMATCH, "the structure arrays changed since the plan was built");
    }
    return run_op(plan, AUTOSAGE_OP_SPMM, &Ap, a, s);
  }
  autosage_plan_t P = nullptr;
  st = autosage_plan_typed(A, edge_type, num_types, F, dt, AUTOSAGE_PLAN_NO_CACHE, &P, stream);
  if (st == AUTOSAGE_OK) {
    const autosage_csr Ap{A->n_rows, (int64_t)num_types * A->n_cols, A->nnz, A->row_ptr,
                          P->typed_idx.as<int32_t>(), A->vals};
    st = run_op(P, AUTOSAGE_OP_SPMM, &Ap, a, s);
  }
  cudaError_t e = cudaStreamSynchronize(s);
  autosage_plan_destroy(P);
  if (st == AUTOSAGE_OK && e != cudaSuccess) return cuda_fail(e, "typed SpMM");
  return st;
}

// ---------------------------------------------------------------- utilities

autosage_status autosage_row_stats(const autosage_csr *A, int64_t long_threshold, int64_t *ints, double *reals,
                                   void *stream) {
  autosage_status st = check_csr(A, false);
  if (st != AUTOSAGE_OK) return st;
  if (!ints || !reals) return fail(AUTOSAGE_ERR_INVALID_ARG, "output arrays are NULL");
  RowStats rs;
  st = gpu_row_stats(A->n_rows, A->row_ptr, long_threshold, rs, as_stream(stream));
  if (st != AUTOSAGE_OK) return st;
  for (int i = 0; i < 40; ++i) ints[i] = rs.ints[i];
  reals[0] = rs.mean;
  reals[1] = rs.cv;
  return AUTOSAGE_OK;
}

autosage_status autosage_fingerprint(const autosage_csr *A, uint64_t *out, void *stream) {
  autosage_status st = check_csr(A, false);
  if (st != AUTOSAGE_OK) return st;
  if (!out) return fail(AUTOSAGE_ERR_INVALID_ARG, "out is NULL");
  cudaStream_t s = as_stream(stream);
  unsigned long long *d = nullptr, h = 0;
  CUDA_TRY(cudaMallocAsync(&d, sizeof h, s));
  cudaError_t e = launch_fingerprint(A->n_rows, A->nnz, A->row_ptr, A->col_idx, d, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof h, cudaMemcpyDeviceToHost, s);
  cudaFreeAsync(d, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "fingerprint");
  // the seed term mix(n_rows) is added on the host
  uint64_t z = (uint64_t)A->n_rows;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  z ^= z >> 31;
  *out = h + z;
  return AUTOSAGE_OK;
}

autosage_status autosage_validate_csr(const autosage_csr *A, void *stream) {
  if (!A || !A->row_ptr || A->n_rows < 0 || A->nnz < 0 || (A->nnz > 0 && !A->col_idx))
    return fail(AUTOSAGE_ERR_INVALID_ARG, "bad CSR descriptor");
  cudaStream_t s = as_stream(stream);
  int *d = nullptr, h = 0;
  CUDA_TRY(cudaMallocAsync(&d, sizeof h, s));
  cudaError_t e = launch_validate(A->n_rows, A->n_cols, A->nnz, A->row_ptr, A->col_idx, d, s);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, d, sizeof h, cudaMemcpyDeviceToHost, s);
  cudaFreeAsync(d, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "validate");
  if (h) return fail(AUTOSAGE_ERR_INVALID_CSR, "invalid CSR (flags 0x%x: 1 row_ptr[0]!=0, 2 decreasing row_ptr, "
                     "4 row_ptr[n]!=nnz, 8 col_idx out of range)", h);
  return AUTOSAGE_OK;
}

autosage_status autosage_measure_gather(int64_t table_bytes, int row_bytes, int64_t n_gathers, int reps,
                                        double *gbps, void *stream) {
  if (!gbps) return fail(AUTOSAGE_ERR_INVALID_ARG, "gbps is NULL");
  *gbps = 0;
  if (row_bytes < 16 || row_bytes > 4096 || row_bytes % 16)
    return fail(AUTOSAGE_ERR_INVALID_ARG, "row_bytes must be a multiple of 16 in [16, 4096]");
  if (table_bytes < row_bytes) return fail(AUTOSAGE_ERR_INVALID_ARG, "the table must hold at least one row");
  if (n_gathers < 1 || n_gathers >= INT32_MAX) return fail(AUTOSAGE_ERR_INVALID_ARG, "n_gathers out of range");
  if (reps < 1 || reps > 1000) return fail(AUTOSAGE_ERR_INVALID_ARG, "reps must be in [1, 1000]");
  const int64_t rows = table_bytes / row_bytes;
  if (rows >= INT32_MAX) return fail(AUTOSAGE_ERR_UNSUPPORTED, "more table rows than int32 indices address");
  cudaStream_t s = as_stream(stream);
  int dev = 0, sms = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int grid = sms * 4;  // four 256-thread blocks per SM: the fastest of 4 and 8 measured
  void *table = nullptr, *sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  float best = -1.f;
  cudaError_t e = cudaMallocAsync(&table, (size_t)(rows * row_bytes), s);
  if (e == cudaSuccess) e = cudaMallocAsync(&sink, sizeof(unsigned), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(table, 0x5a, (size_t)(rows * row_bytes), s);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  // one untimed run, then `reps` timed runs (each its own rows); the fastest is the rate
  if (e == cudaSuccess)
    e = launch_gather_rate(table, rows, n_gathers, row_bytes, grid, 0x5EEDull, static_cast<unsigned *>(sink), s);
  for (int r = 0; r < reps && e == cudaSuccess; ++r) {
    e = cudaEventRecord(e0, s);
    if (e == cudaSuccess)
      e = launch_gather_rate(table, rows, n_gathers, row_bytes, grid, 0x5EEDull + 0x1000ull * (r + 1),
                             static_cast<unsigned *>(sink), s);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    float ms = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e == cudaSuccess && ms > 0.f && (best < 0.f || ms < best)) best = ms;
  }
  if (table) cudaFreeAsync(table, s);
  if (sink) cudaFreeAsync(sink, s);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  const cudaError_t es = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = es;
  if (e != cudaSuccess) return cuda_fail(e, "gather rate");
  if (best <= 0.f) return fail(AUTOSAGE_ERR_CUDA, "gather rate: no timed run");
  *gbps = (double)n_gathers * row_bytes / (best * 1e-3) / 1e9;
  return AUTOSAGE_OK;
}

autosage_status autosage_csr_transpose(const autosage_csr *A, int32_t *row_ptr_t, int32_t *col_idx_t,
                                       float *vals_t, void *stream) {
  autosage_status st = check_csr(A, true);
  if (st != AUTOSAGE_OK) return st;
  if (!row_ptr_t || (A->nnz > 0 && !col_idx_t)) return fail(AUTOSAGE_ERR_INVALID_ARG, "output is NULL");
  cudaError_t e = csr_transpose(A->n_rows, A->n_cols, A->nnz, A->row_ptr, A->col_idx,
                                vals_t ? A->vals : nullptr, row_ptr_t, col_idx_t, vals_t, nullptr,
                                as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "transpose");
  return AUTOSAGE_OK;
}

// ---------------------------------------------------------------- cache I/O

autosage_status autosage_cache_clear(void) {
  std::lock_guard<std::mutex> lk(g_cache_mu);
  g_cache.clear();
  return AUTOSAGE_OK;
}

int64_t autosage_cache_size(void) {
  std::lock_guard<std::mutex> lk(g_cache_mu);
  return (int64_t)g_cache.size();
}

autosage_status autosage_cache_save(const char *path) {
  if (!path) return fail(AUTOSAGE_ERR_INVALID_ARG, "path is NULL");
  std::string tmp = std::string(path) + ".tmp";
  FILE *f = fopen(tmp.c_str(), "w");
  if (!f) return fail(AUTOSAGE_ERR_CACHE_IO, "cannot write %s", tmp.c_str());
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    fprintf(f, "%s\n", kCacheHeader);
    for (const auto &kv : g_cache) {
      fprintf(f, "%s\t%s %d %d %d %.6f%s", kv.first.c_str(), sched_name(kv.second.sched.kind),
              kv.second.sched.G, kv.second.sched.E, kv.second.sched.split, kv.second.probe_ms,
              kv.second.sched.pe ? " edge" : "");
      if (kv.second.sched.G2 > 0) fprintf(f, " agg=%d", kv.second.sched.G2);
      fputc('\n', f);
    }
  }
  const bool ok = fflush(f) == 0;
  fclose(f);
  if (!ok || rename(tmp.c_str(), path) != 0) return fail(AUTOSAGE_ERR_CACHE_IO, "cannot replace %s", path);
  return AUTOSAGE_OK;
}

autosage_status autosage_cache_load(const char *path) {
  if (!path) return fail(AUTOSAGE_ERR_INVALID_ARG, "path is NULL");
  std::ifstream in(path);
  if (!in) return fail(AUTOSAGE_ERR_CACHE_IO, "cannot read %s", path);
  std::string line;
  if (!std::getline(in, line) || line != kCacheHeader)
    return fail(AUTOSAGE_ERR_CACHE_FORMAT, "%s: missing or wrong header", path);
  int bad = 0, lineno = 1;
  std::map<std::string, CacheEntry> got;
  while (std::getline(in, line)) {
    ++lineno;
    if (line.empty() || line[0] == '#') continue;
    const size_t tab = line.find('\t');
    if (tab == std::string::npos || tab == 0) {
      ++bad;
      continue;
    }
    std::istringstream vs(line.substr(tab + 1));
    std::string kind;
    CacheEntry e;
    if (!(vs >> kind >> e.sched.G >> e.sched.E >> e.sched.split >> e.probe_ms)) {
      ++bad;
      continue;
    }
    // optional markers: per-edge SDDMM reductions ("edge"), the aggregation
    // stage's feature lanes of unfused attention ("agg=G")
    std::string tok;
    bool ok = true;
    while (ok && vs >> tok) {
      if (tok == "edge" && !e.sched.pe) {
        e.sched.pe = 1;
      } else if (tok.compare(0, 4, "agg=") == 0 && e.sched.G2 == 0) {
        char *end = nullptr;
        const long v = strtol(tok.c_str() + 4, &end, 10);
        ok = end && *end == 0 && v >= 1 && v <= 32 && is_pow2(v);
        e.sched.G2 = ok ? (int)v : 0;
      } else {
        ok = false;
      }
    }
    if (!ok) {
      ++bad;
      continue;
    }
    if (kind == "rowgroup") e.sched.kind = AUTOSAGE_SCHED_ROWGROUP;
    else if (kind == "split") e.sched.kind = AUTOSAGE_SCHED_SPLIT;
    else if (kind == "mergepath") e.sched.kind = AUTOSAGE_SCHED_MERGEPATH;
    else if (kind == "binned") e.sched.kind = AUTOSAGE_SCHED_BINNED;
    else if (kind == "hybrid") e.sched.kind = AUTOSAGE_SCHED_HYBRID;
    else {
      ++bad;
      continue;
    }
    const Sched &s = e.sched;
    const bool lanes_ok = (s.G == 0 || (is_pow2(s.G) && s.G <= 32)) && (s.E == 0 || (is_pow2(s.E) && s.E <= 32)) &&
                          std::max(1, s.G) * std::max(1, s.E) <= 32;
    const bool split_ok = s.kind == AUTOSAGE_SCHED_ROWGROUP ? s.split == 0 : s.split > 0;
    if (!lanes_ok || !split_ok) {
      ++bad;
      continue;
    }
    got[line.substr(0, tab)] = e;
  }
  {
    std::lock_guard<std::mutex> lk(g_cache_mu);
    for (auto &kv : got) g_cache[kv.first] = kv.second;
  }
  if (bad) return fail(AUTOSAGE_ERR_CACHE_FORMAT, "%s: %d bad line(s) skipped", path, bad);
  return AUTOSAGE_OK;
}

}  // extern "C"

namespace autosage {
// Record a status with a message for autosage_last_error().
autosage_status report(autosage_status st, const char *msg) { return fail(st, "%s", msg); }
}  // namespace autosage

// Unfused CSR attention with a caller-supplied fp32 score buffer of at least
// nnz * heads elements, default schedule, no plan, no device allocation.
// check_attention_args runs the same host-side checks as
// autosage_csr_attention (no GPU work, so no allocation: the structural
// validation of AUTOSAGE_CHECK is left out); attention_unfused_with_scores
// launches the three kernels on arguments that passed it.
namespace autosage {
autosage_status check_attention_args(const autosage_csr *A, const void *Q, const void *K, const void *V, int heads,
                                     int64_t D, autosage_dtype dt, const void *out) {
  autosage_status st = check_csr(A, false);
  if (st != AUTOSAGE_OK) return st;
  if (heads < 1 || D < 1) return fail(AUTOSAGE_ERR_INVALID_ARG, "heads and D must be >= 1");
  if (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16) return fail(AUTOSAGE_ERR_INVALID_ARG, "bad dtype");
  const int64_t W = (int64_t)heads * D;
  if ((st = check_mat(Q, W, W, A->n_rows, "Q")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(K, W, W, A->n_cols, "K")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(V, W, W, A->n_cols, "V")) != AUTOSAGE_OK) return st;
  if ((st = check_mat(out, W, W, A->n_rows, "out")) != AUTOSAGE_OK) return st;
  return AUTOSAGE_OK;
}

autosage_status attention_unfused_with_scores(const autosage_csr *A, const void *Q, const void *K,
                                              const void *V, int heads, int64_t D, autosage_dtype dt,
                                              float scale, void *out, float *scores, cudaStream_t s) {
  if (A->n_rows == 0) return AUTOSAGE_OK;
  OpArgs a;
  a.Q = Q; a.K = K; a.X = V; a.Y = out; a.alpha = scale; a.S = scores;
  autosage_plan_s P = transient(A, AUTOSAGE_OP_ATTN_UNFUSED, D, heads, dt);
  return run_op(&P, AUTOSAGE_OP_ATTN_UNFUSED, A, a, s);
}
}  // namespace autosage
