/*
 * autosage.h -- C ABI of the GB300 (sm_103a) CSR sparse-aggregation library.
 *
 * Operations follow AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN
 * Aggregation (SpMM/SDDMM) and CSR Attention" (Abstract): CSR SpMM, SDDMM,
 * and the CSR attention pipeline SDDMM -> row-softmax -> SpMM, each run by
 * a schedule that an input-aware planner picks from a cost estimate, checks
 * with short timed runs on the device, and stores in a persistent cache so
 * that later runs reuse the same choice. The graph interface follows the
 * benchmark page
 * "fused sparse attention-value aggregation" (problem statement): rows are
 * destination nodes, row_ptr has n_rows + 1 int32 entries, col_idx holds
 * each edge's source node, an edgeless row produces zeros.
 *
 * Conventions shared by every entry point
 *  - Pointers named in an autosage_csr and every feature/output pointer are
 *    DEVICE pointers owned by the caller; the library never frees them.
 *  - Dense matrices are row-major with a leading dimension (elements) >= the
 *    row width. Attention tensors are [n, heads, D], contiguous.
 *  - Indices are int32; all offsets are formed in 64-bit inside kernels.
 *  - Outputs are overwritten, never accumulated into.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Every op is asynchronous on it, except where stated.
 *  - Argument errors are detected on the host before any launch and return
 *    a status; nothing is launched then. A failed launch returns
 *    AUTOSAGE_ERR_CUDA. autosage_last_error() gives a message for the
 *    calling thread's last failure.
 *  - The library allocates device memory only for plan workspace (owned by
 *    the plan, freed by autosage_plan_destroy) and, where stated, for
 *    stream-ordered temporaries released before the call's work completes.
 */
#ifndef AUTOSAGE_H
#define AUTOSAGE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  AUTOSAGE_OK = 0,
  AUTOSAGE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld < width, misalignment */
  AUTOSAGE_ERR_INVALID_CSR = 2,   /* row_ptr not monotone / col_idx out of range (checked modes) */
  AUTOSAGE_ERR_UNSUPPORTED = 3,   /* shape outside what a kernel handles (e.g. width too large) */
  AUTOSAGE_ERR_CUDA = 4,          /* a CUDA call or launch failed */
  AUTOSAGE_ERR_CACHE_IO = 5,      /* cache file cannot be opened / written */
  AUTOSAGE_ERR_CACHE_FORMAT = 6,  /* cache file has a bad header or bad lines (good lines still load) */
  AUTOSAGE_ERR_PROBE = 7,         /* every probed candidate failed; the default schedule is used */
  AUTOSAGE_ERR_PLAN_MISMATCH = 8  /* plan built for another graph, op, width or dtype */
} autosage_status;

typedef enum { AUTOSAGE_F32 = 0, AUTOSAGE_BF16 = 1 } autosage_dtype;

typedef enum {
  AUTOSAGE_OP_SPMM = 0,          /* Y = A X */
  AUTOSAGE_OP_SPMM_T = 1,        /* Y = A^T X (plan holds the transposed CSR) */
  AUTOSAGE_OP_SDDMM = 2,         /* S = alpha * (Q K^T) sampled on A's pattern */
  AUTOSAGE_OP_ATTN = 3,          /* fused CSR attention */
  AUTOSAGE_OP_ATTN_UNFUSED = 4,  /* SDDMM -> row softmax -> SpMM with scores in HBM */
  AUTOSAGE_OP_SOFTMAX = 5,       /* per-row softmax of edge scores */
  AUTOSAGE_OP_ATTN_BACKWARD = 6  /* gradients of CSR attention (plan holds A^T) */
} autosage_op;

/* Schedule families the planner chooses among (all are this library's own kernels). */
typedef enum {
  AUTOSAGE_SCHED_AUTO = -1,      /* let the planner decide */
  AUTOSAGE_SCHED_ROWGROUP = 0,   /* one lane group per row: G feature lanes x E edge lanes */
  AUTOSAGE_SCHED_SPLIT = 1,      /* rows longer than `split` edges are cut into chunks whose
                                    partial results are combined in a fixed order */
  AUTOSAGE_SCHED_MERGEPATH = 2,  /* equal (rows + edges) share per warp along the merge path,
                                    carry-out of rows cut at warp boundaries, fixed-order fix-up
                                    (SpMM); SDDMM: an equal share per lane group, no carries */
  AUTOSAGE_SCHED_BINNED = 3,     /* SPLIT, with rows taken in order of degree bucket (longest
                                    first) so the lane groups of a warp get rows of similar length */
  AUTOSAGE_SCHED_HYBRID = 4      /* SpMM only: BINNED for rows of 8 or more edges, and the rows of
                                    1..7 edges kept in an ELL slab (8 column slots per row,
                                    column-major) that one lane group per row reads with
                                    coalesced loads (composable formats: ELL + CSR) */
} autosage_sched_kind;

typedef struct {
  int kind;        /* autosage_sched_kind */
  int lanes_f;     /* G: lanes across the feature vector (power of two, 1..32); 0 = auto */
  int lanes_e;     /* E: lanes across edges of one row (power of two, G*E <= 32); 0 = auto */
  int split;       /* SPLIT/BINNED: chunk length in edges; MERGEPATH: items per warp; 0 = auto */
  int per_edge;    /* SDDMM with one head: 1 = finish each edge's dot product with its own
                      shuffle reduction; 0 = lane groups of 4 or more lanes reduce batches of
                      4 or 8 edges with one transpose-reduction. Other ops ignore it. */
  int lanes_f_agg; /* unfused attention: feature lanes of the aggregation stage (the SpMM
                      with the softmax weights; power of two, lanes_f_agg * lanes_e <= 32);
                      0 = lanes_f. The score stage uses lanes_f. Must be 0 for other ops. */
} autosage_schedule;

/* A CSR matrix in device memory. Rows are destinations, col_idx are sources.
 * vals may be NULL (every edge value is 1). nnz must equal row_ptr[n_rows]. */
typedef struct {
  int64_t n_rows;
  int64_t n_cols;
  int64_t nnz;
  const int32_t *row_ptr; /* [n_rows + 1] */
  const int32_t *col_idx; /* [nnz], each in [0, n_cols) */
  const float *vals;      /* [nnz] or NULL */
} autosage_csr;

typedef struct autosage_plan_s *autosage_plan_t;

/* Plan flags. */
#define AUTOSAGE_PLAN_PROBE 1u     /* refine the estimate with on-device micro-probes */
#define AUTOSAGE_PLAN_NO_CACHE 2u  /* neither read nor write the persistent cache */
#define AUTOSAGE_PLAN_VERIFY 4u    /* spot-check each probed candidate against the default */
/* The edge values given at plan time are fixed for the plan's life (a normalised adjacency
 * such as mean aggregation, 1/deg): every call must pass the same A->vals array (checked;
 * AUTOSAGE_ERR_PLAN_MISMATCH otherwise) and must not have changed its contents. SpMM with
 * A^T then gathers the values into A^T's edge order once, at plan time (and again in
 * autosage_plan_rebind), instead of at every call. Without this flag every call reads the
 * values it is passed. */
#define AUTOSAGE_PLAN_FIXED_VALUES 8u

/* ---------------------------------------------------------------- ops */

/* SpMM (Abstract: CSR SpMM). transpose == 0: Y[i,:] = sum_p vals[p] * X[col_idx[p],:]
 * for the n_rows rows of A; X has n_cols rows. transpose == 1: Y = A^T X, which needs a
 * plan built for AUTOSAGE_OP_SPMM_T (it holds A^T); Y has n_cols rows, X has n_rows rows.
 * dt is the type of X and Y (values, accumulation and softmax math are fp32).
 * plan may be NULL (transpose == 0 only): the default row-group schedule runs. */
autosage_status autosage_spmm(const autosage_csr *A, const void *X, int64_t ldx, void *Y,
                              int64_t ldy, int64_t F, autosage_dtype dt, int transpose,
                              autosage_plan_t plan, void *stream);

/* SDDMM (Abstract: SDDMM): out[p] = alpha * <Q[row(p),:], K[col_idx[p],:]> for every
 * edge p, written in CSR order as fp32 [nnz]. Edge values are not multiplied in.
 * Q has n_rows rows, K has n_cols rows, both of width F and type dt. */
autosage_status autosage_sddmm(const autosage_csr *A, const void *Q, int64_t ldq, const void *K,
                               int64_t ldk, int64_t F, autosage_dtype dt, float alpha,
                               float *out, autosage_plan_t plan, void *stream);

/* Row softmax of edge scores in place (Abstract: row-softmax; benchmark page: the row
 * maximum is subtracted first). scores is fp32 [nnz, heads]; each row and head is
 * normalised over the row's edges. */
autosage_status autosage_row_softmax(const autosage_csr *A, float *scores, int heads,
                                     autosage_plan_t plan, void *stream);

/* CSR attention (Abstract: the pipeline SDDMM -> row-softmax -> SpMM):
 * per head h, s_p = scale * <Q[i,h,:], K[col_idx[p],h,:]>, w = softmax over row i,
 * out[i,h,:] = sum_p w_p V[col_idx[p],h,:]. Q/K/V/out are [n, heads, D] of type dt.
 * fused != 0: one pass per row with an online softmax; scores never reach HBM.
 * fused == 0: SDDMM, softmax and SpMM kernels with an fp32 [nnz, heads] score array,
 * taken from the plan's workspace, or (plan == NULL) stream-ordered memory freed
 * on the same stream. Empty rows give zeros. A must be square-compatible: K and V
 * have n_cols rows, Q and out have n_rows rows. */
autosage_status autosage_csr_attention(const autosage_csr *A, const void *Q, const void *K,
                                       const void *V, int heads, int64_t D, autosage_dtype dt,
                                       float scale, void *out, int fused, autosage_plan_t plan,
                                       void *stream);

/* Multi-relation (typed) SpMM, the aggregation of an RGCN-style layer (SparseTIR's
 * RGCN workload): Y[i,:] = sum_p vals[p] * Z[edge_type[p] * n_cols + col_idx[p], :].
 * Z stacks one [n_cols, F] feature block per relation (typically X W_r computed by a
 * dense GEMM), row stride ldz, type dt. edge_type is a device int32 [nnz] array with
 * values in [0, num_types). The plan (autosage_plan_typed) checks the types on the GPU,
 * stores the combined gather index and picks an SpMM schedule for it; plan == NULL
 * builds a temporary plan inside the call (allocates and SYNCHRONISES `stream`).
 * num_types * n_cols must fit int32. */
autosage_status autosage_plan_typed(const autosage_csr *A, const int32_t *edge_type, int num_types,
                                    int64_t F, autosage_dtype dt, unsigned flags,
                                    autosage_plan_t *out, void *stream);
autosage_status autosage_spmm_typed(const autosage_csr *A, const int32_t *edge_type, int num_types,
                                    const void *Z, int64_t ldz, void *Y, int64_t ldy, int64_t F,
                                    autosage_dtype dt, autosage_plan_t plan, void *stream);

/* Backward of CSR attention (the chain rule through the composition SDDMM -> row-softmax
 * -> SpMM of the Abstract): for the upstream gradient dO [n_rows, heads, D], per head,
 *   w = softmax over row i of scale * <Q[i], K[j]>,  dW_p = <dO[i], V[j]>,
 *   dS_p = w_p (dW_p - sum_q w_q dW_q),
 *   dQ[i] = scale * sum_p dS_p K[j],  dK[j] = scale * sum_{p: col(p)=j} dS_p Q[i],
 *   dV[j] = sum_{p: col(p)=j} w_p dO[i].
 * One pass over the rows of A recomputes the scores, keeps an online softmax state and
 * produces dW, the row sums and dQ (each K and V row gathered once per edge); it writes
 * w and scale * dS into the edge order of A^T, where two SpMMs give dV and dK.
 * heads * D may be at most 256 fragments of 16 bytes (fp32 1024, bf16 2048) when aligned.
 * Q, dO, dQ have n_rows rows; K, V, dK, dV have n_cols rows; all [., heads, D] of type dt,
 * contiguous. plan: built for AUTOSAGE_OP_ATTN_BACKWARD with F = D (it holds A^T, the
 * permutation and the edge buffers); NULL builds a temporary plan inside the call, which
 * allocates device memory and SYNCHRONISES `stream`. */
autosage_status autosage_csr_attention_backward(const autosage_csr *A, const void *Q, const void *K,
                                                const void *V, const void *dO, int heads, int64_t D,
                                                autosage_dtype dt, float scale, void *dQ, void *dK,
                                                void *dV, autosage_plan_t plan, void *stream);

/* The benchmark page's op (fused softmax + aggregation with given scores): per head,
 * w = softmax over row i of scores[p, h]; out[i,h,:] = sum_p w_p V[col_idx[p],h,:].
 * scores is fp32 [nnz, heads]; V and out are [n, heads, D] of type dt. */
autosage_status autosage_edge_softmax_aggregate(const autosage_csr *A, const float *scores,
                                                const void *V, int heads, int64_t D,
                                                autosage_dtype dt, void *out,
                                                autosage_plan_t plan, void *stream);

/* Unfused CSR attention that allocates no device memory. This entry point has no
 * counterpart in the paper; it is for callers that must not allocate inside their
 * work loop (a serving process that reserved all device memory for its own pool,
 * or a latency-critical loop where a driver allocation could synchronise the
 * device). It computes what autosage_csr_attention(fused = 0, plan = NULL)
 * computes, with the same kernels, but keeps the fp32 score array in a fixed
 * device array owned by the library: AUTOSAGE_NOALLOC_MAX_SCORES fp32 elements
 * (16 MiB), held on every GPU the library is loaded on until the process exits.
 *  - nnz * heads above AUTOSAGE_NOALLOC_MAX_SCORES returns AUTOSAGE_ERR_UNSUPPORTED
 *    before any launch; no cudaMalloc / cudaFree or allocating routine is called.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture. The address is kept for the life of the process: after
 *    cudaDeviceReset (or in another primary context of that device) it is stale,
 *    so do not call this entry point again after resetting the device.
 *  - The CSR descriptor gets the same host-side checks as autosage_csr_attention
 *    (sizes, NULL pointers, 4-byte alignment); the GPU structural validation of
 *    AUTOSAGE_CHECK=1 is not run here, because it allocates.
 *  - Every call on a device shares the one array and leaves its scores there.
 *    Calls whose work overlaps on the GPU (other streams, other threads) race on
 *    it: serialise them. Nothing in the array needs to start at zero.
 * Arguments as autosage_csr_attention (Q/K/V/out [n, heads, D] of type dt). */
#define AUTOSAGE_NOALLOC_MAX_SCORES (4u * 1024u * 1024u)
autosage_status autosage_csr_attention_unfused_noalloc(const autosage_csr *A, const void *Q,
                                                       const void *K, const void *V, int heads,
                                                       int64_t D, autosage_dtype dt, float scale,
                                                       void *out, void *stream);

/* ---------------------------------------------------------------- row sharding (several GPUs)
 *
 * Every op is defined per destination row (Abstract; benchmark page, problem statement: an
 * output row per destination node from its incoming edges), so contiguous row ranges are
 * independent units. A multi-GPU job gives each process (one per GPU) a shard: a range of rows
 * with about equal edge counts. The shard needs the feature rows its edges reference (its
 * halo), which one exchange step brings to its GPU (e.g. an all-gather of the row blocks the
 * processes own, then autosage_gather_rows); its outputs are its own rows, so nothing is
 * reduced afterwards. SpMM with A^T shards the rows of A^T. The partition and halo are
 * computed on the host once per graph; the ops themselves run unchanged on the shard's CSR. */

/* Cut the n_rows rows of a CSR into `parts` contiguous ranges of about equal nnz. row_ptr is
 * a HOST array [n_rows + 1]; bounds is a HOST array [parts + 1] that receives the first row of
 * each part (bounds[0] = 0, bounds[parts] = n_rows; part k is rows [bounds[k], bounds[k+1]),
 * possibly empty). Returns AUTOSAGE_ERR_INVALID_CSR if row_ptr[0] != 0 or row_ptr decreases. */
autosage_status autosage_partition_rows(const int32_t *row_ptr, int64_t n_rows, int parts, int64_t *bounds);

/* Halo of the shard of rows [row_begin, row_end) of a HOST CSR (row_ptr, col_idx): the distinct
 * columns its edges reference, in increasing order, written to halo (HOST, capacity n_cols;
 * their count to *n_halo), and for each edge p of the shard (p - row_ptr[row_begin] in
 * [0, shard nnz)) the position of its column in halo, written to local_col (HOST). The shard's
 * CSR with row_ptr[row_begin..row_end] - row_ptr[row_begin], local_col and n_cols = *n_halo
 * then addresses a dense matrix of the halo rows only. Columns outside [0, n_cols) return
 * AUTOSAGE_ERR_INVALID_CSR. */
autosage_status autosage_shard_halo(const int32_t *row_ptr, const int32_t *col_idx, int64_t n_cols,
                                    int64_t row_begin, int64_t row_end, int32_t *halo, int64_t *n_halo,
                                    int32_t *local_col);

/* out[k, :] = X[idx[k], :] for k < n on the GPU (DEVICE pointers; rows of F elements of type
 * dt, leading dimensions ldx and ldo in elements; each idx[k] must be a row of X). Packs a
 * shard's halo rows into a dense matrix. Asynchronous on `stream`. */
autosage_status autosage_gather_rows(const void *X, int64_t ldx, const int32_t *idx, int64_t n, int64_t F,
                                     autosage_dtype dt, void *out, int64_t ldo, void *stream);

/* ---------------------------------------------------------------- planning */

/* Build a plan for (A, op, F, heads, dt). For attention ops F is the head dimension D.
 * Computes row statistics and a structure fingerprint on the GPU, looks the key up in
 * the process-wide cache (unless AUTOSAGE_PLAN_NO_CACHE); on a miss scores candidate
 * schedules with the cost estimate, and with AUTOSAGE_PLAN_PROBE times the best few on
 * the device (on scratch buffers, never on caller data), keeps the fastest, and records
 * it in the cache. Workspace (chunk lists, partial buffers, A^T) is allocated and built.
 * SYNCHRONISES `stream`. Returns AUTOSAGE_ERR_PROBE (with a usable default plan in
 * *out) if every probe failed. */
autosage_status autosage_plan(const autosage_csr *A, autosage_op op, int64_t F, int heads,
                              autosage_dtype dt, unsigned flags, autosage_plan_t *out,
                              void *stream);

/* Build a plan with an explicit schedule (no cache, no probes). SYNCHRONISES `stream`. */
autosage_status autosage_plan_with_schedule(const autosage_csr *A, autosage_op op, int64_t F,
                                            int heads, autosage_dtype dt,
                                            const autosage_schedule *sched,
                                            autosage_plan_t *out, void *stream);

/* A plan is bound to the structure of the A it was built for: its workspace (chunk lists,
 * row order, merge-path partitions, A^T and the edge permutation) is derived from row_ptr
 * and col_idx. Every op called with a plan therefore requires A->row_ptr and A->col_idx to
 * be the very arrays given at plan time (same pointers, contents unchanged) and returns
 * AUTOSAGE_ERR_PLAN_MISMATCH before any launch otherwise; with the environment variable
 * AUTOSAGE_CHECK=1 it also recomputes the structure fingerprint (synchronising) and
 * refuses arrays that were overwritten with another graph. The edge values are NOT part
 * of the binding: every call reads A->vals as passed (for SpMM with A^T they are gathered
 * into A^T's edge order on the stream at each call), so new values per layer or step need
 * no new plan, unless the plan was built with AUTOSAGE_PLAN_FIXED_VALUES (see there).
 * A typed plan is bound to row_ptr, col_idx and edge_type.
 * A plan's workspace is shared by its calls: calls of one plan that overlap on the GPU
 * (several streams or threads) race on it; serialise them or use one plan per stream. */

/* Rebind a plan to structure arrays that moved (a copy of the same graph in new device
 * memory). Computes the fingerprint of A's structure on the GPU (SYNCHRONISES `stream`)
 * and accepts A only if its sizes and fingerprint equal those of the plan's graph;
 * otherwise returns AUTOSAGE_ERR_PLAN_MISMATCH and leaves the plan unchanged. A plan with
 * fixed values takes A->vals as its new fixed values. Typed plans
 * return AUTOSAGE_ERR_UNSUPPORTED (their combined index is built from the edge types). */
autosage_status autosage_plan_rebind(autosage_plan_t plan, const autosage_csr *A, void *stream);

/* Free a plan and its workspace (synchronises the device). NULL is allowed. */
autosage_status autosage_plan_destroy(autosage_plan_t plan);

/* Write a one-line description of the plan's schedule into buf (always NUL-terminated). */
autosage_status autosage_plan_describe(autosage_plan_t plan, char *buf, size_t len);

/* The schedule a plan runs (kind, lanes, split) and its probe time in ms (or -1). */
autosage_status autosage_plan_schedule(autosage_plan_t plan, autosage_schedule *sched,
                                       double *probe_ms);

/* ---------------------------------------------------------------- persistent cache */

/* Merge entries from a cache file into the process-wide cache. Lines that do not parse
 * are skipped and reported with AUTOSAGE_ERR_CACHE_FORMAT; good lines still load. */
autosage_status autosage_cache_load(const char *path);
/* Write the process-wide cache (entries sorted by key) to path, atomically replaced. */
autosage_status autosage_cache_save(const char *path);
/* Drop every cached entry. */
autosage_status autosage_cache_clear(void);
/* Number of cached entries. */
int64_t autosage_cache_size(void);

/* ---------------------------------------------------------------- graph utilities */

/* Row statistics of A computed on the GPU (planner input). ints[40] and reals[2] are
 * HOST arrays: ints = {n_rows, nnz, max deg, min deg, empty rows, sum deg^2,
 * rows with deg > long_threshold, edges in them, 32 log2 buckets (bucket 0: deg 0,
 * bucket b: 2^(b-1) <= deg < 2^b)}, reals = {mean degree, coefficient of variation}.
 * SYNCHRONISES `stream`. */
autosage_status autosage_row_stats(const autosage_csr *A, int64_t long_threshold, int64_t *ints,
                                   double *reals, void *stream);

/* 64-bit fingerprint of A's structure (order-independent sum of SplitMix64-mixed
 * (index, value) words of row_ptr and col_idx); *out is a HOST pointer. SYNCHRONISES. */
autosage_status autosage_fingerprint(const autosage_csr *A, uint64_t *out, void *stream);

/* Full structural check of A on the GPU: row_ptr[0] == 0, non-decreasing,
 * row_ptr[n_rows] == nnz, every col_idx in [0, n_cols). Returns AUTOSAGE_OK or
 * AUTOSAGE_ERR_INVALID_CSR. SYNCHRONISES `stream`. */
autosage_status autosage_validate_csr(const autosage_csr *A, void *stream);

/* CSR of A^T by a stable counting sort on the GPU: row_ptr_t [n_cols + 1],
 * col_idx_t [nnz] (original rows, increasing inside each new row), vals_t [nnz]
 * (may be NULL; ignored if A->vals is NULL). Device outputs owned by the caller.
 * Uses stream-ordered temporaries. */
autosage_status autosage_csr_transpose(const autosage_csr *A, int32_t *row_ptr_t,
                                       int32_t *col_idx_t, float *vals_t, void *stream);

/* ---------------------------------------------------------------- measurement */

/* Read rate of random row gathers on this GPU: the ceiling a gather kernel meets when its
 * rows come from a table of table_bytes. A table that fits in L2 gives the rate at which L2
 * serves repeatedly gathered (hot) rows; one far larger than L2 gives the DRAM rate. One warp
 * per gathered row reads row_bytes (a multiple of 16 in [16, 4096]) in 16-byte words, all of
 * a lane's words in flight together; each run reads n_gathers rows of the table, row k chosen
 * by a SplitMix64 hash of (run, k) computed in the kernel (no index array is read). *gbps
 * (HOST) receives n_gathers * row_bytes / the fastest of `reps` timed runs (after one untimed
 * run), in GB/s. Allocates (stream-ordered) a table of table_bytes rounded down to whole rows,
 * and frees it before returning. SYNCHRONISES `stream`. Argument errors return
 * AUTOSAGE_ERR_INVALID_ARG before any device call. */
autosage_status autosage_measure_gather(int64_t table_bytes, int row_bytes, int64_t n_gathers, int reps,
                                        double *gbps, void *stream);

/* ---------------------------------------------------------------- misc */

const char *autosage_status_string(autosage_status s);
/* Message of the calling thread's last failed call ("" if none). */
const char *autosage_last_error(void);
/* Library version string. */
const char *autosage_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AUTOSAGE_H */
