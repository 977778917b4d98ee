// Internal launcher interface between the host runtime and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace autosage {

enum class DType { F32 = 0, BF16 = 1 };

inline int dtype_size(DType t) { return t == DType::F32 ? 4 : 2; }

// Feature geometry of one launch: rows of F = H * D elements are read in
// fragments of VW elements (VW * size = vector bytes); nfrag = F / VW;
// cph = D / VW fragments per head; lanes G with NV fragments per lane.
struct Geom {
  DType dt;
  int H = 1;
  int64_t D = 0;
  int VW = 1;
  int nfrag = 0;
  int cph = 0;
  int G = 1;
  int E = 1;
  int NV = 1;
  int R = 1;       // lanes in one head reduction
  int es = 1;      // elements between consecutive edges in per-edge arrays (vals, scores)
  int fs = 1;      // fragment of slot k on lane g: g * fs + k * ks
  int ks = 1;
  bool one = true;       // all slots of a lane belong to one head
  bool batched = false;  // single-head SDDMM: transpose-reduction over G-edge batches
  bool comp = false;     // SpMM: compensated (Kahan) accumulation for long serial sums
};

// SpMM over rows (and chunks of cut rows) with per-edge (per-head) weights.
// vals: [nnz * H] or null. partial: [n_chunks * F] fp32 for chunk results.
cudaError_t launch_spmm(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                        const int32_t *col_idx, const float *vals, const void *X, int64_t ldx,
                        void *Y, int64_t ldy, const ChunkList &cl, float *partial,
                        cudaStream_t s);

// Two SpMMs over one CSR in one pass: Y1 = A_vals1 X1 and Y2 = A_vals2 X2
// (same geometry and leading dimensions); partial: [2 * n_chunks * F] fp32.
cudaError_t launch_spmm2(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                         const float *vals1, const float *vals2, const void *X1, const void *X2, int64_t ldx,
                         void *Y1, void *Y2, int64_t ldy, const ChunkList &cl, float *partial, cudaStream_t s);

// SDDMM: S[p*H + h] = alpha * <Q[row, h], K[col, h]>. Items come from the
// chunk list's deal, or (mp_part != null) from a merge path: lane group w
// takes diagonals [mp_part[w], mp_part[w + 1]) of the (rows + edges) path,
// n_groups groups.
cudaError_t launch_sddmm(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                         const int32_t *col_idx, const void *Q, int64_t ldq, const void *K,
                         int64_t ldk, float alpha, float *S, const ChunkList &cl, const int2 *mp_part,
                         int64_t n_groups, cudaStream_t s);

// Row softmax in place on S [nnz, H]. ml: [n_chunks * H * 2] fp32 workspace,
// row_ml: [n_long * H * 2] fp32 workspace (only with cut rows).
cudaError_t launch_row_softmax(int64_t n_rows, const int32_t *row_ptr, int H, float *S,
                               const ChunkList &cl, float *ml, float *row_ml, cudaStream_t s);

// Fused attention (scores from Q.K, or given scores when `scores` != null).
// part_acc: [n_chunks * F], part_ml: [n_chunks * H * 2] fp32 workspace.
cudaError_t launch_attention(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                             const int32_t *col_idx, const void *Q, const void *K,
                             const float *scores, const void *V, int64_t ld, float scale,
                             void *O, const ChunkList &cl, float *part_acc, float *part_ml,
                             cudaStream_t s);

// Merge-path SpMM: warp w covers diagonals [w*items, (w+1)*items) of the
// (rows + edges) merge path; part: [n_warps + 1] int2 (row, edge) starts.
// Shares of at most 256 items are staged in shared memory first.
// carry_val: [n_warps * F] fp32 (the row left unfinished at a warp's end),
// carry_row: [n_warps] int32, head_val: [n_warps * F] fp32 (the last segment
// of a row that earlier warps began, added and rounded by the fix-up).
cudaError_t launch_spmm_mergepath(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                                  const int32_t *col_idx, const float *vals, const void *X,
                                  int64_t ldx, void *Y, int64_t ldy, const int2 *part,
                                  int64_t n_warps, int items, float *carry_val, int32_t *carry_row,
                                  float *head_val, cudaStream_t s);
cudaError_t launch_mergepath_partition(int64_t n_rows, int64_t nnz, const int32_t *row_ptr,
                                       int64_t items, int64_t n_warps, int2 *part, cudaStream_t s);

// ---- graph utilities (graph.cu)
// stats: ints[40] (int64) and a double sum, device buffers.
cudaError_t launch_row_stats(int64_t n_rows, const int32_t *row_ptr, int64_t long_threshold,
                             unsigned long long *ints, cudaStream_t s);
cudaError_t launch_fingerprint(int64_t n_rows, int64_t nnz, const int32_t *row_ptr,
                               const int32_t *col_idx, unsigned long long *out, cudaStream_t s);
cudaError_t launch_validate(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *row_ptr,
                            const int32_t *col_idx, int *err, cudaStream_t s);
// Exclusive scan of n int32 values into out[n + 1] (out[n] = total). tmp: scan_tmp_bytes(n).
size_t scan_tmp_bytes(int64_t n);
cudaError_t launch_exclusive_scan(const int32_t *in, int32_t *out, int64_t n, void *tmp,
                                  cudaStream_t s);
// Long-row chunk lists for `split`: flags/scan over rows. Writes n_long and n_chunks
// to host (synchronises), allocating nothing; buffers sized by the caller from
// upper bounds (n_rows + 1 and nnz / split + n_rows + 1).
cudaError_t build_chunk_lists(int64_t n_rows, const int32_t *row_ptr, int split, int32_t *flags,
                              int32_t *scan_out, void *scan_tmp, int32_t *long_rows,
                              int32_t *long_ptr, int32_t *chunk_row, int32_t *chunk_begin,
                              int64_t *n_long_out, int64_t *n_chunks_out, cudaStream_t s);
// Stable transpose by LSD radix sort; temporaries from cudaMallocAsync on s.
// perm (optional, [nnz]): position k of A^T holds edge perm[k] of A.
cudaError_t csr_transpose(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *row_ptr,
                          const int32_t *col_idx, const float *vals, int32_t *row_ptr_t,
                          int32_t *col_idx_t, float *vals_t, int32_t *perm, cudaStream_t s);
// CSR-attention backward over the edges of A, one pass per row, for the g.H
// heads that Q, K, V, dO, dQ point at (row stride ld elements): dQ, and the
// softmax weights w and score gradients scale * dS written into the edge order
// of A^T (Wt, dSt: edge p's head h at p * es + h; inv[p] = position of edge
// p in A^T). S, dW: scratch with the same layout (scores and dW). part: per
// chunk 2 * H * D + 3 * H fp32 plus one int32; row_st: [n_long * H * 3] fp32
// (cut rows only).
cudaError_t launch_attention_backward(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                                      const int32_t *col_idx, const void *Q, const void *K, const void *V,
                                      const void *dO, int64_t ld, int es, float scale, void *dQ, float *S,
                                      float *dW, const int32_t *inv, float *Wt, float *dSt, const ChunkList &cl,
                                      float *part, float *row_st, cudaStream_t s);
// inv[perm[k]] = k for a permutation of n entries.
cudaError_t launch_invert_perm(int64_t n, const int32_t *perm, int32_t *inv, cudaStream_t s);
// Degree-binned row order: rows sorted (stably) by degree bucket, longest first,
// rows longer than `split` last. order: [n_rows]. Temporaries from cudaMallocAsync.
// bucket_start (host, optional, 33 entries): where rows of key k start in the
// order (key 0: the longest degree bucket; key 31: empty rows and rows longer
// than split); bucket_start[32] = n_rows. Synchronises s when given.
cudaError_t build_row_order(int64_t n_rows, const int32_t *row_ptr, int split, int32_t *order,
                            int32_t *bucket_start, cudaStream_t s);
// ELL slab (hybrid schedule) of the n rows at positions [pos0, pos0 + n) of a
// degree-binned order, each of degree <= W: col [W * n] column-major (-1
// pads), start [n] the first edge of each row.
cudaError_t build_ell(int64_t n, int W, const int32_t *order, int64_t pos0, const int32_t *row_ptr,
                      const int32_t *col_idx, int32_t *col, int32_t *start, cudaStream_t s);
// SpMM over an ELL slab (hybrid schedule): rows order[pos0 + e] for e < n,
// edge j of row e has column ell_col[j * n + e] (or -1) and value
// vals[ell_start[e] + j] (vals may be null: 1). Output rows of Y overwritten.
cudaError_t launch_spmm_ell(const Geom &g, int64_t n, const int32_t *rows, const int32_t *ell_col,
                            const int32_t *ell_start, const float *vals, const void *X, int64_t ldx, void *Y,
                            int64_t ldy, cudaStream_t s);
// out[k] = vals[perm[k]] for k < nnz (edge values carried into A^T's edge order).
cudaError_t launch_gather_vals(int64_t nnz, const int32_t *perm, const float *vals, float *out, cudaStream_t s);
// combined[p] = edge_type[p] * n_cols + col_idx[p]; *err (device) gets 1 for a type out of range.
cudaError_t launch_typed_index(int64_t nnz, int64_t n_cols, int n_types, const int32_t *col_idx,
                               const int32_t *edge_type, int32_t *combined, int *err, cudaStream_t s);
// Deterministic pseudo-random fill of probe buffers (values in [-1, 1)).
cudaError_t fill_probe(void *p, int64_t n_elems, DType dt, uint64_t seed, cudaStream_t s);
// Gather-rate measurement: n rows of `table` (rows rows of row_bytes, a
// multiple of 16 up to 4096) read by one warp each, row k chosen by a hash of
// (seed, k).
cudaError_t launch_gather_rate(const void *table, int64_t rows, int64_t n, int row_bytes, int grid,
                               uint64_t seed, unsigned *sink, cudaStream_t s);
// Count elements with |a - b| > atol + rtol * |b| (fp32 or bf16 arrays) into *count (device).
cudaError_t launch_compare(const void *a, const void *b, int64_t n, DType dt, float rtol,
                           float atol, unsigned long long *count, cudaStream_t s);

}  // namespace autosage
