/*
 * CPU oracle for CSR sparse aggregation: TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct loops in double precision. Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg may
 * load this library; the product path never calls it and shares no code
 * with it.
 *
 * What is computed follows AutoSAGE ("Input-Aware CUDA Scheduling for
 * Sparse GNN Aggregation (SpMM/SDDMM) and CSR Attention", Abstract): CSR
 * SpMM, SDDMM, and the CSR attention pipeline SDDMM -> row-softmax -> SpMM;
 * plus the benchmark page "fused sparse attention-value aggregation"
 * (problem statement and kernel discussion): rows are destinations,
 * col_idx holds sources, the softmax subtracts the row maximum, and a row
 * with no edges yields zeros.
 *
 * Precision: inputs are float32 (bfloat16 inputs are widened exactly by the
 * caller), every sum is accumulated in double, results are returned in
 * double; the caller rounds to the output type once.
 *
 * Row subsets: functions taking (rows, n_out) compute only the listed rows
 * (any order, repeats allowed) and write output row k for rows[k]. rows ==
 * NULL means every row, in order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ROW(k) (rows ? rows[(k)] : (int64_t)(k))

/* Y[i, h*D + d] = sum_{p in row i} vals[p*H + h] * X[col_idx[p], h*D + d].
 * H = 1 is plain SpMM Y = A X (Abstract: CSR SpMM); H > 1 aggregates each
 * head with its own per-edge weight (the SpMM half of multi-head CSR
 * attention). vals == NULL means every weight is 1. */
void oracle_spmm(int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                 const float *vals, int64_t H, int64_t D, const float *X, int64_t ldx,
                 const int64_t *rows, int64_t n_out, double *Y) {
  (void)n_rows;
  const int64_t F = H * D;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t k = 0; k < n_out; ++k) {
    const int64_t i = ROW(k);
    double *y = Y + k * F;
    for (int64_t f = 0; f < F; ++f) y[f] = 0.0;
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const float *x = X + (int64_t)col_idx[p] * ldx;
      for (int64_t h = 0; h < H; ++h) {
        const double w = vals ? (double)vals[p * H + h] : 1.0;
        for (int64_t d = 0; d < D; ++d) y[h * D + d] += w * (double)x[h * D + d];
      }
    }
  }
}

/* S[p*H + h] = alpha * sum_d Q[i, h*D + d] * K[col_idx[p], h*D + d] for every
 * edge p of row i (Abstract: SDDMM). Edge values are not multiplied in: the
 * output is the dense product Q K^T sampled on the sparsity pattern. For a
 * row subset the edges of rows[0], rows[1], ... are written one after the
 * other into S (the caller sizes S from the row degrees). */
void oracle_sddmm(int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                  int64_t H, int64_t D, const float *Q, int64_t ldq, const float *K,
                  int64_t ldk, double alpha, const int64_t *rows, int64_t n_out,
                  const int64_t *out_off, double *S) {
  (void)n_rows;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t k = 0; k < n_out; ++k) {
    const int64_t i = ROW(k);
    const int64_t base = rows ? out_off[k] : (int64_t)row_ptr[i];
    const float *q = Q + i * ldq;
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const float *kk = K + (int64_t)col_idx[p] * ldk;
      for (int64_t h = 0; h < H; ++h) {
        double s = 0.0;
        for (int64_t d = 0; d < D; ++d) s += (double)q[h * D + d] * (double)kk[h * D + d];
        S[(base + (p - row_ptr[i])) * H + h] = alpha * s;
      }
    }
  }
}

/* Row softmax of edge scores, per head: W[p,h] = exp(S[p,h] - m) / sum_q exp(S[q,h] - m)
 * with m the maximum of S[., h] over the row (benchmark page: the row maximum is
 * subtracted first, for numerical stability). Rows are given by row_ptr; S and W hold
 * nnz * H entries. A row with no edges has nothing to write. */
void oracle_row_softmax(int64_t n_rows, const int32_t *row_ptr, int64_t H,
                        const double *S, double *W) {
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t b = row_ptr[i], e = row_ptr[i + 1];
    if (e == b) continue;
    for (int64_t h = 0; h < H; ++h) {
      double m = -INFINITY;
      for (int64_t p = b; p < e; ++p)
        if (S[p * H + h] > m) m = S[p * H + h];
      double sum = 0.0;
      for (int64_t p = b; p < e; ++p) sum += exp(S[p * H + h] - m);
      for (int64_t p = b; p < e; ++p) W[p * H + h] = exp(S[p * H + h] - m) / sum;
    }
  }
}

/* CSR attention (Abstract: the pipeline SDDMM -> row-softmax -> SpMM), per head h:
 *   s_p = scale * <Q[i,h,:], K[col_idx[p],h,:]>,   w_p = softmax over the row,
 *   O[i,h,:] = sum_p w_p * V[col_idx[p],h,:].
 * Scores stay in double (never rounded to float). Empty rows give zeros.
 * Q, K, V, O are [n, H*D] with row strides ldq, ldk, ldv and H*D. */
void oracle_csr_attention(int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                          int64_t H, int64_t D, const float *Q, int64_t ldq, const float *K,
                          int64_t ldk, const float *V, int64_t ldv, double scale,
                          const int64_t *rows, int64_t n_out, double *O) {
  (void)n_rows;
  const int64_t F = H * D;
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t k = 0; k < n_out; ++k) {
    const int64_t i = ROW(k);
    const int64_t b = row_ptr[i], e = row_ptr[i + 1];
    double *o = O + k * F;
    for (int64_t f = 0; f < F; ++f) o[f] = 0.0;
    if (e == b) continue;
    double *s = (double *)malloc(sizeof(double) * (size_t)(e - b));
    const float *q = Q + i * ldq;
    for (int64_t h = 0; h < H; ++h) {
      double m = -INFINITY;
      for (int64_t p = b; p < e; ++p) {
        const float *kk = K + (int64_t)col_idx[p] * ldk;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += (double)q[h * D + d] * (double)kk[h * D + d];
        s[p - b] = scale * acc;
        if (s[p - b] > m) m = s[p - b];
      }
      double sum = 0.0;
      for (int64_t p = b; p < e; ++p) sum += exp(s[p - b] - m);
      for (int64_t p = b; p < e; ++p) {
        const double w = exp(s[p - b] - m) / sum;
        const float *v = V + (int64_t)col_idx[p] * ldv;
        for (int64_t d = 0; d < D; ++d) o[h * D + d] += w * (double)v[h * D + d];
      }
    }
    free(s);
  }
}

/* CSR of A^T by a stable counting sort: column j of A becomes row j of A^T,
 * and its entries keep the order of increasing original row (then original
 * edge position). Edge values move with their edges. Outputs: row_ptr_t
 * [n_cols + 1], col_idx_t [nnz] (original row ids), vals_t [nnz] (if vals). */
void oracle_transpose(int64_t n_rows, int64_t n_cols, const int32_t *row_ptr,
                      const int32_t *col_idx, const float *vals, int32_t *row_ptr_t,
                      int32_t *col_idx_t, float *vals_t) {
  const int64_t nnz = row_ptr[n_rows];
  int64_t *next = (int64_t *)calloc((size_t)n_cols + 1, sizeof(int64_t));
  for (int64_t p = 0; p < nnz; ++p) next[col_idx[p] + 1] += 1;
  for (int64_t j = 0; j < n_cols; ++j) next[j + 1] += next[j];
  for (int64_t j = 0; j <= n_cols; ++j) row_ptr_t[j] = (int32_t)next[j];
  for (int64_t i = 0; i < n_rows; ++i) {
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const int64_t dst = next[col_idx[p]]++;
      col_idx_t[dst] = (int32_t)i;
      if (vals && vals_t) vals_t[dst] = vals[p];
    }
  }
  free(next);
}

/* Second route to A^T X, used to cross-check the transpose: scatter every
 * edge's contribution straight into the output, in double.
 * GX[j, :] += vals[p] * G[i, :] for each edge p = (i -> j). GX is [n_cols, F]. */
void oracle_spmm_t_scatter(int64_t n_rows, int64_t n_cols, const int32_t *row_ptr,
                           const int32_t *col_idx, const float *vals, const float *G,
                           int64_t ldg, int64_t F, double *GX) {
  memset(GX, 0, sizeof(double) * (size_t)(n_cols * F));
  for (int64_t i = 0; i < n_rows; ++i) {
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const double w = vals ? (double)vals[p] : 1.0;
      double *gx = GX + (int64_t)col_idx[p] * F;
      const float *g = G + i * ldg;
      for (int64_t f = 0; f < F; ++f) gx[f] += w * (double)g[f];
    }
  }
}

/* Row-length statistics used by the schedule picker. Integer outputs:
 *   ints[0] n_rows, ints[1] nnz, ints[2] max degree, ints[3] min degree,
 *   ints[4] rows with no edges, ints[5] sum of squared degrees,
 *   ints[6] number of rows with degree > long_threshold,
 *   ints[7] edges in those rows,
 *   ints[8 + b] rows whose degree d has bucket b, where bucket 0 holds
 *   d == 0 and bucket b >= 1 holds 2^(b-1) <= d < 2^b (b up to 31).
 * Real outputs: reals[0] mean degree, reals[1] coefficient of variation. */
void oracle_row_stats(int64_t n_rows, const int32_t *row_ptr, int64_t long_threshold,
                      int64_t *ints, double *reals) {
  for (int k = 0; k < 8 + 32; ++k) ints[k] = 0;
  int64_t mx = 0, mn = n_rows > 0 ? INT64_MAX : 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t d = (int64_t)row_ptr[i + 1] - row_ptr[i];
    if (d > mx) mx = d;
    if (d < mn) mn = d;
    if (d == 0) ints[4] += 1;
    ints[5] += d * d;
    if (d > long_threshold) {
      ints[6] += 1;
      ints[7] += d;
    }
    int b = 0;
    while (b < 31 && d >= ((int64_t)1 << b)) ++b;
    ints[8 + b] += 1;
  }
  ints[0] = n_rows;
  ints[1] = n_rows > 0 ? row_ptr[n_rows] - row_ptr[0] : 0;
  ints[2] = mx;
  ints[3] = mn;
  const double mean = n_rows > 0 ? (double)ints[1] / (double)n_rows : 0.0;
  const double var = n_rows > 0 ? (double)ints[5] / (double)n_rows - mean * mean : 0.0;
  reals[0] = mean;
  reals[1] = mean > 0.0 ? sqrt(var > 0.0 ? var : 0.0) / mean : 0.0;
}

/* 64-bit fingerprint of a CSR structure, the key of the persistent plan
 * cache. Every element contributes mix(tag ^ (index << 32) ^ value) and the
 * contributions are added modulo 2^64, so the result does not depend on the
 * order of summation. mix is the SplitMix64 output function (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014). */
static uint64_t splitmix64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t oracle_fingerprint(int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx) {
  const uint64_t tag_rows = 0x9E3779B97F4A7C15ULL, tag_cols = 0xD1B54A32D192ED03ULL;
  uint64_t h = splitmix64_mix((uint64_t)n_rows);
  for (int64_t i = 0; i <= n_rows; ++i)
    h += splitmix64_mix(tag_rows ^ ((uint64_t)i << 32) ^ (uint32_t)row_ptr[i]);
  const int64_t nnz = row_ptr[n_rows];
  for (int64_t p = 0; p < nnz; ++p)
    h += splitmix64_mix(tag_cols ^ ((uint64_t)p << 32) ^ (uint32_t)col_idx[p]);
  return h;
}

/* Backward of CSR attention for a loss L with dL/dO = dO, per head h:
 *   w_p = softmax over row i of s_p = scale * <Q[i], K[j]>     (j = col_idx[p])
 *   dW_p = <dO[i], V[j]>,  D_i = sum_p w_p dW_p,  dS_p = w_p (dW_p - D_i)
 *   dQ[i] = scale * sum_p dS_p K[j],   dK[j] += scale * dS_p Q[i],   dV[j] += w_p dO[i]
 * (the chain rule through o_i = sum_p w_p v_j and the softmax). All in double.
 * Q, dO, dQ have n_rows rows; K, V, dK, dV have n_cols rows; width H*D. */
void oracle_csr_attention_backward(int64_t n_rows, int64_t n_cols, const int32_t *row_ptr,
                                   const int32_t *col_idx, int64_t H, int64_t D, const float *Q,
                                   const float *K, const float *V, const float *dO, double scale,
                                   double *dQ, double *dK, double *dV) {
  const int64_t F = H * D;
  memset(dQ, 0, sizeof(double) * (size_t)(n_rows * F));
  memset(dK, 0, sizeof(double) * (size_t)(n_cols * F));
  memset(dV, 0, sizeof(double) * (size_t)(n_cols * F));
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t b = row_ptr[i], e = row_ptr[i + 1];
    if (e == b) continue;
    double *w = (double *)malloc(sizeof(double) * (size_t)(e - b));
    double *dw = (double *)malloc(sizeof(double) * (size_t)(e - b));
    for (int64_t h = 0; h < H; ++h) {
      const float *q = Q + i * F + h * D;
      const float *go = dO + i * F + h * D;
      double m = -INFINITY;
      for (int64_t p = b; p < e; ++p) {
        const float *k = K + (int64_t)col_idx[p] * F + h * D;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += (double)q[d] * (double)k[d];
        w[p - b] = scale * acc;
        if (w[p - b] > m) m = w[p - b];
      }
      double sum = 0.0;
      for (int64_t p = b; p < e; ++p) sum += exp(w[p - b] - m);
      double Di = 0.0;
      for (int64_t p = b; p < e; ++p) {
        w[p - b] = exp(w[p - b] - m) / sum;
        const float *v = V + (int64_t)col_idx[p] * F + h * D;
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += (double)go[d] * (double)v[d];
        dw[p - b] = acc;
        Di += w[p - b] * acc;
      }
      for (int64_t p = b; p < e; ++p) {
        const int64_t j = col_idx[p];
        const double ds = w[p - b] * (dw[p - b] - Di);
        const float *k = K + j * F + h * D;
        for (int64_t d = 0; d < D; ++d) {
          dQ[i * F + h * D + d] += scale * ds * (double)k[d];
          dK[j * F + h * D + d] += scale * ds * (double)q[d];
          dV[j * F + h * D + d] += w[p - b] * (double)go[d];
        }
      }
    }
    free(w);
    free(dw);
  }
}

/* Multi-relation (typed) SpMM, the aggregation of an RGCN-style layer:
 * Y[i, :] = sum_p vals[p] * Z[edge_type[p], col_idx[p], :], with Z holding one
 * [n_cols, F] block per relation (block r starts at row r * n_cols). */
void oracle_spmm_typed(int64_t n_rows, int64_t n_cols, const int32_t *row_ptr, const int32_t *col_idx,
                       const int32_t *edge_type, const float *vals, const float *Z, int64_t ldz,
                       int64_t F, double *Y) {
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t i = 0; i < n_rows; ++i) {
    double *y = Y + i * F;
    for (int64_t f = 0; f < F; ++f) y[f] = 0.0;
    for (int64_t p = row_ptr[i]; p < row_ptr[i + 1]; ++p) {
      const double w = vals ? (double)vals[p] : 1.0;
      const float *z = Z + ((int64_t)edge_type[p] * n_cols + col_idx[p]) * ldz;
      for (int64_t f = 0; f < F; ++f) y[f] += w * (double)z[f];
    }
  }
}

/* Threads of the row-parallel loops (timing only: every row is computed by
 * one thread in a fixed order, so results do not depend on it). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
