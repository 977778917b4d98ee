// CSR SpMM kernels: Y = A X (AutoSAGE, "Input-Aware CUDA Scheduling for
// Sparse GNN Aggregation (SpMM/SDDMM) and CSR Attention", Abstract: CSR
// SpMM), with per-head edge weights for the aggregation step of CSR
// attention (Abstract: the pipeline SDDMM -> row-softmax -> SpMM).
//
// The work is a gather: every edge reads one source row of X. Kernels are
// HBM-bound; they use no tensor cores. Three schedules:
//  * row groups: G feature lanes x E edge lanes per row (rows of degree
//    <= split), E partial sums combined by shuffles in a fixed order;
//  * split: rows longer than `split` edges are cut into chunks that write
//    fp32 partials; a fix-up adds each row's chunks in chunk order;
//  * merge path: each warp takes an equal share of (rows + edges); rows cut
//    at warp boundaries leave carry-outs that a fix-up adds in warp order.
// No floating-point atomics anywhere: repeat runs give identical bits.
#include "internal.h"

namespace autosage {

namespace {

template <int NV, int VW>
__device__ __forceinline__ void zero(float (&acc)[NV][VW]) {
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[k][v] = 0.f;
}

// acc += w * x, plain or compensated (Kahan): long rows of signed terms can
// cancel to a small result whose fp32 rounding error, accumulated over tens of
// thousands of additions, would otherwise approach the result itself.
template <bool COMP>
__device__ __forceinline__ void accum(float &acc, float &comp, float w, float x) {
  if constexpr (COMP) {
    const float y = fmaf(w, x, -comp);
    const float t = acc + y;
    comp = (t - acc) - y;
    acc = t;
  } else {
    acc = fmaf(w, x, acc);
  }
}

// Column indices and edge weights of the U edges p, p + E, ... (those below
// pe; the others get column 0 and are never used) for every fragment slot.
// Slots share one weight when there is one head or every slot of the lane
// lies in the same head (`one`); otherwise each slot loads its head's weight.
template <int U, int NV>
__device__ __forceinline__ void load_weights(const int32_t *__restrict__ col_idx,
                                             const float *__restrict__ vals, int H, int es, bool one,
                                             const int (&head)[NV], int p, int E, int pe, int (&c)[U],
                                             float (&w)[U][NV]) {
#pragma unroll
  for (int u = 0; u < U; ++u) c[u] = p + u * E < pe ? ld_stream_i32(col_idx + p + u * E) : 0;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int q = p + u * E;
    if (vals == nullptr || q >= pe) {
#pragma unroll
      for (int k = 0; k < NV; ++k) w[u][k] = 1.f;
    } else if (H == 1 || one) {
      const float x = H == 1 ? ld_stream_f32(vals + (int64_t)q * es) : __ldg(vals + (int64_t)q * es + head[0]);
#pragma unroll
      for (int k = 0; k < NV; ++k) w[u][k] = x;
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k) w[u][k] = __ldg(vals + (int64_t)q * es + head[k]);
    }
  }
}

// Accumulate edges p = p0, p0 + E, ... < pe into acc (per lane fragments).
// Each round takes U edges per edge lane, predicated at the row's end (a
// short row is one round with all its loads in flight); the next round's
// column indices and weights are loaded while this round's rows are in
// flight, so a round waits on one memory round trip, not two.
template <typename T, int VW, int NV, int U, bool COMP>
__device__ __forceinline__ void gather_edges(const int32_t *__restrict__ col_idx,
                                             const float *__restrict__ vals, int H, int es, bool one,
                                             const int (&head)[NV], const T *__restrict__ X,
                                             int64_t ldx, int nfrag, const int (&frag)[NV], int E, int p0,
                                             int pe, float (&acc)[NV][VW], float (&comp)[NV][VW]) {
  if (p0 >= pe) return;
  int c[U];
  float w[U][NV];
  load_weights<U, NV>(col_idx, vals, H, es, one, head, p0, E, pe, c, w);
  for (int p = p0; p < pe; p += U * E) {
    Frag<T, VW> f[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (p + u * E < pe && frag[k] < nfrag) f[u][k].load(X + (int64_t)c[u] * ldx + (int64_t)frag[k] * VW);
    const int pn = p + U * E;
    int cn[U];
    float wn[U][NV];
    if (pn < pe) load_weights<U, NV>(col_idx, vals, H, es, one, head, pn, E, pe, cn, wn);
    // rows of edges past the end were never loaded: skip them (0 * garbage may be NaN)
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (p + u * E < pe)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (frag[k] < nfrag)
#pragma unroll
            for (int v = 0; v < VW; ++v) accum<COMP>(acc[k][v], comp[k][v], w[u][k], f[u][k].get(v));
#pragma unroll
    for (int u = 0; u < U; ++u) {
      c[u] = cn[u];
#pragma unroll
      for (int k = 0; k < NV; ++k) w[u][k] = wn[u][k];
    }
  }
}

// Two products over the same edges in one walk: acc1 += w1 * X1[col] and
// acc2 += w2 * X2[col] (per-head weights vals1, vals2 with the same layout).
// Each edge's column is loaded once and both rows are in flight together;
// each sum takes its edges in the order gather_edges would, so both outputs
// have the bits of two separate SpMMs.
template <typename T, int VW, int NV, int U, bool COMP>
__device__ __forceinline__ void gather_edges2(const int32_t *__restrict__ col_idx, const float *__restrict__ vals1,
                                              const float *__restrict__ vals2, int H, int es, bool one,
                                              const int (&head)[NV], const T *__restrict__ X1,
                                              const T *__restrict__ X2, int64_t ldx, int nfrag,
                                              const int (&frag)[NV], int E, int p0, int pe,
                                              float (&acc1)[NV][VW], float (&comp1)[NV][VW],
                                              float (&acc2)[NV][VW], float (&comp2)[NV][VW]) {
  if (p0 >= pe) return;
  int c[U];
  float w1[U][NV], w2[U][NV];
  load_weights<U, NV>(col_idx, vals1, H, es, one, head, p0, E, pe, c, w1);
  load_weights<U, NV>(col_idx, vals2, H, es, one, head, p0, E, pe, c, w2);
  for (int p = p0; p < pe; p += U * E) {
    Frag<T, VW> f1[U][NV], f2[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (p + u * E < pe && frag[k] < nfrag) {
          f1[u][k].load(X1 + (int64_t)c[u] * ldx + (int64_t)frag[k] * VW);
          f2[u][k].load(X2 + (int64_t)c[u] * ldx + (int64_t)frag[k] * VW);
        }
    const int pn = p + U * E;
    int cn[U];
    float wn1[U][NV], wn2[U][NV];
    if (pn < pe) {
      load_weights<U, NV>(col_idx, vals1, H, es, one, head, pn, E, pe, cn, wn1);
      load_weights<U, NV>(col_idx, vals2, H, es, one, head, pn, E, pe, cn, wn2);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (p + u * E < pe)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (frag[k] < nfrag)
#pragma unroll
            for (int v = 0; v < VW; ++v) {
              accum<COMP>(acc1[k][v], comp1[k][v], w1[u][k], f1[u][k].get(v));
              accum<COMP>(acc2[k][v], comp2[k][v], w2[u][k], f2[u][k].get(v));
            }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      c[u] = cn[u];
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        w1[u][k] = wn1[u][k];
        w2[u][k] = wn2[u][k];
      }
    }
  }
}

// gather_edges over column indices and weights staged in shared memory (sc,
// sv: entries for the edges from `base` on; sv null: weight 1): the same
// rounds and the same order of additions, with the index and weight loads
// served from shared memory instead of global memory.
template <typename T, int VW, int NV, int U, bool COMP>
__device__ __forceinline__ void gather_staged(const int32_t *sc, const float *sv, int base, const T *__restrict__ X,
                                              int64_t ldx, int nfrag, const int (&frag)[NV], int E, int p0, int pe,
                                              float (&acc)[NV][VW], float (&comp)[NV][VW]) {
  for (int p = p0; p < pe; p += U * E) {
    int c[U];
    float w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = p + u * E;
      c[u] = q < pe ? sc[q - base] : 0;
      w[u] = (q < pe && sv) ? sv[q - base] : 1.f;
    }
    Frag<T, VW> f[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (p + u * E < pe && frag[k] < nfrag) f[u][k].load(X + (int64_t)c[u] * ldx + (int64_t)frag[k] * VW);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (p + u * E < pe)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (frag[k] < nfrag)
#pragma unroll
            for (int v = 0; v < VW; ++v) accum<COMP>(acc[k][v], comp[k][v], w[u], f[u][k].get(v));
  }
}

// Sum the E edge-lane partials of a group (xor butterfly, fixed order).
template <int NV, int VW>
__device__ __forceinline__ void reduce_edge_lanes(float (&acc)[NV][VW], unsigned mask, int G, int GE) {
  for (int off = G; off < GE; off <<= 1) {
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int v = 0; v < VW; ++v) acc[k][v] += __shfl_xor_sync(mask, acc[k][v], off);
  }
}

template <int NV, int VW> constexpr int unroll_for() {
  return NV * VW <= 8 ? 4 : (NV * VW <= 16 ? 2 : 1);
}

template <typename T, int VW, int NV, bool COMP>
__global__ void __launch_bounds__(kBlock) spmm_rows_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const float *__restrict__ vals, int H, int es, int cph, const T *__restrict__ X, int64_t ldx,
    T *__restrict__ Y, int64_t ldy, int nfrag, int G, int E, int fs, int ks, bool one, ChunkList cl,
    int ipb, float *__restrict__ partial) {
  const Lanes L(G, E);
  int frag[NV], head[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    frag[k] = L.g * fs + k * ks;
    head[k] = (H > 1 && frag[k] < nfrag) ? frag[k] / cph : 0;
  }
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
    const Item it = item_at(idx, n_rows, row_ptr, cl);
    float acc[NV][VW], comp[NV][VW];
    zero(acc);
    zero(comp);
    gather_edges<T, VW, NV, unroll_for<NV, VW>(), COMP>(col_idx, vals, H, es, one, head, X, ldx, nfrag, frag,
                                                         E, it.b + L.e, it.e, acc, comp);
    reduce_edge_lanes(acc, L.group_mask, G, L.GE);
    if (!it.active || L.e != 0) continue;
    if (it.chunk < 0) {
      T *y = Y + it.row * ldy;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (frag[k] < nfrag) store_frag<T, VW>(y + (int64_t)frag[k] * VW, acc[k]);
    } else {
      float *y = partial + (int64_t)it.chunk * nfrag * VW;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (frag[k] < nfrag) store_partial<VW>(y + (int64_t)frag[k] * VW, acc[k]);
    }
  }
}

// Two SpMMs over one CSR in one pass (Y1 = A_w1 X1, Y2 = A_w2 X2; the edge
// weights differ, the structure is shared): the attention backward's dV and
// dK over the rows of A^T. Cut rows write both partials (partial and
// partial + n_chunks * F).
// Blocks per SM the two-product kernel is sized for: three 256-thread blocks
// (80 registers) where a lane holds few values, with one edge per round for
// both products (measured on the attention backward, R-MAT scale 20, bf16,
// H = 8, D = 64: 11.64 ms against 11.73 ms for two edges per round at two
// blocks, and 11.99 ms for two separate SpMMs).
// Narrower fragments and compensated sums spilled at that bound, so they keep
// the registers they need.
template <typename T, int VW, int NV, bool COMP>
constexpr int spmm2_min_blocks() {
  return (!COMP && VW * sizeof(T) == 16 && (NV * VW <= 4 || (sizeof(T) == 2 && NV * VW <= 16))) ? 3 : 1;
}

template <typename T, int VW, int NV, bool COMP>
__global__ void __launch_bounds__(kBlock, spmm2_min_blocks<T, VW, NV, COMP>()) spmm2_rows_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const float *__restrict__ vals1, const float *__restrict__ vals2, int H, int es, int cph,
    const T *__restrict__ X1, const T *__restrict__ X2, int64_t ldx, T *__restrict__ Y1, T *__restrict__ Y2,
    int64_t ldy, int nfrag, int G, int E, int fs, int ks, bool one, ChunkList cl, int ipb,
    float *__restrict__ partial) {
  const Lanes L(G, E);
  int frag[NV], head[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    frag[k] = L.g * fs + k * ks;
    head[k] = (H > 1 && frag[k] < nfrag) ? frag[k] / cph : 0;
  }
  const int64_t F = (int64_t)nfrag * VW;
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
    const Item it = item_at(idx, n_rows, row_ptr, cl);
    float acc1[NV][VW], comp1[NV][VW], acc2[NV][VW], comp2[NV][VW];
    zero(acc1);
    zero(comp1);
    zero(acc2);
    zero(comp2);
    gather_edges2<T, VW, NV, (unroll_for<NV, VW>() > 1 ? unroll_for<NV, VW>() / 2 : 1), COMP>(col_idx, vals1, vals2, H, es, one, head, X1, X2, ldx,
                                                          nfrag, frag, E, it.b + L.e, it.e, acc1, comp1, acc2,
                                                          comp2);
    reduce_edge_lanes(acc1, L.group_mask, G, L.GE);
    reduce_edge_lanes(acc2, L.group_mask, G, L.GE);
    if (!it.active || L.e != 0) continue;
    if (it.chunk < 0) {
      T *y1 = Y1 + it.row * ldy, *y2 = Y2 + it.row * ldy;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (frag[k] < nfrag) {
          store_frag<T, VW>(y1 + (int64_t)frag[k] * VW, acc1[k]);
          store_frag<T, VW>(y2 + (int64_t)frag[k] * VW, acc2[k]);
        }
    } else {
      float *p1 = partial + (int64_t)it.chunk * F, *p2 = partial + ((int64_t)cl.n_chunks + it.chunk) * F;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (frag[k] < nfrag) {
          store_partial<VW>(p1 + (int64_t)frag[k] * VW, acc1[k]);
          store_partial<VW>(p2 + (int64_t)frag[k] * VW, acc2[k]);
        }
    }
  }
}

// One warp per cut row: add its chunk partials in chunk order.
template <typename T, int VW>
__global__ void __launch_bounds__(kBlock) spmm_fixup_kernel(ChunkList cl, int nfrag,
                                                            const float *__restrict__ partial,
                                                            T *__restrict__ Y, int64_t ldy) {
  const int64_t j = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (j >= cl.n_long) return;
  const int lane = threadIdx.x & 31;
  const int64_t row = cl.long_rows[j];
  const int c0 = cl.long_ptr[j], c1 = cl.long_ptr[j + 1];
  const int64_t F = (int64_t)nfrag * VW;
  for (int f = lane; f < nfrag; f += 32) {
    float acc[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] = 0.f;
    float comp[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) comp[v] = 0.f;
    for (int c = c0; c < c1; ++c) {
      const float *src = partial + (int64_t)c * F + (int64_t)f * VW;
#pragma unroll
      for (int v = 0; v < VW; ++v) accum<true>(acc[v], comp[v], 1.f, __ldcg(src + v));
    }
    store_frag<T, VW>(Y + row * ldy + (int64_t)f * VW, acc);
  }
}

// ---------------------------------------------------------------- merge path

// Diagonal d of the merge of row ends (row_ptr[1..n]) with edge indices:
// returns (rows consumed, edges consumed), row ends taken first on ties.
__device__ __forceinline__ int2 merge_path_search(int64_t d, int64_t n_rows, int64_t nnz,
                                                  const int32_t *__restrict__ row_ptr) {
  int64_t lo = d - nnz > 0 ? d - nnz : 0;
  int64_t hi = d < n_rows ? d : n_rows;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if ((int64_t)row_ptr[mid + 1] <= d - mid - 1)
      lo = mid + 1;
    else
      hi = mid;
  }
  return make_int2(static_cast<int>(lo), static_cast<int>(d - lo));
}

__global__ void mergepath_partition_kernel(int64_t n_rows, int64_t nnz,
                                           const int32_t *__restrict__ row_ptr, int64_t items,
                                           int64_t n_warps, int2 *__restrict__ part) {
  const int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (w > n_warps) return;
  int64_t d = w * items;
  if (d > n_rows + nnz) d = n_rows + nnz;
  part[w] = merge_path_search(d, n_rows, nnz, row_ptr);
}

// Edges of one warp's share that the staged merge path keeps in shared
// memory (with their weights and the share's row bounds): shares of at most
// this many items are staged.
constexpr int kStageItems = 256;

// STAGED: the warp first copies its share's column indices, weights and row
// bounds into shared memory with coalesced loads (one memory round trip for
// the share), so no row waits on its own index loads; the gathers and the
// order of additions are those of the plain form.
// Blocks per SM the staged form's register budget is sized for: lanes of up
// to 4 elements run four 256-thread blocks (64 registers), lanes of 8 three
// (80 registers; at 85 the allocation rounds up and only two fit: R-MAT
// F = 256 ran 1.84 ms against 1.49 ms at three blocks, F = 64 0.57 ms at
// three blocks against 0.52 ms at four). Lanes of more than 4 fragments
// (single-element fragments of unaligned rows) spilled at those bounds.
template <int VW, int NV, bool STAGED>
constexpr int mp_min_blocks() {
  return (!STAGED || NV > 4) ? 1 : (NV * VW <= 4 ? 4 : (NV * VW <= 8 ? 3 : 1));
}

template <typename T, int VW, int NV, bool COMP, bool STAGED>
__global__ void __launch_bounds__(kBlock, mp_min_blocks<VW, NV, STAGED>()) spmm_mergepath_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const float *__restrict__ vals, const T *__restrict__ X, int64_t ldx, T *__restrict__ Y,
    int64_t ldy, int nfrag, int G, int E, const int2 *__restrict__ part, int64_t n_warps,
    float *__restrict__ carry_val, int32_t *__restrict__ carry_row, float *__restrict__ head_val) {
  const int64_t w = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (w >= n_warps) return;  // whole warps leave together
  const Lanes L(G, E);       // G * E == 32: one group per warp
  const int2 s0 = part[w], s1 = part[w + 1];
  const int head[NV] = {};
  int frag[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) frag[k] = L.g + k * G;
  constexpr int U = unroll_for<NV, VW>();
  // the share's row bounds (rp[j] = row_ptr[s0.x + j], j <= rows of the share),
  // column indices and weights
  const int32_t *rp = row_ptr + s0.x;
  const int32_t *sc = nullptr;
  const float *sv = nullptr;
  if constexpr (STAGED) {
    __shared__ int32_t s_rp[kBlock / 32][kStageItems + 1];
    __shared__ int32_t s_col[kBlock / 32][kStageItems];
    __shared__ float s_val[kBlock / 32][kStageItems];
    const int wl = threadIdx.x >> 5;
    const int nr = s1.x - s0.x, ne = s1.y - s0.y;  // nr + ne <= items <= kStageItems
    for (int j = L.lane; j <= nr; j += 32) s_rp[wl][j] = __ldg(row_ptr + s0.x + j);
    for (int j = L.lane; j < ne; j += 32) s_col[wl][j] = ld_stream_i32(col_idx + s0.y + j);
    if (vals)
      for (int j = L.lane; j < ne; j += 32) s_val[wl][j] = ld_stream_f32(vals + s0.y + j);
    __syncwarp();
    rp = s_rp[wl];
    sc = s_col[wl];
    sv = vals ? s_val[wl] : nullptr;
  }
  auto gather = [&](int p0, int pe, float (&acc)[NV][VW], float (&comp)[NV][VW]) {
    if constexpr (STAGED)
      gather_staged<T, VW, NV, U, COMP>(sc, sv, s0.y, X, ldx, nfrag, frag, E, p0, pe, acc, comp);
    else
      gather_edges<T, VW, NV, U, COMP>(col_idx, vals, 1, 1, true, head, X, ldx, nfrag, frag, E, p0, pe, acc,
                                       comp);
  };
  for (int i = s0.x; i < s1.x; ++i) {
    const int b = max(rp[i - s0.x], s0.y), e = rp[i + 1 - s0.x];
    float acc[NV][VW], comp[NV][VW];
    zero(acc);
    zero(comp);
    gather(b + L.e, e, acc, comp);
    reduce_edge_lanes(acc, FULL, G, 32);
    if (L.e != 0) continue;
    if (i == s0.x && rp[0] < s0.y) {
      // the last segment of a row that earlier warps began: kept in fp32 for
      // the fix-up, which adds the carries and rounds the row once
      float *hv = head_val + w * (int64_t)nfrag * VW;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (L.g + k * G < nfrag) store_partial<VW>(hv + (int64_t)(L.g + k * G) * VW, acc[k]);
    } else {
      T *y = Y + (int64_t)i * ldy;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (L.g + k * G < nfrag) store_frag<T, VW>(y + (int64_t)(L.g + k * G) * VW, acc[k]);
    }
  }
  // the row left unfinished at the warp's end becomes a carry-out
  int crow = -1;
  if (s1.x < n_rows) {
    const int b = max(rp[s1.x - s0.x], s0.y);
    if (s1.y > b) {
      crow = s1.x;
      float acc[NV][VW], comp[NV][VW];
      zero(acc);
      zero(comp);
      gather(b + L.e, s1.y, acc, comp);
      reduce_edge_lanes(acc, FULL, G, 32);
      if (L.e == 0) {
        float *cv = carry_val + w * (int64_t)nfrag * VW;
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (L.g + k * G < nfrag) store_partial<VW>(cv + (int64_t)(L.g + k * G) * VW, acc[k]);
      }
    }
  }
  if (L.lane == 0) carry_row[w] = crow;
}

// The first warp carrying a row adds every carry of that row (in warp order)
// and then the fp32 segment of the row's finishing warp (the warp after the
// last carry), and rounds the sum to T once. The run of warps carrying the
// row is found 32 at a time with a ballot, and four carries are loaded ahead
// of their additions (a hub row of the skewed graph is carried by a hundred
// warps and more; loading them one by one, each behind the test for the next
// warp's row, made this the merge path's long tail).
template <typename T, int VW>
__global__ void __launch_bounds__(kBlock) mergepath_fixup_kernel(
    int64_t n_warps, int nfrag, const float *__restrict__ carry_val,
    const int32_t *__restrict__ carry_row, const float *__restrict__ head_val, T *__restrict__ Y,
    int64_t ldy) {
  const int64_t w = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (w >= n_warps) return;
  const int r = carry_row[w];
  if (r < 0 || (w > 0 && carry_row[w - 1] == r)) return;
  const int lane = threadIdx.x & 31;
  // warps w .. q_end - 1 carry row r
  int64_t q_end = w + 1;
  for (;;) {
    const int64_t q = q_end + lane;
    const bool same = q < n_warps && carry_row[q] == r;
    const unsigned other = __ballot_sync(FULL, !same);
    if (other) {
      q_end += __ffs(other) - 1;
      break;
    }
    q_end += 32;
  }
  const int64_t F = (int64_t)nfrag * VW;
  for (int f = lane; f < nfrag; f += 32) {
    float acc[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] = 0.f;
    float comp[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) comp[v] = 0.f;
    int64_t q = w;
    for (; q + 4 <= q_end; q += 4) {
      float x[4][VW];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < VW; ++v) x[u][v] = __ldcg(carry_val + (q + u) * F + (int64_t)f * VW + v);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < VW; ++v) accum<true>(acc[v], comp[v], 1.f, x[u][v]);
    }
    for (; q < q_end; ++q) {
      const float *src = carry_val + q * F + (int64_t)f * VW;
#pragma unroll
      for (int v = 0; v < VW; ++v) accum<true>(acc[v], comp[v], 1.f, __ldcg(src + v));
    }
    // warp q_end finishes row r (a carried row always ends in a later warp, so q_end < n_warps)
    if (q_end < n_warps) {
      const float *hv = head_val + q_end * F + (int64_t)f * VW;
#pragma unroll
      for (int v = 0; v < VW; ++v) accum<true>(acc[v], comp[v], 1.f, __ldcg(hv + v));
    }
    store_frag<T, VW>(Y + (int64_t)r * ldy + (int64_t)f * VW, acc);
  }
}

// ---------------------------------------------------------------- ELL slab (hybrid schedule)

// Width of the ELL slab: the rows of degree 1..7 (three degree buckets).
constexpr int kEllWidth = 8;

// G feature lanes per row, one row per lane group: the row's kEllWidth column
// slots are loaded at once (column-major, so consecutive rows' lanes read
// consecutive words); the gathers of SU real slots are in flight together
// (SU * NV <= 8 fragments per lane), and the row's sum is taken in slot order.
template <typename T, int VW, int NV>
__global__ void __launch_bounds__(kBlock) spmm_ell_kernel(int64_t n, const int32_t *__restrict__ rows,
                                                          const int32_t *__restrict__ ell_col,
                                                          const int32_t *__restrict__ ell_start,
                                                          const float *__restrict__ vals, const T *__restrict__ X,
                                                          int64_t ldx, T *__restrict__ Y, int64_t ldy, int nfrag,
                                                          int G) {
  constexpr int SU = NV >= 8 ? 1 : 8 / NV;
  const int64_t t = (int64_t)blockIdx.x * kBlock + threadIdx.x;
  const int64_t e = t / G;
  const int g = (int)(t - e * G);
  if (e >= n) return;  // no shuffles below: lanes may leave on their own
  int c[kEllWidth];
#pragma unroll
  for (int j = 0; j < kEllWidth; ++j) c[j] = ld_stream_i32(ell_col + (int64_t)j * n + e);
  const int st = ld_stream_i32(ell_start + e);
  float acc[NV][VW];
  zero(acc);
#pragma unroll
  for (int j0 = 0; j0 < kEllWidth; j0 += SU) {
    float w[SU];
    Frag<T, VW> f[SU][NV];
#pragma unroll
    for (int j = 0; j < SU; ++j) {
      w[j] = (vals && c[j0 + j] >= 0) ? __ldg(vals + st + j0 + j) : 1.f;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (c[j0 + j] >= 0 && g + k * G < nfrag) f[j][k].load(X + (int64_t)c[j0 + j] * ldx + (int64_t)(g + k * G) * VW);
    }
#pragma unroll
    for (int j = 0; j < SU; ++j)
      if (c[j0 + j] >= 0)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (g + k * G < nfrag)
#pragma unroll
            for (int v = 0; v < VW; ++v) acc[k][v] = fmaf(w[j], f[j][k].get(v), acc[k][v]);
  }
  T *y = Y + (int64_t)ld_stream_i32(rows + e) * ldy;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    if (g + k * G < nfrag) store_frag<T, VW>(y + (int64_t)(g + k * G) * VW, acc[k]);
}

template <typename T, int VW>
cudaError_t spmm_ell_vw(const Geom &g, int64_t n, const int32_t *rows, const int32_t *ell_col,
                        const int32_t *ell_start, const float *vals, const T *X, int64_t ldx, T *Y, int64_t ldy,
                        cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n * g.G + kBlock - 1) / kBlock);
#define AUTOSAGE_ELL(NVV) \
  spmm_ell_kernel<T, VW, NVV><<<grid, kBlock, 0, s>>>(n, rows, ell_col, ell_start, vals, X, ldx, Y, ldy, g.nfrag, g.G)
  switch (g.NV) {
    case 1: AUTOSAGE_ELL(1); break;
    case 2: AUTOSAGE_ELL(2); break;
    case 4: AUTOSAGE_ELL(4); break;
    case 8: AUTOSAGE_ELL(8); break;
    case 16: AUTOSAGE_ELL(16); break;
    default: return cudaErrorInvalidValue;
  }
#undef AUTOSAGE_ELL
  return cudaGetLastError();
}

// ---------------------------------------------------------------- dispatch

template <typename T, int VW>
cudaError_t spmm_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                    const float *vals, const T *X, int64_t ldx, T *Y, int64_t ldy,
                    const ChunkList &cl_in, float *partial, cudaStream_t s) {
  const Deal dl = deal_items(cl_in, n_rows, g.G * g.E, g.G);
  const ChunkList &cl = dl.cl;
  const int ipb = dl.ipb;
  const int64_t grid = dl.grid;
  if (grid > 0) {
#define AUTOSAGE_SPMM_K(NVV, CMP)                                                                 \
  spmm_rows_kernel<T, VW, NVV, CMP><<<(unsigned)grid, kBlock, 0, s>>>(                          \
      n_rows, row_ptr, col_idx, vals, g.H, g.es, g.cph, X, ldx, Y, ldy, g.nfrag, g.G, g.E, g.fs, g.ks,  \
      g.one, cl, ipb, partial)
#define AUTOSAGE_SPMM_NV(NVV)          \
  if (g.comp) AUTOSAGE_SPMM_K(NVV, true); \
  else AUTOSAGE_SPMM_K(NVV, false);
    switch (g.NV) {
      case 1: AUTOSAGE_SPMM_NV(1); break;
      case 2: AUTOSAGE_SPMM_NV(2); break;
      case 4: AUTOSAGE_SPMM_NV(4); break;
      case 8: AUTOSAGE_SPMM_NV(8); break;
      case 16: AUTOSAGE_SPMM_NV(16); break;
      default: return cudaErrorInvalidValue;
    }
#undef AUTOSAGE_SPMM_NV
#undef AUTOSAGE_SPMM_K
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cl.n_long > 0) {
    const unsigned fgrid = (unsigned)((cl.n_long + kBlock / 32 - 1) / (kBlock / 32));
    spmm_fixup_kernel<T, VW><<<fgrid, kBlock, 0, s>>>(cl, g.nfrag, partial, Y, ldy);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <typename T, int VW>
cudaError_t spmm2_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                     const float *vals1, const float *vals2, const T *X1, const T *X2, int64_t ldx, T *Y1, T *Y2,
                     int64_t ldy, const ChunkList &cl_in, float *partial, cudaStream_t s) {
  const Deal dl = deal_items(cl_in, n_rows, g.G * g.E, g.G);
  const ChunkList &cl = dl.cl;
  const int ipb = dl.ipb;
  const int64_t grid = dl.grid;
  if (grid > 0) {
#define AUTOSAGE_SPMM2_K(NVV, CMP)                                                                    \
  spmm2_rows_kernel<T, VW, NVV, CMP><<<(unsigned)grid, kBlock, 0, s>>>(                              \
      n_rows, row_ptr, col_idx, vals1, vals2, g.H, g.es, g.cph, X1, X2, ldx, Y1, Y2, ldy, g.nfrag, g.G, g.E, \
      g.fs, g.ks, g.one, cl, ipb, partial)
#define AUTOSAGE_SPMM2_NV(NVV)          \
  if (g.comp) AUTOSAGE_SPMM2_K(NVV, true); \
  else AUTOSAGE_SPMM2_K(NVV, false);
    switch (g.NV) {
      case 1: AUTOSAGE_SPMM2_NV(1); break;
      case 2: AUTOSAGE_SPMM2_NV(2); break;
      case 4: AUTOSAGE_SPMM2_NV(4); break;
      case 8: AUTOSAGE_SPMM2_NV(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef AUTOSAGE_SPMM2_NV
#undef AUTOSAGE_SPMM2_K
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cl.n_long > 0) {
    const unsigned fgrid = (unsigned)((cl.n_long + kBlock / 32 - 1) / (kBlock / 32));
    const int64_t F = (int64_t)g.nfrag * g.VW;
    spmm_fixup_kernel<T, VW><<<fgrid, kBlock, 0, s>>>(cl, g.nfrag, partial, Y1, ldy);
    spmm_fixup_kernel<T, VW><<<fgrid, kBlock, 0, s>>>(cl, g.nfrag, partial + (int64_t)cl.n_chunks * F, Y2, ldy);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <typename T, int VW>
cudaError_t mergepath_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                         const int32_t *col_idx, const float *vals, const T *X, int64_t ldx, T *Y,
                         int64_t ldy, const int2 *part, int64_t n_warps, int items, float *carry_val,
                         int32_t *carry_row, float *head_val, cudaStream_t s) {
  if (n_warps <= 0) return cudaSuccess;
  const unsigned grid = (unsigned)((n_warps + kBlock / 32 - 1) / (kBlock / 32));
  const bool staged = items <= kStageItems;
#define AUTOSAGE_MP_K(NVV, CMP, STG)                                                                    \
  spmm_mergepath_kernel<T, VW, NVV, CMP, STG><<<grid, kBlock, 0, s>>>(n_rows, row_ptr, col_idx, vals, X,  \
                                                                     ldx, Y, ldy, g.nfrag, g.G, g.E,     \
                                                                     part, n_warps, carry_val, carry_row, head_val)
#define AUTOSAGE_MP_NV(NVV)                                     \
  if (g.comp) {                                                 \
    if (staged) AUTOSAGE_MP_K(NVV, true, true);                 \
    else AUTOSAGE_MP_K(NVV, true, false);                       \
  } else {                                                      \
    if (staged) AUTOSAGE_MP_K(NVV, false, true);                \
    else AUTOSAGE_MP_K(NVV, false, false);                      \
  }
  switch (g.NV) {
    case 1: AUTOSAGE_MP_NV(1); break;
    case 2: AUTOSAGE_MP_NV(2); break;
    case 4: AUTOSAGE_MP_NV(4); break;
    case 8: AUTOSAGE_MP_NV(8); break;
    case 16: AUTOSAGE_MP_NV(16); break;
    default: return cudaErrorInvalidValue;
  }
#undef AUTOSAGE_MP_NV
#undef AUTOSAGE_MP_K
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  mergepath_fixup_kernel<T, VW><<<grid, kBlock, 0, s>>>(n_warps, g.nfrag, carry_val, carry_row, head_val, Y, ldy);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_spmm2(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                         const float *vals1, const float *vals2, const void *X1, const void *X2, int64_t ldx,
                         void *Y1, void *Y2, int64_t ldy, const ChunkList &cl, float *partial, cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto x1 = static_cast<const float *>(X1), x2 = static_cast<const float *>(X2);
    auto y1 = static_cast<float *>(Y1), y2 = static_cast<float *>(Y2);
    switch (g.VW) {
      case 4: return spmm2_vw<float, 4>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
      case 2: return spmm2_vw<float, 2>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
      case 1: return spmm2_vw<float, 1>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
    }
  } else {
    auto x1 = static_cast<const __nv_bfloat16 *>(X1), x2 = static_cast<const __nv_bfloat16 *>(X2);
    auto y1 = static_cast<__nv_bfloat16 *>(Y1), y2 = static_cast<__nv_bfloat16 *>(Y2);
    switch (g.VW) {
      case 8: return spmm2_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
      case 4: return spmm2_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
      case 2: return spmm2_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
      case 1: return spmm2_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, vals1, vals2, x1, x2, ldx, y1, y2, ldy, cl, partial, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_spmm(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                        const int32_t *col_idx, const float *vals, const void *X, int64_t ldx,
                        void *Y, int64_t ldy, const ChunkList &cl, float *partial,
                        cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto x = static_cast<const float *>(X);
    auto y = static_cast<float *>(Y);
    switch (g.VW) {
      case 4: return spmm_vw<float, 4>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
      case 2: return spmm_vw<float, 2>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
      case 1: return spmm_vw<float, 1>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
    }
  } else {
    auto x = static_cast<const __nv_bfloat16 *>(X);
    auto y = static_cast<__nv_bfloat16 *>(Y);
    switch (g.VW) {
      case 8: return spmm_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
      case 4: return spmm_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
      case 2: return spmm_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
      case 1: return spmm_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, cl, partial, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_spmm_ell(const Geom &g, int64_t n, const int32_t *rows, const int32_t *ell_col,
                            const int32_t *ell_start, const float *vals, const void *X, int64_t ldx, void *Y,
                            int64_t ldy, cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto x = static_cast<const float *>(X);
    auto y = static_cast<float *>(Y);
    switch (g.VW) {
      case 4: return spmm_ell_vw<float, 4>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
      case 2: return spmm_ell_vw<float, 2>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
      case 1: return spmm_ell_vw<float, 1>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
    }
  } else {
    auto x = static_cast<const __nv_bfloat16 *>(X);
    auto y = static_cast<__nv_bfloat16 *>(Y);
    switch (g.VW) {
      case 8: return spmm_ell_vw<__nv_bfloat16, 8>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
      case 4: return spmm_ell_vw<__nv_bfloat16, 4>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
      case 2: return spmm_ell_vw<__nv_bfloat16, 2>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
      case 1: return spmm_ell_vw<__nv_bfloat16, 1>(g, n, rows, ell_col, ell_start, vals, x, ldx, y, ldy, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_mergepath_partition(int64_t n_rows, int64_t nnz, const int32_t *row_ptr,
                                       int64_t items, int64_t n_warps, int2 *part, cudaStream_t s) {
  const int64_t n = n_warps + 1;
  mergepath_partition_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(n_rows, nnz, row_ptr, items,
                                                                          n_warps, part);
  return cudaGetLastError();
}

cudaError_t launch_spmm_mergepath(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                                  const int32_t *col_idx, const float *vals, const void *X,
                                  int64_t ldx, void *Y, int64_t ldy, const int2 *part,
                                  int64_t n_warps, int items, float *carry_val, int32_t *carry_row,
                                  float *head_val, cudaStream_t s) {
  if (g.G * g.E != 32) return cudaErrorInvalidValue;
  if (g.dt == DType::F32) {
    auto x = static_cast<const float *>(X);
    auto y = static_cast<float *>(Y);
    switch (g.VW) {
      case 4: return mergepath_vw<float, 4>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
      case 2: return mergepath_vw<float, 2>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
      case 1: return mergepath_vw<float, 1>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
    }
  } else {
    auto x = static_cast<const __nv_bfloat16 *>(X);
    auto y = static_cast<__nv_bfloat16 *>(Y);
    switch (g.VW) {
      case 8: return mergepath_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
      case 4: return mergepath_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
      case 2: return mergepath_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
      case 1: return mergepath_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, vals, x, ldx, y, ldy, part, n_warps, items, carry_val, carry_row, head_val, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace autosage
