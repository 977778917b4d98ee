// CSR SDDMM: S[p, h] = alpha * <Q[row(p), h, :], K[col_idx[p], h, :]>
// (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN Aggregation
// (SpMM/SDDMM) and CSR Attention", Abstract: SDDMM; the first step of the
// CSR attention pipeline). Edge values of A are not multiplied in.
//
// A lane group owns a row (or a chunk of a cut row): its G feature lanes hold
// the row's Q fragments in registers for the whole row and every edge gathers
// one K row. Two ways to finish the dot products:
//  * per edge: the lanes holding a head reduce it with xor shuffles
//    (log2 R rounds per edge and head);
//  * batched (single head): each lane keeps its partial dot for G edges and
//    one transpose-reduction over the G lanes (G - 1 shuffles for G edges)
//    leaves edge j's total on lane j, which also makes the score writes of a
//    batch one contiguous store.
// Cut rows need no fix-up: every edge's score is complete within its chunk.
#include "internal.h"

namespace autosage {

namespace {

// Per-edge reduction. Fragment slot k of lane g is fragment g * fs + k * ks.
// ONE: all slots of a lane belong to one head; otherwise slot k is its own head.
// Items of an SDDMM launch: dealt from the run table (MP = false), or (MP =
// true) a merge path: lane group w walks its equal share of (rows + edges),
// diagonals [part[w], part[w + 1]), one item per row it touches. SDDMM writes
// one value per edge, so a row cut between groups needs no carry.
template <bool MP, typename Body>
__device__ __forceinline__ void for_items(const Lanes &L, int64_t n_rows, const int32_t *__restrict__ row_ptr,
                                          const ChunkList &cl, int ipb, const int2 *__restrict__ part,
                                          int64_t n_groups, Body body) {
  if constexpr (MP) {
    const int64_t w = ((int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5)) * (32 / L.GE) + L.slot;
    if (w >= n_groups) return;  // the whole group leaves together
    const int2 s0 = part[w], s1 = part[w + 1];
    for (int64_t i = s0.x; i <= s1.x && i < n_rows; ++i) {
      const int b = max(row_ptr[i], s0.y), e = min(row_ptr[i + 1], s1.y);
      if (e > b) body(Item{i, b, e, -1, true});
    }
  } else {
    __shared__ int s_items;
    const ItemQueue queue(n_rows, cl, ipb, &s_items);
    int64_t idx;
    while (queue.next(L, idx)) body(item_at(idx, n_rows, row_ptr, cl));
  }
}

template <typename T, int VW, int NV, bool ONE, bool MP>
__global__ void __launch_bounds__(kBlock) sddmm_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const T *__restrict__ Q, int64_t ldq, const T *__restrict__ K, int64_t ldk, float alpha,
    int H, int es, int cph, int R, int nfrag, int G, int E, int fs, int ks, float *__restrict__ S,
    ChunkList cl, int ipb, const int2 *__restrict__ mp_part, int64_t n_groups) {
  constexpr int NG = ONE ? 1 : NV;
  const Lanes L(G, E);
  for_items<MP>(L, n_rows, row_ptr, cl, ipb, mp_part, n_groups, [&](const Item &it) {
  const int g = L.g;
  int frag[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) frag[k] = g * fs + k * ks;
  float q[NV][VW];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    Frag<T, VW> f;
    const bool ok = it.active && it.e > it.b && frag[k] < nfrag;
    if (ok) f.load(Q + it.row * ldq + (int64_t)frag[k] * VW);
#pragma unroll
    for (int v = 0; v < VW; ++v) q[k][v] = ok ? alpha * f.get(v) : 0.f;
  }
  constexpr int U = NV * VW <= 8 ? 4 : (NV * VW <= 16 ? 2 : 1);
  const int p0 = it.b + L.e, pe = it.e;
  int c[U];
#pragma unroll
  for (int u = 0; u < U; ++u) c[u] = p0 + u * E < pe ? ld_stream_i32(col_idx + p0 + u * E) : 0;
  for (int p = p0; p < pe; p += U * E) {
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) live[u] = p + u * E < pe;
    Frag<T, VW> f[U][NV];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (live[u] && frag[k] < nfrag) f[u][k].load(K + (int64_t)c[u] * ldk + (int64_t)frag[k] * VW);
    // next iteration's columns are fetched while these rows are in flight
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int qe = p + U * E + u * E;
      c[u] = qe < pe ? ld_stream_i32(col_idx + qe) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float hs[NG];
#pragma unroll
      for (int j = 0; j < NG; ++j) hs[j] = 0.f;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (live[u] && frag[k] < nfrag) {
          float d = 0.f;
#pragma unroll
          for (int v = 0; v < VW; ++v) d = fmaf(q[k][v], f[u][k].get(v), d);
          hs[ONE ? 0 : k] += d;
        }
      }
      // every lane of this edge lane's G-lane segment runs the same trip count
#pragma unroll
      for (int j = 0; j < NG; ++j)
        for (int off = 1; off < R; off <<= 1) hs[j] += __shfl_xor_sync(L.sub_mask, hs[j], off);
      if (live[u] && (g % R) == 0) {
        const int64_t pp = p + u * E;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          if (frag[j] < nfrag) {
            const int h = H > 1 ? frag[j] / cph : 0;
            S[pp * es + h] = hs[j];
          }
        }
      }
    }
  }
  });
}

// Batched single-head SDDMM: each edge lane's G feature lanes take B edges
// at a time (B divides G). Every lane computes its partial dot for all B
// edges; a transpose-reduction inside each aligned B-lane segment (B - 1
// shuffles) leaves edge j's segment sum on lane j of the segment, and log2(G/B)
// plain xor rounds add the segments. Lanes 0..B-1 then hold the B scores.
template <typename T, int VW, int NV, int B, bool MP>
__global__ void __launch_bounds__(kBlock) sddmm_batched_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const T *__restrict__ Q, int64_t ldq, const T *__restrict__ K, int64_t ldk, float alpha, int es,
    int nfrag, int G, int E, float *__restrict__ S, ChunkList cl, int ipb, const int2 *__restrict__ mp_part,
    int64_t n_groups) {
  const Lanes L(G, E);
  const int g = L.g;
  const int base_lane = L.slot * L.GE + L.e * G;  // lane 0 of this edge lane's segment
  // loads of the whole batch in flight when a lane holds at most two fragments
  constexpr int U = NV <= 2 ? B : (B < 4 ? B : 4);
  for_items<MP>(L, n_rows, row_ptr, cl, ipb, mp_part, n_groups, [&](const Item &it) {
    Frag<T, VW> q[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (it.active && it.e > it.b && g + k * G < nfrag)
        q[k].load(Q + it.row * ldq + (int64_t)(g + k * G) * VW);
      else
        q[k].zero();
    }
    // edges of this edge lane: p = it.b + e + E * t; batches of B consecutive t
    const int first = it.b + L.e;
    const int n_mine = it.e > first ? (it.e - first + E - 1) / E : 0;
    // one load brings a batch's column indices (lane j holding edge j's); the
    // next batch's indices are requested while this batch's rows are in flight
    int next_col = (g < B && g < n_mine) ? ld_stream_i32(col_idx + first + g * E) : 0;
    for (int t0 = 0; t0 < n_mine; t0 += B) {
      const int nb = min(B, n_mine - t0);
      const int pj = first + (t0 + g) * E;
      const int my_col = next_col;
      next_col = (g < B && t0 + B + g < n_mine) ? ld_stream_i32(col_idx + first + (t0 + B + g) * E) : 0;
      float part[B];
#pragma unroll
      for (int j0 = 0; j0 < B; j0 += U) {
        Frag<T, VW> f[U][NV];
        int cj[U];
#pragma unroll
        for (int u = 0; u < U; ++u) cj[u] = __shfl_sync(L.sub_mask, my_col, base_lane + j0 + u);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int k = 0; k < NV; ++k)
            if (j0 + u < nb && g + k * G < nfrag)
              f[u][k].load(K + (int64_t)cj[u] * ldk + (int64_t)(g + k * G) * VW);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          float d = 0.f;
#pragma unroll
          for (int k = 0; k < NV; ++k)
            if (j0 + u < nb && g + k * G < nfrag)
#pragma unroll
              for (int v = 0; v < VW; ++v) d = fmaf(q[k].get(v), f[u][k].get(v), d);
          part[j0 + u] = d;
        }
      }
      // after the stage on bit s, a lane keeps the half of the edges whose
      // index has its own bit s, summed with its partner's half
#pragma unroll
      for (int sbit = B / 2; sbit >= 1; sbit >>= 1) {
        const bool upper = (g & sbit) != 0;
#pragma unroll
        for (int i = 0; i < sbit; ++i) {
          const float send = upper ? part[i] : part[i + sbit];
          const float keep = upper ? part[i + sbit] : part[i];
          part[i] = keep + __shfl_xor_sync(L.sub_mask, send, sbit);
        }
      }
      for (int off = B; off < G; off <<= 1) part[0] += __shfl_xor_sync(L.sub_mask, part[0], off);
      if (g < nb) S[(int64_t)pj * es] = alpha * part[0];
    }
  });
}

template <typename T, int VW, int NV>
cudaError_t launch_batched(const Geom &g, int64_t grid, int ipb, int64_t n_rows, const int32_t *row_ptr,
                           const int32_t *col_idx, const T *Q, int64_t ldq, const T *K, int64_t ldk,
                           float alpha, float *S, const ChunkList &cl, const int2 *mp_part, int64_t n_groups,
                           cudaStream_t s) {
#define AUTOSAGE_SDDMM_B(BB, MPP)                                                                         \
  sddmm_batched_kernel<T, VW, NV, BB, MPP><<<(unsigned)grid, kBlock, 0, s>>>(                           \
      n_rows, row_ptr, col_idx, Q, ldq, K, ldk, alpha, g.es, g.nfrag, g.G, g.E, S, cl, ipb, mp_part, n_groups)
  if (g.G >= 8) {
    if (mp_part) AUTOSAGE_SDDMM_B(8, true);
    else AUTOSAGE_SDDMM_B(8, false);
  } else if (g.G == 4) {
    if (mp_part) AUTOSAGE_SDDMM_B(4, true);
    else AUTOSAGE_SDDMM_B(4, false);
  } else {
    return cudaErrorInvalidValue;
  }
#undef AUTOSAGE_SDDMM_B
  return cudaGetLastError();
}

template <typename T, int VW>
cudaError_t sddmm_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                     const T *Q, int64_t ldq, const T *K, int64_t ldk, float alpha, float *S,
                     const ChunkList &cl_in, const int2 *mp_part, int64_t n_groups, cudaStream_t s) {
  const Deal dl = deal_items(cl_in, n_rows, g.G * g.E, g.G);
  const ChunkList &cl = dl.cl;
  const int ipb = dl.ipb;
  // merge path: one lane group per partition, 256 / (G * E) groups per block
  const int64_t gpb = (int64_t)(kBlock / 32) * (32 / (g.G * g.E));
  const int64_t grid = mp_part ? (n_groups + gpb - 1) / gpb : dl.grid;
  if (grid <= 0) return cudaSuccess;
  // batched transpose-reduction: single head, 16-byte fragments, 2..32 lanes
  if constexpr (sizeof(T) * VW == 16) {
    if (g.H == 1 && g.batched && g.G >= 2 && g.fs == 1 && g.NV <= 4) {
      switch (g.NV) {
        case 1: return launch_batched<T, VW, 1>(g, grid, ipb, n_rows, row_ptr, col_idx, Q, ldq, K, ldk, alpha, S, cl, mp_part, n_groups, s);
        case 2: return launch_batched<T, VW, 2>(g, grid, ipb, n_rows, row_ptr, col_idx, Q, ldq, K, ldk, alpha, S, cl, mp_part, n_groups, s);
        case 4: return launch_batched<T, VW, 4>(g, grid, ipb, n_rows, row_ptr, col_idx, Q, ldq, K, ldk, alpha, S, cl, mp_part, n_groups, s);
      }
    }
  }
#define AUTOSAGE_SDDMM2(NVV, ONEG, MPP)                                                              \
  sddmm_kernel<T, VW, NVV, ONEG, MPP><<<(unsigned)grid, kBlock, 0, s>>>(                            \
      n_rows, row_ptr, col_idx, Q, ldq, K, ldk, alpha, g.H, g.es, g.cph, g.R, g.nfrag, g.G, g.E,     \
      g.fs, g.ks, S, cl, ipb, mp_part, n_groups)
#define AUTOSAGE_SDDMM(NVV, ONEG)                      \
  if (mp_part) AUTOSAGE_SDDMM2(NVV, ONEG, true);       \
  else AUTOSAGE_SDDMM2(NVV, ONEG, false);
#define AUTOSAGE_SDDMM_NV(NVV)                \
  if (g.one) { AUTOSAGE_SDDMM(NVV, true) }    \
  else { AUTOSAGE_SDDMM(NVV, false) }
  switch (g.NV) {
    case 1: AUTOSAGE_SDDMM_NV(1); break;
    case 2: AUTOSAGE_SDDMM_NV(2); break;
    case 4: AUTOSAGE_SDDMM_NV(4); break;
    case 8: AUTOSAGE_SDDMM_NV(8); break;
    case 16: AUTOSAGE_SDDMM_NV(16); break;
    default: return cudaErrorInvalidValue;
  }
#undef AUTOSAGE_SDDMM_NV
#undef AUTOSAGE_SDDMM
#undef AUTOSAGE_SDDMM2
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sddmm(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                         const int32_t *col_idx, const void *Q, int64_t ldq, const void *K,
                         int64_t ldk, float alpha, float *S, const ChunkList &cl, const int2 *mp_part,
                         int64_t n_groups, cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto q = static_cast<const float *>(Q);
    auto k = static_cast<const float *>(K);
    switch (g.VW) {
      case 4: return sddmm_vw<float, 4>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
      case 2: return sddmm_vw<float, 2>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
      case 1: return sddmm_vw<float, 1>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
    }
  } else {
    auto q = static_cast<const __nv_bfloat16 *>(Q);
    auto k = static_cast<const __nv_bfloat16 *>(K);
    switch (g.VW) {
      case 8: return sddmm_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
      case 4: return sddmm_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
      case 2: return sddmm_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
      case 1: return sddmm_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, mp_part, n_groups, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace autosage
