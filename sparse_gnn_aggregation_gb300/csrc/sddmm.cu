// CSR SDDMM: S[p, h] = alpha * <Q[row(p), h, :], K[col_idx[p], h, :]>
// (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse GNN Aggregation
// (SpMM/SDDMM) and CSR Attention", Abstract: "SDDMM"; the first step of the
// CSR attention pipeline). Edge values of A are not multiplied in.
//
// A lane group owns a row (or a chunk of a cut row): its G feature lanes hold
// the row's Q fragments in registers for the whole row, every edge gathers one
// K row, and the per-head dot product is finished by xor shuffles among the
// lanes holding that head. Cut rows need no fix-up: every edge's score is
// complete within its chunk.
#include "internal.h"

namespace autosage {

namespace {

template <typename T, int VW, int NV, int U>
__device__ __forceinline__ void sddmm_edges(const Lanes &L, const int32_t *__restrict__ col_idx,
                                            const T *__restrict__ K, int64_t ldk,
                                            const float (&q)[NV][VW], int nfrag, int H, int es,
                                            int cph, int mshift, int R, float *__restrict__ S, int p0,
                                            int pe) {
  const int G = L.G, E = L.E, g = L.g;
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
        if (live[u] && g + k * G < nfrag) f[u][k].load(K + (int64_t)c[u] * ldk + (int64_t)(g + k * G) * VW);
    // next iteration's columns are fetched while these rows are in flight
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = p + U * E + u * E;
      c[u] = q < pe ? ld_stream_i32(col_idx + q) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      // partial dot per fragment slot, summed into head groups of 2^mshift slots
      float hs[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k) hs[k] = 0.f;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (live[u] && g + k * G < nfrag) {
          float d = 0.f;
#pragma unroll
          for (int v = 0; v < VW; ++v) d = fmaf(q[k][v], f[u][k].get(v), d);
          hs[k >> mshift] += d;
        }
      }
      // every lane of this edge lane's G-lane segment runs the same trip count
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        if ((j << mshift) >= NV) break;
        for (int off = 1; off < R; off <<= 1) hs[j] += __shfl_xor_sync(L.sub_mask, hs[j], off);
      }
      if (live[u]) {
        const int64_t pp = p + u * E;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          if ((j << mshift) >= NV) break;
          const int c0 = g + (j << mshift) * G;  // first fragment of this head group
          if (c0 < nfrag && (g % R) == 0) {
            const int h = H > 1 ? c0 / cph : 0;
            S[pp * es + h] = hs[j];
          }
        }
      }
    }
  }
}

template <typename T, int VW, int NV>
__global__ void __launch_bounds__(kBlock) sddmm_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const T *__restrict__ Q, int64_t ldq, const T *__restrict__ K, int64_t ldk, float alpha,
    int H, int es, int cph, int mshift, int R, int nfrag, int G, int E, float *__restrict__ S,
    ChunkList cl, int64_t chunk_blocks) {
  const Lanes L(G, E);
  const Item it = resolve_item(L, n_rows, row_ptr, cl, chunk_blocks);
  float q[NV][VW];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    Frag<T, VW> f;
    const bool ok = it.active && it.e > it.b && L.g + k * G < nfrag;
    if (ok) f.load(Q + it.row * ldq + (int64_t)(L.g + k * G) * VW);
#pragma unroll
    for (int v = 0; v < VW; ++v) q[k][v] = ok ? alpha * f.get(v) : 0.f;
  }
  constexpr int U = NV * VW <= 8 ? 4 : (NV * VW <= 16 ? 2 : 1);
  sddmm_edges<T, VW, NV, U>(L, col_idx, K, ldk, q, nfrag, H, es, cph, mshift, R, S, it.b + L.e, it.e);
}

template <typename T, int VW>
cudaError_t sddmm_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                     const T *Q, int64_t ldq, const T *K, int64_t ldk, float alpha, float *S,
                     const ChunkList &cl, cudaStream_t s) {
  const int64_t per_block = (kBlock / 32) * (32 / (g.G * g.E));
  const int64_t chunk_blocks = (cl.n_chunks + per_block - 1) / per_block;
  const int64_t grid = chunk_blocks + (n_rows + per_block - 1) / per_block;
  if (grid <= 0) return cudaSuccess;
#define AUTOSAGE_SDDMM_NV(NVV)                                                                    \
  sddmm_kernel<T, VW, NVV><<<(unsigned)grid, kBlock, 0, s>>>(n_rows, row_ptr, col_idx, Q, ldq, K, \
                                                             ldk, alpha, g.H, g.es, g.cph, g.mshift, \
                                                             g.R, g.nfrag, g.G, g.E, S, cl,      \
                                                             chunk_blocks)
  switch (g.NV) {
    case 1: AUTOSAGE_SDDMM_NV(1); break;
    case 2: AUTOSAGE_SDDMM_NV(2); break;
    case 4: AUTOSAGE_SDDMM_NV(4); break;
    case 8: AUTOSAGE_SDDMM_NV(8); break;
    case 16: AUTOSAGE_SDDMM_NV(16); break;
    default: return cudaErrorInvalidValue;
  }
#undef AUTOSAGE_SDDMM_NV
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sddmm(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                         const int32_t *col_idx, const void *Q, int64_t ldq, const void *K,
                         int64_t ldk, float alpha, float *S, const ChunkList &cl, cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto q = static_cast<const float *>(Q);
    auto k = static_cast<const float *>(K);
    switch (g.VW) {
      case 4: return sddmm_vw<float, 4>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
      case 2: return sddmm_vw<float, 2>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
      case 1: return sddmm_vw<float, 1>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
    }
  } else {
    auto q = static_cast<const __nv_bfloat16 *>(Q);
    auto k = static_cast<const __nv_bfloat16 *>(K);
    switch (g.VW) {
      case 8: return sddmm_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
      case 4: return sddmm_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
      case 2: return sddmm_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
      case 1: return sddmm_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, q, ldq, k, ldk, alpha, S, cl, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace autosage
