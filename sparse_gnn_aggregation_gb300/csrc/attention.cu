// Fused CSR attention (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse
// GNN Aggregation (SpMM/SDDMM) and CSR Attention", Abstract: the pipeline
// SDDMM -> row-softmax -> SpMM; benchmark page "fused sparse
// attention-value aggregation": softmax weights of a destination's incoming
// edges aggregate the source values, an edgeless row gives zeros).
//
// One pass per row with an online softmax: per head a running maximum m,
// running sum l and running weighted sum acc; each new score s rescales the
// state by exp(m_old - m_new). Scores never reach HBM. A group of G feature
// lanes x E edge lanes owns a row: lanes hold the row's (pre-scaled) Q
// fragments, gather K and V rows of the row's sources, finish each head's
// dot product by xor shuffles, and at the end merge the E edge-lane states
// in a fixed order. Rows longer than `split` edges are cut into chunks that
// write (m, l, acc) partials; a fix-up merges them in chunk order. With
// given scores (the benchmark page's op) the dot products are replaced by
// reads of the score array.
#include "internal.h"

namespace autosage {

namespace {

template <typename T, int VW, int NV, bool GIVEN>
__global__ void __launch_bounds__(kBlock) attention_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const T *__restrict__ Q, const T *__restrict__ K, const float *__restrict__ scores,
    const T *__restrict__ V, int64_t ld, float scale, int H, int es, int cph, int mshift, int R, int nfrag,
    int G, int E, T *__restrict__ O, ChunkList cl, int64_t chunk_blocks,
    float *__restrict__ part_acc, float *__restrict__ part_ml) {
  const Lanes L(G, E);
  const Item it = resolve_item(L, n_rows, row_ptr, cl, chunk_blocks);
  const int g = L.g;
  bool valid[NV];
  int head[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    valid[k] = g + k * G < nfrag;
    head[k] = (H > 1 && valid[k]) ? (g + k * G) / cph : 0;
  }
  float q[NV][VW];
  if constexpr (!GIVEN) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      Frag<T, VW> f;
      const bool ok = it.e > it.b && valid[k];
      if (ok) f.load(Q + it.row * ld + (int64_t)(g + k * G) * VW);
#pragma unroll
      for (int v = 0; v < VW; ++v) q[k][v] = ok ? scale * f.get(v) : 0.f;
    }
  }
  float m[NV], l[NV], acc[NV][VW];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    m[k] = -INFINITY;
    l[k] = 0.f;
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[k][v] = 0.f;
  }
  constexpr int U = NV * VW <= 8 ? 4 : 2;
  int c[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int q = it.b + L.e + u * E;
    c[u] = q < it.e ? ld_stream_i32(col_idx + q) : 0;
  }
  for (int p = it.b + L.e; p < it.e; p += U * E) {
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) live[u] = p + u * E < it.e;
    int cn[U];  // next iteration's columns, fetched while this iteration's rows are in flight
    Frag<T, VW> fv[U][NV];
    float s[U][NV];
    if constexpr (GIVEN) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          s[u][k] = live[u] ? __ldg(scores + (int64_t)(p + u * E) * es + head[k]) : -INFINITY;
    } else {
      Frag<T, VW> fk[U][NV];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (live[u] && valid[k]) fk[u][k].load(K + (int64_t)c[u] * ld + (int64_t)(g + k * G) * VW);
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (live[u] && valid[k]) fv[u][k].load(V + (int64_t)c[u] * ld + (int64_t)(g + k * G) * VW);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int q = p + U * E + u * E;
        cn[u] = q < it.e ? ld_stream_i32(col_idx + q) : 0;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float hs[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) hs[k] = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          if (valid[k]) {
            float d = 0.f;
#pragma unroll
            for (int v = 0; v < VW; ++v) d = fmaf(q[k][v], fk[u][k].get(v), d);
            hs[k >> mshift] += d;
          }
        }
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          if ((j << mshift) >= NV) break;
          for (int off = 1; off < R; off <<= 1) hs[j] += __shfl_xor_sync(L.sub_mask, hs[j], off);
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) s[u][k] = live[u] ? hs[k >> mshift] : -INFINITY;
      }
    }
    if constexpr (GIVEN) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (live[u] && valid[k]) fv[u][k].load(V + (int64_t)c[u] * ld + (int64_t)(g + k * G) * VW);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int q = p + U * E + u * E;
        cn[u] = q < it.e ? ld_stream_i32(col_idx + q) : 0;
      }
    }
    // online softmax update with U new scores per fragment slot
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float mx = m[k];
#pragma unroll
      for (int u = 0; u < U; ++u) mx = fmaxf(mx, s[u][k]);
      // m[k] = -inf (first edges) gives 0; an all -inf set of scores leaves the state as is
      const float corr = mx == -INFINITY ? 1.f : __expf(m[k] - mx);
      l[k] *= corr;
#pragma unroll
      for (int v = 0; v < VW; ++v) acc[k][v] *= corr;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (live[u]) {
          const float w = mx == -INFINITY ? 0.f : __expf(s[u][k] - mx);
          l[k] += w;
          if (valid[k]) {
#pragma unroll
            for (int v = 0; v < VW; ++v) acc[k][v] = fmaf(w, fv[u][k].get(v), acc[k][v]);
          }
        }
      }
      m[k] = mx;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) c[u] = cn[u];
  }
  // merge the E edge-lane states (fixed xor order)
  for (int off = G; off < L.GE; off <<= 1) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float mo = __shfl_xor_sync(L.group_mask, m[k], off);
      const float lo = __shfl_xor_sync(L.group_mask, l[k], off);
      const float mx = fmaxf(m[k], mo);
      const float a = mx == -INFINITY ? 0.f : __expf(m[k] - mx);
      const float b = mx == -INFINITY ? 0.f : __expf(mo - mx);
      l[k] = l[k] * a + lo * b;
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        const float ao = __shfl_xor_sync(L.group_mask, acc[k][v], off);
        acc[k][v] = acc[k][v] * a + ao * b;
      }
      m[k] = mx;
    }
  }
  if (!it.active || L.e != 0) return;
  if (it.chunk < 0) {
    T *o = O + it.row * ld;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (!valid[k]) continue;
      const float inv = l[k] > 0.f ? 1.f / l[k] : 0.f;
      float r[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) r[v] = acc[k][v] * inv;
      store_frag<T, VW>(o + (int64_t)(g + k * G) * VW, r);
    }
  } else {
    float *pa = part_acc + (int64_t)it.chunk * nfrag * VW;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (!valid[k]) continue;
      store_partial<VW>(pa + (int64_t)(g + k * G) * VW, acc[k]);
      if ((g + k * G) % cph == 0) {
        float *pm = part_ml + ((int64_t)it.chunk * H + head[k]) * 2;
        __stcg(pm, m[k]);
        __stcg(pm + 1, l[k]);
      }
    }
  }
}

// One warp per cut row: merge the (m, l, acc) partials of its chunks in order.
template <typename T, int VW>
__global__ void __launch_bounds__(kBlock) attention_fixup_kernel(ChunkList cl, int H, int cph,
                                                                 int nfrag,
                                                                 const float *__restrict__ part_acc,
                                                                 const float *__restrict__ part_ml,
                                                                 T *__restrict__ O, int64_t ld) {
  const int64_t j = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (j >= cl.n_long) return;
  const int lane = threadIdx.x & 31;
  const int64_t row = cl.long_rows[j];
  const int c0 = cl.long_ptr[j], c1 = cl.long_ptr[j + 1];
  const int64_t F = (int64_t)nfrag * VW;
  for (int f = lane; f < nfrag; f += 32) {
    const int h = f / cph;
    float m = -INFINITY, l = 0.f, acc[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] = 0.f;
    for (int c = c0; c < c1; ++c) {
      const float mc = __ldcg(part_ml + ((int64_t)c * H + h) * 2);
      const float lc = __ldcg(part_ml + ((int64_t)c * H + h) * 2 + 1);
      const float mx = fmaxf(m, mc);
      const float a = mx == -INFINITY ? 0.f : __expf(m - mx);
      const float b = mx == -INFINITY ? 0.f : __expf(mc - mx);
      l = l * a + lc * b;
      const float *src = part_acc + (int64_t)c * F + (int64_t)f * VW;
#pragma unroll
      for (int v = 0; v < VW; ++v) acc[v] = acc[v] * a + __ldcg(src + v) * b;
      m = mx;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int v = 0; v < VW; ++v) acc[v] *= inv;
    store_frag<T, VW>(O + row * ld + (int64_t)f * VW, acc);
  }
}

template <typename T, int VW>
cudaError_t attention_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                         const int32_t *col_idx, const T *Q, const T *K, const float *scores,
                         const T *V, int64_t ld, float scale, T *O, const ChunkList &cl,
                         float *part_acc, float *part_ml, cudaStream_t s) {
  const int64_t per_block = (kBlock / 32) * (32 / (g.G * g.E));
  const int64_t chunk_blocks = (cl.n_chunks + per_block - 1) / per_block;
  const int64_t grid = chunk_blocks + (n_rows + per_block - 1) / per_block;
  if (grid > 0) {
#define AUTOSAGE_ATTN(NVV, GIV)                                                                    \
  attention_kernel<T, VW, NVV, GIV><<<(unsigned)grid, kBlock, 0, s>>>(                           \
      n_rows, row_ptr, col_idx, Q, K, scores, V, ld, scale, g.H, g.es, g.cph, g.mshift, g.R, g.nfrag, \
      g.G, g.E, O, cl, chunk_blocks, part_acc, part_ml)
#define AUTOSAGE_ATTN_NV(NVV)           \
  if (scores) AUTOSAGE_ATTN(NVV, true); \
  else AUTOSAGE_ATTN(NVV, false);
    switch (g.NV) {
      case 1: AUTOSAGE_ATTN_NV(1); break;
      case 2: AUTOSAGE_ATTN_NV(2); break;
      case 4: AUTOSAGE_ATTN_NV(4); break;
      case 8: AUTOSAGE_ATTN_NV(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef AUTOSAGE_ATTN_NV
#undef AUTOSAGE_ATTN
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cl.n_long > 0) {
    const unsigned fgrid = (unsigned)((cl.n_long + kBlock / 32 - 1) / (kBlock / 32));
    attention_fixup_kernel<T, VW><<<fgrid, kBlock, 0, s>>>(cl, g.H, g.cph, g.nfrag, part_acc,
                                                            part_ml, O, ld);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_attention(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                             const int32_t *col_idx, const void *Q, const void *K,
                             const float *scores, const void *V, int64_t ld, float scale,
                             void *O, const ChunkList &cl, float *part_acc, float *part_ml,
                             cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto q = static_cast<const float *>(Q);
    auto k = static_cast<const float *>(K);
    auto v = static_cast<const float *>(V);
    auto o = static_cast<float *>(O);
    switch (g.VW) {
      case 4: return attention_vw<float, 4>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
      case 2: return attention_vw<float, 2>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
      case 1: return attention_vw<float, 1>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
    }
  } else {
    auto q = static_cast<const __nv_bfloat16 *>(Q);
    auto k = static_cast<const __nv_bfloat16 *>(K);
    auto v = static_cast<const __nv_bfloat16 *>(V);
    auto o = static_cast<__nv_bfloat16 *>(O);
    switch (g.VW) {
      case 8: return attention_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
      case 4: return attention_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
      case 2: return attention_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
      case 1: return attention_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, q, k, scores, v, ld, scale, o, cl, part_acc, part_ml, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace autosage
