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
#include <type_traits>

#include "internal.h"

namespace autosage {

namespace {

// Scores more than kRescale above the running reference m trigger a rescale
// of (l, acc) to the new maximum; smaller increases keep the old reference,
// so exp(s - m) stays below e^kRescale and the common case skips the rescale.
// The result acc / l does not depend on which reference was used.
constexpr float kRescale = 8.f;

// Fragment slot k of lane g covers fragment g * fs + k * ks: fs = 1, ks = G
// interleaves lanes (one coalesced load per slot); fs = NV, ks = 1 gives each
// lane NV consecutive fragments, which keeps a lane inside one head.
// ONE: all of a lane's slots belong to one head (single-head rows, or
// consecutive fragments within a head): one running (m, l) and one exp per
// edge. Otherwise every slot is its own head (interleaved lanes, heads of
// at most G fragments). R lanes share a head and finish its dot product with
// xor shuffles. ALLV: every slot of every lane holds a fragment (nfrag =
// G * NV), so the per-slot validity tests drop out.
// Blocks per SM the register budget is sized for: lanes holding few values
// (bf16 up to 16, fp32 up to 4) leave room for three 256-thread blocks
// (85 registers per thread); wider ones get two.
template <typename T, int VW, int NV>
constexpr int attn_min_blocks() {
  return (NV * VW <= 4 || (sizeof(T) == 2 && NV * VW <= 16)) ? 3 : 2;
}

template <typename T, int VW, int NV, bool GIVEN, bool ONE, bool ALLV>
__global__ void __launch_bounds__(kBlock, attn_min_blocks<T, VW, NV>()) attention_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const T *__restrict__ Q, const T *__restrict__ K, const float *__restrict__ scores,
    const T *__restrict__ V, int64_t ld, float scale, int H, int es, int cph, int R, int nfrag,
    int G, int E, int fs, int ks, T *__restrict__ O, ChunkList cl, int ipb,
    float *__restrict__ part_acc, float *__restrict__ part_ml) {
  constexpr int NG = ONE ? 1 : NV;  // head groups per lane
  const Lanes L(G, E);
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
  const Item it = item_at(idx, n_rows, row_ptr, cl);
  const int g = L.g;
  bool valid[NV];
  int frag[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    frag[k] = g * fs + k * ks;
    valid[k] = frag[k] < nfrag;
  }
  int head[NG];
#pragma unroll
  for (int j = 0; j < NG; ++j) head[j] = (H > 1 && frag[j] < nfrag) ? frag[j] / cph : 0;
  // the row's Q fragments stay packed (bf16 halves the registers); the scale
  // is applied to the finished dot product
  Frag<T, VW> q[NV];
  if constexpr (!GIVEN) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (it.e > it.b && valid[k])
        q[k].load(Q + it.row * ld + (int64_t)frag[k] * VW);
      else
        q[k].zero();
    }
  }
  float m[NG], l[NG];
  Acc<VW> acc[NV];
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    m[j] = -INFINITY;
    l[j] = 0.f;
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) acc[k].zero();
  constexpr int U = NV * VW <= 8 ? 4 : 2;
  int c[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int qe = it.b + L.e + u * E;
    c[u] = qe < it.e ? ld_stream_i32(col_idx + qe) : 0;
  }
  // one round: U edges per edge lane. Full rounds (every lane's U edges
  // exist) run without the per-edge predicates; the row's last round is TAIL.
  // (Measured on R-MAT scale 20, bf16, H = 8, D = 64: 4.48 -> 3.50 ms, the
  // same bits.)
  auto round = [&](const int p, auto tail_tag) {
    constexpr bool TAIL = decltype(tail_tag)::value;
    bool live[U];
#pragma unroll
    for (int u = 0; u < U; ++u) live[u] = TAIL ? p + u * E < it.e : true;
    Frag<T, VW> fv[U][NV];
    float s[U][NG];
    if constexpr (GIVEN) {
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int j = 0; j < NG; ++j)
          s[u][j] = live[u] ? __ldg(scores + (int64_t)(p + u * E) * es + head[j]) : -INFINITY;
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (live[u] && (ALLV || valid[k])) fv[u][k].load(V + (int64_t)c[u] * ld + (int64_t)frag[k] * VW);
    } else {
      Frag<T, VW> fk[U][NV];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (live[u] && (ALLV || valid[k])) fk[u][k].load(K + (int64_t)c[u] * ld + (int64_t)frag[k] * VW);
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (live[u] && (ALLV || valid[k])) fv[u][k].load(V + (int64_t)c[u] * ld + (int64_t)frag[k] * VW);
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int j = 0; j < NG; ++j) s[u][j] = 0.f;
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (ALLV || valid[k]) s[u][ONE ? 0 : k] += frag_dot(q[k], fk[u][k]);
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          for (int off = 1; off < R; off <<= 1) s[u][j] += __shfl_xor_sync(L.sub_mask, s[u][j], off);
          s[u][j] = live[u] ? scale * s[u][j] : -INFINITY;
        }
      }
    }
    // next iteration's columns, fetched while this iteration's rows are in flight
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int qe = p + U * E + u * E;
      c[u] = qe < it.e ? ld_stream_i32(col_idx + qe) : 0;
    }
    // online softmax per head group, with a lazily moved reference maximum
    float w[U][NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      float mx = s[0][j];
#pragma unroll
      for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[u][j]);
      if (mx > m[j] + kRescale) {  // m[j] = -inf: the first finite score sets the reference
        const float corr = __expf(m[j] - mx);
        l[j] *= corr;
#pragma unroll
        for (int k = 0; k < NV; ++k)
          if (ONE || k == j) acc[k].scale(corr);
        m[j] = mx;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        w[u][j] = (live[u] && m[j] != -INFINITY) ? __expf(s[u][j] - m[j]) : 0.f;
        l[j] += w[u][j];
      }
    }
    // rows of edges that are not live were never loaded: skip them (0 * garbage may be NaN)
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (ALLV || valid[k])
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (live[u]) acc[k].fma(w[u][ONE ? 0 : k], fv[u][k]);
  };
  int p = it.b + L.e;
  for (; p + (U - 1) * E < it.e; p += U * E) round(p, std::false_type{});
  if (p < it.e) round(p, std::true_type{});
  // merge the E edge-lane states (fixed xor order)
  for (int off = G; off < L.GE; off <<= 1) {
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const float mo = __shfl_xor_sync(L.group_mask, m[j], off);
      const float lo = __shfl_xor_sync(L.group_mask, l[j], off);
      const float mx = fmaxf(m[j], mo);
      const float a = mx == -INFINITY ? 0.f : __expf(m[j] - mx);
      const float b = mx == -INFINITY ? 0.f : __expf(mo - mx);
      l[j] = l[j] * a + lo * b;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (!(ONE || k == j)) continue;
#pragma unroll
        for (int v = 0; v < VW; ++v) {
          const float ao = __shfl_xor_sync(L.group_mask, acc[k].get(v), off);
          acc[k].set(v, acc[k].get(v) * a + ao * b);
        }
      }
      m[j] = mx;
    }
  }
  if (!it.active || L.e != 0) continue;
  if (it.chunk < 0) {
    T *o = O + it.row * ld;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (!valid[k]) continue;
      const float lk = l[ONE ? 0 : k];
      const float inv = lk > 0.f ? 1.f / lk : 0.f;
      float r[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) r[v] = acc[k].get(v) * inv;
      store_frag<T, VW>(o + (int64_t)frag[k] * VW, r);
    }
  } else {
    float *pa = part_acc + (int64_t)it.chunk * nfrag * VW;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (!valid[k]) continue;
      float r[VW];
#pragma unroll
      for (int v = 0; v < VW; ++v) r[v] = acc[k].get(v);
      store_partial<VW>(pa + (int64_t)frag[k] * VW, r);
      if (frag[k] % cph == 0) {
        const int h = H > 1 ? frag[k] / cph : 0;
        float *pm = part_ml + ((int64_t)it.chunk * H + h) * 2;
        __stcg(pm, m[ONE ? 0 : k]);
        __stcg(pm + 1, l[ONE ? 0 : k]);
      }
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
                         const T *V, int64_t ld, float scale, T *O, const ChunkList &cl_in,
                         float *part_acc, float *part_ml, cudaStream_t s) {
  const Deal dl = deal_items(cl_in, n_rows, g.G * g.E, g.G);
  const ChunkList &cl = dl.cl;
  const int ipb = dl.ipb;
  const int64_t grid = dl.grid;
  if (grid > 0) {
#define AUTOSAGE_ATTN2(NVV, GIV, ONEG, AV)                                                          \
  attention_kernel<T, VW, NVV, GIV, ONEG, AV><<<(unsigned)grid, kBlock, 0, s>>>(                   \
      n_rows, row_ptr, col_idx, Q, K, scores, V, ld, scale, g.H, g.es, g.cph, g.R, g.nfrag, g.G,     \
      g.E, g.fs, g.ks, O, cl, ipb, part_acc, part_ml)
#define AUTOSAGE_ATTN(NVV, GIV, ONEG)                                           \
  do {                                                                          \
    if (g.nfrag == g.G * (NVV)) AUTOSAGE_ATTN2(NVV, GIV, ONEG, true);          \
    else AUTOSAGE_ATTN2(NVV, GIV, ONEG, false);                                 \
  } while (0)
#define AUTOSAGE_ATTN_NV(NVV)                     \
  if (scores) AUTOSAGE_ATTN(NVV, true, true);     \
  else if (g.one) AUTOSAGE_ATTN(NVV, false, true); \
  else AUTOSAGE_ATTN(NVV, false, false);
    if (scores && !g.one) return cudaErrorInvalidValue;
    switch (g.NV) {
      case 1: AUTOSAGE_ATTN_NV(1); break;
      case 2: AUTOSAGE_ATTN_NV(2); break;
      case 4: AUTOSAGE_ATTN_NV(4); break;
      case 8: AUTOSAGE_ATTN_NV(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef AUTOSAGE_ATTN_NV
#undef AUTOSAGE_ATTN
#undef AUTOSAGE_ATTN2
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
