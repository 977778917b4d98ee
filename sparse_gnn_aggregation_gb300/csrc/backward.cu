// CSR-attention backward, forward direction in one pass per row.
//
// The forward pipeline (AutoSAGE, "Input-Aware CUDA Scheduling for Sparse
// GNN Aggregation (SpMM/SDDMM) and CSR Attention", Abstract: SDDMM ->
// row-softmax -> SpMM) computes, per row i, head h and edge p = (i, j):
//   s_p = scale <q_i, k_j>,  w_p = exp(s_p - m_i) / l_i,  o_i = sum_p w_p v_j.
// Its gradients follow from the chain rule (the identities the oracle states):
//   dW_p = <do_i, v_j>,  D_i = sum_p w_p dW_p,  dS_p = w_p (dW_p - D_i),
//   dQ_i = scale sum_p dS_p k_j,  dK_j = scale sum_{p into j} dS_p q_i,
//   dV_j = sum_{p into j} w_p do_i.
// dK and dV run over the edges of A^T (an SpMM over the transposed pattern).
// Everything that runs over the edges of A -- the scores, the softmax, dW,
// D, dS and dQ -- is one kernel here: a lane group owns a row, gathers k_j
// and v_j once per edge, and keeps an online softmax state per head
// (reference maximum m, l = sum e_p, sum e_p dW_p, and the feature vectors
// A = sum e_p dW_p k_j and B = sum e_p k_j, with e_p = exp(s_p - m)). At the
// row's end D = sum e dW / l and dQ = scale (A - D B) / l, which equals the
// sum above without a second gather of K. A second walk over the row's own
// edges (no gathers: the scores and dW it wrote are re-read) writes w_p and
// scale * dS_p straight into the edge order of A^T for the dK / dV SpMMs.
// Rows longer than `split` edges are cut into chunks that write their state;
// a fix-up merges each cut row's chunks in chunk order (fixed order: repeat
// runs give identical bits) and a last pass writes the chunks' w and dS.
#include <type_traits>

#include "internal.h"

namespace autosage {

namespace {

// Same lazy rescale as the forward kernel: the reference maximum moves only
// when a score exceeds it by more than kRescale, so exp(s - m) < e^kRescale.
constexpr float kRescaleB = 8.f;

// Edges in flight per edge lane: two while a lane's Q and dO fragments take
// less than 32 bytes each, else one.
template <typename T, int VW, int NV>
__host__ __device__ constexpr int bwd_unroll() {
  return NV * VW * (int)sizeof(T) < 32 ? 2 : 1;
}

// Blocks per SM the register budget is sized for: lanes holding at most 32
// bytes of a row fit three 256-thread blocks (85 registers), wider ones two.
// The pass is bound by memory latency, so occupancy wins over edges in
// flight per lane (measured on R-MAT scale 20, bf16, H = 8, D = 64: three
// blocks with one edge in flight 12.0 ms against two blocks with two edges
// 12.5 ms).
template <typename T, int VW, int NV>
constexpr int bwd_min_blocks() {
  return NV * VW * (int)sizeof(T) <= 32 ? 3 : 2;
}

// Per-chunk state layout in `part`: [n_chunks][2][width] for (A, B), then
// [n_chunks][H][3] for (m, l, sum e dW), then [n_chunks] cut-row indices.
struct BwdPart {
  float *acc;
  float *st;
  int32_t *chunk_long;
};

__device__ __forceinline__ BwdPart bwd_part(float *part, int64_t n_chunks, int64_t width, int H) {
  BwdPart b;
  b.acc = part;
  b.st = part + n_chunks * 2 * width;
  b.chunk_long = reinterpret_cast<int32_t *>(b.st + n_chunks * H * 3);
  return b;
}

// Fragment slot k of lane g is fragment g * fs + k * ks (as in the forward
// kernel). ONE: all slots of a lane lie in one head; otherwise slot k is its
// own head. R lanes share a head; the first of them (g % R == 0) writes that
// head's per-edge values. ALLV: every slot of every lane holds a fragment.
// The edges run in rounds of U per edge lane; full rounds skip the per-edge
// predicates (measured on R-MAT scale 20, bf16, H = 8, D = 64: 13.7 -> 12.6 ms
// for the whole backward, the same bits).
template <typename T, int VW, int NV, bool ONE, bool ALLV>
__global__ void __launch_bounds__(kBlock, bwd_min_blocks<T, VW, NV>()) attn_bwd_rows_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
    const T *__restrict__ Q, const T *__restrict__ K, const T *__restrict__ V, const T *__restrict__ dO,
    int64_t ld, float scale, int H, int es, int cph, int R, int nfrag, int G, int E, int fs, int ks,
    T *__restrict__ dQ, float *__restrict__ S, float *__restrict__ dW, const int32_t *__restrict__ inv,
    float *__restrict__ Wt, float *__restrict__ dSt, ChunkList cl, int ipb, float *__restrict__ part) {
  constexpr int NG = ONE ? 1 : NV;
  constexpr int U = bwd_unroll<T, VW, NV>();
  const Lanes L(G, E);
  const int64_t width = (int64_t)nfrag * VW;
  const BwdPart bp = bwd_part(part, cl.n_chunks, width, H);
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
    const Item it = item_at(idx, n_rows, row_ptr, cl);
    const int g = L.g;
    const bool writer = (g % R) == 0;
    bool valid[NV];
    int frag[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      frag[k] = g * fs + k * ks;
      valid[k] = frag[k] < nfrag;
    }
    int head[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) head[j] = (H > 1 && valid[j]) ? frag[j] / cph : 0;
    Frag<T, VW> q[NV], go[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (it.e > it.b && valid[k]) {
        q[k].load(Q + it.row * ld + (int64_t)frag[k] * VW);
        go[k].load(dO + it.row * ld + (int64_t)frag[k] * VW);
      } else {
        q[k].zero();
        go[k].zero();
      }
    }
    float m[NG], l[NG], sw[NG];
    Acc<VW> a[NV], b[NV];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
      sw[j] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      a[k].zero();
      b[k].zero();
    }
    int c[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int qe = it.b + L.e + u * E;
      c[u] = qe < it.e ? ld_stream_i32(col_idx + qe) : 0;
    }
    // one round: U edges per edge lane; full rounds run without the per-edge
    // predicates, the row's last round is TAIL
    auto round = [&](const int p, auto tail_tag) {
      constexpr bool TAIL = decltype(tail_tag)::value;
      bool live[U];
#pragma unroll
      for (int u = 0; u < U; ++u) live[u] = TAIL ? p + u * E < it.e : true;
      Frag<T, VW> fk[U][NV], fv[U][NV];
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
      // next iteration's columns, fetched while this iteration's rows are in flight
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int qe = p + U * E + u * E;
        c[u] = qe < it.e ? ld_stream_i32(col_idx + qe) : 0;
      }
      // scores s and dW per edge and head group, finished over the R lanes of a head
      float s[U][NG], dw[U][NG];
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          s[u][j] = 0.f;
          dw[u][j] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          if (live[u] && (ALLV || valid[k])) {
            s[u][ONE ? 0 : k] += frag_dot(q[k], fk[u][k]);
            dw[u][ONE ? 0 : k] += frag_dot(go[k], fv[u][k]);
          }
        }
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          for (int off = 1; off < R; off <<= 1) {
            s[u][j] += __shfl_xor_sync(L.sub_mask, s[u][j], off);
            dw[u][j] += __shfl_xor_sync(L.sub_mask, dw[u][j], off);
          }
          s[u][j] = live[u] ? scale * s[u][j] : -INFINITY;
        }
      }
      // the scores and dW of this edge lane's edges, for the second walk
      if (writer) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (live[u])
#pragma unroll
            for (int j = 0; j < NG; ++j)
              if (ALLV || valid[j]) {
                const int64_t i = (int64_t)(p + u * E) * es + head[j];
                S[i] = s[u][j];
                dW[i] = dw[u][j];
              }
      }
      // online softmax state per head group
      float ew[U][NG];
#pragma unroll
      for (int j = 0; j < NG; ++j) {
        float mx = s[0][j];
#pragma unroll
        for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[u][j]);
        if (mx > m[j] + kRescaleB) {  // m[j] = -inf: the first finite score sets the reference
          const float corr = __expf(m[j] - mx);
          l[j] *= corr;
          sw[j] *= corr;
#pragma unroll
          for (int k = 0; k < NV; ++k)
            if (ONE || k == j) {
              a[k].scale(corr);
              b[k].scale(corr);
            }
          m[j] = mx;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          ew[u][j] = (live[u] && m[j] != -INFINITY) ? __expf(s[u][j] - m[j]) : 0.f;
          l[j] += ew[u][j];
          sw[j] = fmaf(ew[u][j], dw[u][j], sw[j]);
        }
      }
      // K rows of edges that are not live were never loaded: skip them
#pragma unroll
      for (int k = 0; k < NV; ++k)
        if (ALLV || valid[k])
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (live[u]) {
              const float e1 = ew[u][ONE ? 0 : k];
              a[k].fma(e1 * dw[u][ONE ? 0 : k], fk[u][k]);
              b[k].fma(e1, fk[u][k]);
            }
    };
    int p = it.b + L.e;
    for (; p + (U - 1) * E < it.e; p += U * E) round(p, std::false_type{});
    if (p < it.e) round(p, std::true_type{});
    // merge the E edge-lane states (fixed xor order); every lane ends with the group's state
    for (int off = G; off < L.GE; off <<= 1) {
#pragma unroll
      for (int j = 0; j < NG; ++j) {
        const float mo = __shfl_xor_sync(L.group_mask, m[j], off);
        const float lo = __shfl_xor_sync(L.group_mask, l[j], off);
        const float so = __shfl_xor_sync(L.group_mask, sw[j], off);
        const float mx = fmaxf(m[j], mo);
        const float fa = mx == -INFINITY ? 0.f : __expf(m[j] - mx);
        const float fb = mx == -INFINITY ? 0.f : __expf(mo - mx);
        l[j] = l[j] * fa + lo * fb;
        sw[j] = sw[j] * fa + so * fb;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          if (!(ONE || k == j)) continue;
#pragma unroll
          for (int v = 0; v < VW; ++v) {
            const float ao = __shfl_xor_sync(L.group_mask, a[k].get(v), off);
            const float bo = __shfl_xor_sync(L.group_mask, b[k].get(v), off);
            a[k].set(v, a[k].get(v) * fa + ao * fb);
            b[k].set(v, b[k].get(v) * fa + bo * fb);
          }
        }
        m[j] = mx;
      }
    }
    if (!it.active) continue;
    if (it.chunk >= 0) {
      // a chunk of a cut row: its state goes to the fix-up
      if (L.e != 0) continue;
      float *pa = bp.acc + (int64_t)it.chunk * 2 * width;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (!valid[k]) continue;
        float ra[VW], rb[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) {
          ra[v] = a[k].get(v);
          rb[v] = b[k].get(v);
        }
        store_partial<VW>(pa + (int64_t)frag[k] * VW, ra);
        store_partial<VW>(pa + width + (int64_t)frag[k] * VW, rb);
      }
      if (writer) {
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          if (!valid[j]) continue;
          float *ps = bp.st + ((int64_t)it.chunk * H + head[j]) * 3;
          __stcg(ps, m[j]);
          __stcg(ps + 1, l[j]);
          __stcg(ps + 2, sw[j]);
        }
      }
      continue;
    }
    // a whole row: D, dQ, then w and dS of its edges in the edge order of A^T
    float dd[NG], il[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      il[j] = l[j] > 0.f ? 1.f / l[j] : 0.f;
      dd[j] = sw[j] * il[j];
    }
    if (L.e == 0) {
      T *o = dQ + it.row * ld;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (!valid[k]) continue;
        const int j = ONE ? 0 : k;
        float r[VW];
#pragma unroll
        for (int v = 0; v < VW; ++v) r[v] = scale * (a[k].get(v) - dd[j] * b[k].get(v)) * il[j];
        store_frag<T, VW>(o + (int64_t)frag[k] * VW, r);
      }
    }
    {
      // the R lanes of a head share the row's edges (lane g % R takes every
      // R-th one); the head's first lane wrote their scores and dW above, and
      // the warp sync makes those writes visible to the others (measured on
      // R-MAT scale 20, bf16, H = 8, D = 64: 11.63 -> 10.94 ms for the whole
      // backward against the first lane alone, the same bits)
      __syncwarp(L.group_mask);
      for (int p = it.b + L.e + (g % R) * E; p < it.e; p += E * R) {
        const int64_t t = inv[p];
#pragma unroll
        for (int j = 0; j < NG; ++j) {
          if (!valid[j]) continue;
          const int64_t i = (int64_t)p * es + head[j];
          const float w = __expf(S[i] - m[j]) * il[j];
          __stcs(Wt + t * es + head[j], w);
          __stcs(dSt + t * es + head[j], scale * w * (dW[i] - dd[j]));
        }
      }
    }
  }
}

// One warp per cut row: merge its chunks' states in chunk order, write dQ
// and the row's (m, l, D) per head, and map each chunk to its cut row.
template <typename T, int VW>
__global__ void __launch_bounds__(kBlock) attn_bwd_fixup_kernel(ChunkList cl, int H, int cph, int nfrag,
                                                                float scale, float *__restrict__ part,
                                                                float *__restrict__ row_st, T *__restrict__ dQ,
                                                                int64_t ld) {
  const int64_t j = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (j >= cl.n_long) return;
  const int lane = threadIdx.x & 31;
  const int64_t width = (int64_t)nfrag * VW;
  const BwdPart bp = bwd_part(part, cl.n_chunks, width, H);
  const int64_t row = cl.long_rows[j];
  const int c0 = cl.long_ptr[j], c1 = cl.long_ptr[j + 1];
  for (int c = c0 + lane; c < c1; c += 32) bp.chunk_long[c] = static_cast<int32_t>(j);
  for (int f = lane; f < nfrag; f += 32) {
    const int h = f / cph;
    float m = -INFINITY, l = 0.f, sw = 0.f, a[VW], b[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) {
      a[v] = 0.f;
      b[v] = 0.f;
    }
    for (int c = c0; c < c1; ++c) {
      const float *ps = bp.st + ((int64_t)c * H + h) * 3;
      const float mc = __ldcg(ps), lc = __ldcg(ps + 1), sc = __ldcg(ps + 2);
      const float mx = fmaxf(m, mc);
      const float fa = mx == -INFINITY ? 0.f : __expf(m - mx);
      const float fb = mx == -INFINITY ? 0.f : __expf(mc - mx);
      l = l * fa + lc * fb;
      sw = sw * fa + sc * fb;
      const float *pa = bp.acc + (int64_t)c * 2 * width + (int64_t)f * VW;
#pragma unroll
      for (int v = 0; v < VW; ++v) {
        a[v] = a[v] * fa + __ldcg(pa + v) * fb;
        b[v] = b[v] * fa + __ldcg(pa + width + v) * fb;
      }
      m = mx;
    }
    const float il = l > 0.f ? 1.f / l : 0.f;
    const float d = sw * il;
    float r[VW];
#pragma unroll
    for (int v = 0; v < VW; ++v) r[v] = scale * (a[v] - d * b[v]) * il;
    store_frag<T, VW>(dQ + row * ld + (int64_t)f * VW, r);
    if (f % cph == 0) {
      float *rs = row_st + (j * H + h) * 3;
      rs[0] = m;
      rs[1] = il;
      rs[2] = d;
    }
  }
}

// w and dS of the chunks' edges (one warp per chunk), in the edge order of A^T.
__global__ void __launch_bounds__(kBlock) attn_bwd_chunks_kernel(
    const int32_t *__restrict__ row_ptr, ChunkList cl, int H, int es, float scale, const float *__restrict__ S,
    const float *__restrict__ dW, const int32_t *__restrict__ inv, const float *__restrict__ part,
    int64_t width, const float *__restrict__ row_st, float *__restrict__ Wt, float *__restrict__ dSt) {
  const int64_t c = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (c >= cl.n_chunks) return;
  const int lane = threadIdx.x & 31;
  const int32_t *chunk_long =
      reinterpret_cast<const int32_t *>(part + (int64_t)cl.n_chunks * 2 * width + (int64_t)cl.n_chunks * H * 3);
  const int64_t row = cl.chunk_row[c];
  const int b = cl.chunk_begin[c];
  const int re = row_ptr[row + 1];
  const int e = (re - b > cl.split) ? b + cl.split : re;
  const int64_t j = chunk_long[c];
  for (int64_t i = (int64_t)b * H + lane; i < (int64_t)e * H; i += 32) {
    const int64_t p = i / H;
    const int h = static_cast<int>(i - p * H);
    const float *rs = row_st + (j * H + h) * 3;
    const int64_t q = p * es + h;
    const float w = __expf(__ldcs(S + q) - rs[0]) * rs[1];
    const int64_t t = inv[p];
    __stcs(Wt + t * es + h, w);
    __stcs(dSt + t * es + h, scale * w * (__ldcs(dW + q) - rs[2]));
  }
}

// inv[perm[k]] = k
__global__ void invert_perm_kernel(int64_t n, const int32_t *__restrict__ perm, int32_t *__restrict__ inv) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
    inv[perm[k]] = static_cast<int32_t>(k);
}

template <typename T, int VW>
cudaError_t attn_bwd_vw(const Geom &g, int64_t n_rows, const int32_t *row_ptr, const int32_t *col_idx,
                        const T *Q, const T *K, const T *V, const T *dO, int64_t ld, int es, float scale, T *dQ,
                        float *S, float *dW, const int32_t *inv, float *Wt, float *dSt, const ChunkList &cl_in,
                        float *part, float *row_st, cudaStream_t s) {
  const Deal dl = deal_items(cl_in, n_rows, g.G * g.E, g.G);
  const ChunkList &cl = dl.cl;
  const int ipb = dl.ipb;
  const int64_t grid = dl.grid;
  if (grid > 0) {
#define AUTOSAGE_BWD(NVV, ONEG)                                                                            \
  if (g.nfrag == g.G * (NVV)) AUTOSAGE_BWD2(NVV, ONEG, true);                                              \
  else AUTOSAGE_BWD2(NVV, ONEG, false);
#define AUTOSAGE_BWD2(NVV, ONEG, AV)                                                                       \
  attn_bwd_rows_kernel<T, VW, NVV, ONEG, AV><<<(unsigned)grid, kBlock, 0, s>>>(                           \
      n_rows, row_ptr, col_idx, Q, K, V, dO, ld, scale, g.H, es, g.cph, g.R, g.nfrag, g.G, g.E, g.fs, g.ks, dQ, \
      S, dW, inv, Wt, dSt, cl, ipb, part)
#define AUTOSAGE_BWD_NV(NVV)             \
  if (g.one) { AUTOSAGE_BWD(NVV, true) } \
  else { AUTOSAGE_BWD(NVV, false) }
    switch (g.NV) {
      case 1: AUTOSAGE_BWD_NV(1); break;
      case 2: AUTOSAGE_BWD_NV(2); break;
      case 4: AUTOSAGE_BWD_NV(4); break;
      case 8: AUTOSAGE_BWD_NV(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef AUTOSAGE_BWD_NV
#undef AUTOSAGE_BWD
#undef AUTOSAGE_BWD2
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cl.n_long > 0) {
    const unsigned fgrid = (unsigned)((cl.n_long + kBlock / 32 - 1) / (kBlock / 32));
    attn_bwd_fixup_kernel<T, VW><<<fgrid, kBlock, 0, s>>>(cl, g.H, g.cph, g.nfrag, scale, part, row_st, dQ, ld);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const unsigned cgrid = (unsigned)((cl.n_chunks + kBlock / 32 - 1) / (kBlock / 32));
    attn_bwd_chunks_kernel<<<cgrid, kBlock, 0, s>>>(row_ptr, cl, g.H, es, scale, S, dW, inv, part,
                                                     (int64_t)g.nfrag * VW, row_st, Wt, dSt);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_attention_backward(const Geom &g, int64_t n_rows, const int32_t *row_ptr,
                                      const int32_t *col_idx, const void *Q, const void *K, const void *V,
                                      const void *dO, int64_t ld, int es, float scale, void *dQ, float *S,
                                      float *dW, const int32_t *inv, float *Wt, float *dSt, const ChunkList &cl,
                                      float *part, float *row_st, cudaStream_t s) {
  if (g.dt == DType::F32) {
    auto q = static_cast<const float *>(Q);
    auto k = static_cast<const float *>(K);
    auto v = static_cast<const float *>(V);
    auto go = static_cast<const float *>(dO);
    auto o = static_cast<float *>(dQ);
    switch (g.VW) {
      case 4: return attn_bwd_vw<float, 4>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
      case 2: return attn_bwd_vw<float, 2>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
      case 1: return attn_bwd_vw<float, 1>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
    }
  } else {
    auto q = static_cast<const __nv_bfloat16 *>(Q);
    auto k = static_cast<const __nv_bfloat16 *>(K);
    auto v = static_cast<const __nv_bfloat16 *>(V);
    auto go = static_cast<const __nv_bfloat16 *>(dO);
    auto o = static_cast<__nv_bfloat16 *>(dQ);
    switch (g.VW) {
      case 8: return attn_bwd_vw<__nv_bfloat16, 8>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
      case 4: return attn_bwd_vw<__nv_bfloat16, 4>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
      case 2: return attn_bwd_vw<__nv_bfloat16, 2>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
      case 1: return attn_bwd_vw<__nv_bfloat16, 1>(g, n_rows, row_ptr, col_idx, q, k, v, go, ld, es, scale, o, S, dW, inv, Wt, dSt, cl, part, row_st, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_invert_perm(int64_t n, const int32_t *perm, int32_t *inv, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  invert_perm_kernel<<<(unsigned)blocks, 256, 0, s>>>(n, perm, inv);
  return cudaGetLastError();
}

}  // namespace autosage
