// Kernels of the CSR-attention backward that the forward kernels do not
// cover: the softmax backward and the reordering of per-edge arrays into the
// edge order of A^T.
//
// With w the row-softmax weights and dW_p = <dO_i, V_j> (an SDDMM), the
// softmax backward is dS_p = w_p (dW_p - D_i) with D_i = sum_p w_p dW_p, for
// every row i and head (the chain rule through the softmax; the same
// identity the oracle states). Rows longer than `split` edges are cut into
// chunks: chunks write partial sums of w dW, a merge adds each cut row's
// partials in chunk order, and a last pass writes the chunks' dS. The scale of
// the scores is folded into dS, because both dQ and dK carry it.
#include "internal.h"

namespace autosage {

namespace {

// One group of GS lanes per row or chunk; H divides GS, lane g keeps head g % H.
__global__ void __launch_bounds__(kBlock) softmax_bwd_rows_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, int H, int GS, const float *__restrict__ W,
    float *__restrict__ dS, float scale, ChunkList cl, int ipb, float *__restrict__ part) {
  const Lanes L(GS, 1);
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
    const Item it = item_at(idx, n_rows, row_ptr, cl);
    const int64_t i0 = (int64_t)it.b * H, i1 = (int64_t)it.e * H;
    float d = 0.f;
    for (int64_t i = i0 + L.g; i < i1; i += GS) d = fmaf(W[i], dS[i], d);
    for (int off = H; off < GS; off <<= 1) d += __shfl_xor_sync(L.group_mask, d, off);
    if (!it.active) continue;
    if (it.chunk >= 0) {
      if (L.g < H) part[(int64_t)it.chunk * H + L.g] = d;
      continue;
    }
    for (int64_t i = i0 + L.g; i < i1; i += GS) dS[i] = scale * W[i] * (dS[i] - d);
  }
}

// Any head count: heads one after another, lanes over the row's edges.
__global__ void __launch_bounds__(kBlock) softmax_bwd_rows_generic_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, int H, int GS, const float *__restrict__ W,
    float *__restrict__ dS, float scale, ChunkList cl, int ipb, float *__restrict__ part) {
  const Lanes L(GS, 1);
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
    const Item it = item_at(idx, n_rows, row_ptr, cl);
    for (int h = 0; h < H; ++h) {
      float d = 0.f;
      for (int64_t p = it.b + L.g; p < it.e; p += GS) d = fmaf(W[p * H + h], dS[p * H + h], d);
      for (int off = 1; off < GS; off <<= 1) d += __shfl_xor_sync(L.group_mask, d, off);
      if (!it.active) continue;
      if (it.chunk >= 0) {
        if (L.g == 0) part[(int64_t)it.chunk * H + h] = d;
        continue;
      }
      for (int64_t p = it.b + L.g; p < it.e; p += GS) dS[p * H + h] = scale * W[p * H + h] * (dS[p * H + h] - d);
    }
  }
}

// D of each cut row and head: its chunks' partial sums in chunk order.
__global__ void softmax_bwd_merge_kernel(ChunkList cl, int H, const float *__restrict__ part,
                                         float *__restrict__ row_d, int32_t *__restrict__ chunk_long) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)cl.n_long * H) return;
  const int64_t j = t / H;
  const int h = static_cast<int>(t % H);
  float d = 0.f;
  for (int c = cl.long_ptr[j]; c < cl.long_ptr[j + 1]; ++c) {
    d += part[(int64_t)c * H + h];
    if (h == 0) chunk_long[c] = static_cast<int32_t>(j);
  }
  row_d[t] = d;
}

// dS of the chunks of cut rows: one warp per chunk.
__global__ void __launch_bounds__(kBlock) softmax_bwd_chunks_kernel(
    const int32_t *__restrict__ row_ptr, ChunkList cl, int H, const float *__restrict__ W,
    float *__restrict__ dS, float scale, const float *__restrict__ row_d,
    const int32_t *__restrict__ chunk_long) {
  const int64_t c = (int64_t)blockIdx.x * (kBlock / 32) + (threadIdx.x >> 5);
  if (c >= cl.n_chunks) return;
  const int lane = threadIdx.x & 31;
  const int64_t row = cl.chunk_row[c];
  const int b = cl.chunk_begin[c];
  const int re = row_ptr[row + 1];
  const int e = (re - b > cl.split) ? b + cl.split : re;
  const int64_t j = chunk_long[c];
  for (int64_t i = (int64_t)b * H + lane; i < (int64_t)e * H; i += 32) {
    const int h = static_cast<int>(i % H);
    dS[i] = scale * W[i] * (dS[i] - row_d[j * H + h]);
  }
}

// out_a[k, :] = a[perm[k], :] and out_b[k, :] = b[perm[k], :] for rows of H floats.
__global__ void permute_edges_kernel(int64_t nnz, int H, const int32_t *__restrict__ perm,
                                     const float *__restrict__ a, const float *__restrict__ b,
                                     float *__restrict__ out_a, float *__restrict__ out_b) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t total = nnz * H;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += stride) {
    const int64_t k = t / H;
    const int h = static_cast<int>(t - k * H);
    const int64_t src = (int64_t)__ldg(perm + k) * H + h;
    out_a[t] = __ldg(a + src);
    out_b[t] = __ldg(b + src);
  }
}

}  // namespace

cudaError_t launch_softmax_backward(int64_t n_rows, const int32_t *row_ptr, int H, const float *W, float *dS,
                                    float scale, const ChunkList &cl, float *part, float *row_d,
                                    cudaStream_t s) {
  const bool divides = (32 % H) == 0;
  const int GS = 32;
  const int ipb = items_per_block_for(GS, 1);
  const int64_t grid = (cl.n_chunks + n_rows + ipb - 1) / ipb;
  if (grid > 0) {
    if (divides)
      softmax_bwd_rows_kernel<<<(unsigned)grid, kBlock, 0, s>>>(n_rows, row_ptr, H, GS, W, dS, scale, cl, ipb, part);
    else
      softmax_bwd_rows_generic_kernel<<<(unsigned)grid, kBlock, 0, s>>>(n_rows, row_ptr, H, GS, W, dS, scale, cl,
                                                                         ipb, part);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cl.n_long > 0) {
    // chunk -> cut-row map lives after the partial sums in `part`
    int32_t *chunk_long = reinterpret_cast<int32_t *>(part + (int64_t)cl.n_chunks * H);
    const int64_t nt = (int64_t)cl.n_long * H;
    softmax_bwd_merge_kernel<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(cl, H, part, row_d, chunk_long);
    softmax_bwd_chunks_kernel<<<(unsigned)((cl.n_chunks + 7) / 8), kBlock, 0, s>>>(row_ptr, cl, H, W, dS, scale,
                                                                                  row_d, chunk_long);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

cudaError_t launch_permute_edges(int64_t nnz, int H, const int32_t *perm, const float *a, const float *b,
                                 float *out_a, float *out_b, cudaStream_t s) {
  if (nnz <= 0) return cudaSuccess;
  const int64_t total = nnz * H;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  permute_edges_kernel<<<(unsigned)blocks, 256, 0, s>>>(nnz, H, perm, a, b, out_a, out_b);
  return cudaGetLastError();
}

}  // namespace autosage
