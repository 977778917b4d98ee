// Row softmax of edge scores, in place: W[p,h] = exp(S[p,h] - m) / l with
// m the row maximum and l = sum_q exp(S[q,h] - m) (AutoSAGE, Abstract:
// "row-softmax"; benchmark page "fused sparse attention-value aggregation":
// the maximum is subtracted for numerical stability). S is [nnz, H].
//
// A row's scores are the contiguous range [b*H, e*H). A group of GS lanes
// walks it with stride GS; when H divides GS every lane keeps one head, so a
// single read pass keeps a running (max, sum) pair per lane (the sum is
// rescaled when the max grows), pairs are merged across the lanes of a head
// by xor shuffles, and a second pass writes the weights. Rows longer than
// `split` edges are cut into chunks: chunks write (max, sum) partials, a
// fix-up merges each row's partials in chunk order, and a last pass
// normalises the chunks.
#include "internal.h"

namespace autosage {

namespace {

struct ML {
  float m, l;
};

__device__ __forceinline__ void ml_add(ML &a, float s) {
  if (s > a.m) {
    a.l = a.l * __expf(a.m - s);  // a.m = -inf gives exp(-inf) = 0
    a.m = s;
  }
  a.l += __expf(s - a.m);
}

__device__ __forceinline__ ML ml_merge(ML a, ML b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return ML{m, 0.f};
  return ML{m, a.l * __expf(a.m - m) + b.l * __expf(b.m - m)};
}

// One group of GS lanes per row or chunk; H divides GS.
__global__ void __launch_bounds__(kBlock) softmax_rows_kernel(int64_t n_rows,
                                                              const int32_t *__restrict__ row_ptr,
                                                              int H, int GS, float *__restrict__ S,
                                                              ChunkList cl, int ipb,
                                                              float *__restrict__ ml_out) {
  const Lanes L(GS, 1);
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
  const Item it = item_at(idx, n_rows, row_ptr, cl);
  const int64_t i0 = (int64_t)it.b * H, i1 = (int64_t)it.e * H;
  ML a{-INFINITY, 0.f};
  // four scores a lane in flight at a time, taken in the lane's order (the
  // same bits as one at a time; unfused attention on R-MAT scale 20, bf16,
  // H = 8, D = 64: 5.80 -> 5.63 ms)
  for (int64_t i = i0 + L.g; i < i1; i += 4 * GS) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = i + u * GS < i1 ? S[i + u * GS] : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * GS < i1) ml_add(a, x[u]);
  }
  for (int off = H; off < GS; off <<= 1) {
    ML b{__shfl_xor_sync(L.group_mask, a.m, off), __shfl_xor_sync(L.group_mask, a.l, off)};
    a = ml_merge(a, b);
  }
  if (!it.active) continue;
  if (it.chunk >= 0) {
    if (L.g < H) {
      float *o = ml_out + ((int64_t)it.chunk * H + L.g) * 2;
      o[0] = a.m;
      o[1] = a.l;
    }
    continue;
  }
  const float inv = a.l > 0.f ? 1.f / a.l : 0.f;
  for (int64_t i = i0 + L.g; i < i1; i += 4 * GS) {
    float x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) x[u] = i + u * GS < i1 ? S[i + u * GS] : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i + u * GS < i1) S[i + u * GS] = __expf(x[u] - a.m) * inv;
  }
  }
}

// Generic head count: one group per row, heads handled one after another.
__global__ void __launch_bounds__(kBlock) softmax_rows_generic_kernel(
    int64_t n_rows, const int32_t *__restrict__ row_ptr, int H, int GS, float *__restrict__ S,
    ChunkList cl, int ipb, float *__restrict__ ml_out) {
  const Lanes L(GS, 1);
  __shared__ int s_items;
  const ItemQueue queue(n_rows, cl, ipb, &s_items);
  int64_t idx;
  while (queue.next(L, idx)) {
  const Item it = item_at(idx, n_rows, row_ptr, cl);
  for (int h = 0; h < H; ++h) {
    ML a{-INFINITY, 0.f};
    for (int64_t p = it.b + L.g; p < it.e; p += GS) ml_add(a, S[p * H + h]);
    for (int off = 1; off < GS; off <<= 1) {
      ML b{__shfl_xor_sync(L.group_mask, a.m, off), __shfl_xor_sync(L.group_mask, a.l, off)};
      a = ml_merge(a, b);
    }
    if (!it.active) continue;
    if (it.chunk >= 0) {
      if (L.g == 0) {
        float *o = ml_out + ((int64_t)it.chunk * H + h) * 2;
        o[0] = a.m;
        o[1] = a.l;
      }
      continue;
    }
    const float inv = a.l > 0.f ? 1.f / a.l : 0.f;
    for (int64_t p = it.b + L.g; p < it.e; p += GS) S[p * H + h] = __expf(S[p * H + h] - a.m) * inv;
  }
  }
}

// Merge the chunk partials of each cut row (thread per (row, head)), in chunk order.
__global__ void softmax_merge_kernel(ChunkList cl, int H, const float *__restrict__ ml,
                                     float *__restrict__ row_ml) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= (int64_t)cl.n_long * H) return;
  const int64_t j = t / H;
  const int h = static_cast<int>(t % H);
  ML a{-INFINITY, 0.f};
  for (int c = cl.long_ptr[j]; c < cl.long_ptr[j + 1]; ++c) {
    const float *x = ml + ((int64_t)c * H + h) * 2;
    a = ml_merge(a, ML{x[0], x[1]});
  }
  row_ml[t * 2] = a.m;
  row_ml[t * 2 + 1] = a.l;
}

// Normalise the chunks of cut rows: one warp per chunk.
__global__ void __launch_bounds__(kBlock) softmax_normalize_chunks_kernel(
    const int32_t *__restrict__ row_ptr, ChunkList cl, int H, const float *__restrict__ row_ml,
    const int32_t *__restrict__ chunk_long, float *__restrict__ S) {
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
    const float m = row_ml[(j * H + h) * 2], l = row_ml[(j * H + h) * 2 + 1];
    S[i] = __expf(S[i] - m) * (l > 0.f ? 1.f / l : 0.f);
  }
}

// Map each chunk to its cut row (the inverse of long_ptr).
__global__ void chunk_owner_kernel(ChunkList cl, int32_t *__restrict__ chunk_long) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= cl.n_long) return;
  for (int c = cl.long_ptr[j]; c < cl.long_ptr[j + 1]; ++c) chunk_long[c] = static_cast<int32_t>(j);
}

}  // namespace

cudaError_t launch_row_softmax(int64_t n_rows, const int32_t *row_ptr, int H, float *S,
                               const ChunkList &cl_in, float *ml, float *row_ml, cudaStream_t s) {
  // group size: a power of two that H divides when possible, else a full warp
  int GS = 32;
  const bool divides = (32 % H) == 0;
  if (divides) {
    GS = H < 8 ? 8 : H;
  }
  const Deal dl = deal_items(cl_in, n_rows, GS, 1);
  const ChunkList &cl = dl.cl;
  const int ipb = dl.ipb;
  const int64_t grid = dl.grid;
  if (grid > 0) {
    if (divides)
      softmax_rows_kernel<<<(unsigned)grid, kBlock, 0, s>>>(n_rows, row_ptr, H, GS, S, cl, ipb, ml);
    else
      softmax_rows_generic_kernel<<<(unsigned)grid, kBlock, 0, s>>>(n_rows, row_ptr, H, GS, S, cl, ipb, ml);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  if (cl.n_long > 0) {
    const int64_t nt = (int64_t)cl.n_long * H;
    softmax_merge_kernel<<<(unsigned)((nt + 255) / 256), 256, 0, s>>>(cl, H, ml, row_ml);
    // chunk -> cut-row map lives after the (max, sum) partials in `ml`
    int32_t *chunk_long = reinterpret_cast<int32_t *>(ml + (int64_t)cl.n_chunks * H * 2);
    chunk_owner_kernel<<<(unsigned)((cl.n_long + 255) / 256), 256, 0, s>>>(cl, chunk_long);
    softmax_normalize_chunks_kernel<<<(unsigned)((cl.n_chunks + 7) / 8), kBlock, 0, s>>>(
        row_ptr, cl, H, row_ml, chunk_long, S);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace autosage
