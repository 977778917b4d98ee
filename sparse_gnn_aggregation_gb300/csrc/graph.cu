// Graph utilities on the GPU: row statistics for the planner, structure
// fingerprint for the plan cache, CSR validation, exclusive scan, long-row
// chunk lists, the stable CSR transpose (LSD radix sort) used by SpMM with
// A^T, and probe-buffer fill / comparison for the planner's micro-probes.
// All results are deterministic: integer atomics only, stable sorts.
#include <algorithm>

#include "internal.h"

namespace autosage {

namespace {

// ---------------------------------------------------------------- statistics

// ints: [0] n_rows (host fills), [1] sum deg, [2] max, [3] min, [4] empty,
// [5] sum deg^2, [6] rows deg > thr, [7] edges in them, [8 + b] log2 buckets.
__global__ void row_stats_kernel(int64_t n_rows, const int32_t *__restrict__ row_ptr,
                                 int64_t thr, unsigned long long *__restrict__ ints) {
  __shared__ unsigned long long sh[40];
  for (int i = threadIdx.x; i < 40; i += blockDim.x) sh[i] = (i == 3) ? ~0ull : 0ull;
  __syncthreads();
  unsigned long long sum = 0, mx = 0, mn = ~0ull, empty = 0, sq = 0, nl = 0, el = 0;
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n_rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const unsigned long long d = (unsigned long long)(row_ptr[r + 1] - row_ptr[r]);
    sum += d;
    mx = d > mx ? d : mx;
    mn = d < mn ? d : mn;
    empty += d == 0;
    sq += d * d;
    if ((int64_t)d > thr) {
      nl += 1;
      el += d;
    }
    const int b = d == 0 ? 0 : 64 - __clzll((long long)d);  // bit length
    atomicAdd(&sh[8 + (b < 31 ? b : 31)], 1ull);
  }
  atomicAdd(&sh[1], sum);
  atomicMax(&sh[2], mx);
  atomicMin(&sh[3], mn);
  atomicAdd(&sh[4], empty);
  atomicAdd(&sh[5], sq);
  atomicAdd(&sh[6], nl);
  atomicAdd(&sh[7], el);
  __syncthreads();
  for (int i = threadIdx.x; i < 40; i += blockDim.x) {
    if (i == 0) continue;
    if (i == 2)
      atomicMax(&ints[i], sh[i]);
    else if (i == 3)
      atomicMin(&ints[i], sh[i]);
    else if (sh[i])
      atomicAdd(&ints[i], sh[i]);
  }
}

// ---------------------------------------------------------------- fingerprint

__device__ __forceinline__ unsigned long long splitmix64_mix(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fingerprint_kernel(int64_t n_rows, int64_t nnz, const int32_t *__restrict__ row_ptr,
                                   const int32_t *__restrict__ col_idx,
                                   unsigned long long *__restrict__ out) {
  const unsigned long long tag_rows = 0x9E3779B97F4A7C15ull, tag_cols = 0xD1B54A32D192ED03ull;
  unsigned long long h = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= n_rows; i += stride)
    h += splitmix64_mix(tag_rows ^ ((unsigned long long)i << 32) ^ (uint32_t)row_ptr[i]);
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < nnz; p += stride)
    h += splitmix64_mix(tag_cols ^ ((unsigned long long)p << 32) ^ (uint32_t)col_idx[p]);
  for (int off = 16; off > 0; off >>= 1) h += __shfl_xor_sync(FULL, h, off);
  if ((threadIdx.x & 31) == 0) atomicAdd(out, h);
}

// ---------------------------------------------------------------- validation

__global__ void validate_kernel(int64_t n_rows, int64_t n_cols, int64_t nnz,
                                const int32_t *__restrict__ row_ptr,
                                const int32_t *__restrict__ col_idx, int *__restrict__ err) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t0 == 0) {
    if (row_ptr[0] != 0) atomicOr(err, 1);
    if ((int64_t)row_ptr[n_rows] != nnz) atomicOr(err, 4);
  }
  for (int64_t r = t0; r < n_rows; r += stride)
    if (row_ptr[r + 1] < row_ptr[r]) atomicOr(err, 2);
  for (int64_t p = t0; p < nnz; p += stride) {
    const int32_t c = col_idx[p];
    if (c < 0 || (int64_t)c >= n_cols) atomicOr(err, 8);
  }
}

// ---------------------------------------------------------------- scan

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;

// Exclusive scan of one value per thread across the block; returns the block total.
__device__ __forceinline__ int block_exclusive_scan(int v, int &total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(FULL, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(FULL, s, off);
      if (lane >= off) s += y;
    }
    warp_sums[lane] = s;  // inclusive prefix of warp totals
  }
  __syncthreads();
  total = warp_sums[(blockDim.x >> 5) - 1];
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kScanThreads) scan_tile_sums_kernel(const int32_t *__restrict__ in,
                                                                      int64_t n,
                                                                      int32_t *__restrict__ sums) {
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  int v = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) v += in[base + i];
  int total;
  block_exclusive_scan(v, total);
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// Single block: exclusive scan of the tile sums in place, in pieces of kScanThreads.
__global__ void __launch_bounds__(kScanThreads) scan_sums_kernel(int32_t *__restrict__ sums,
                                                                 int64_t n_tiles) {
  int carry = 0;
  for (int64_t base = 0; base < n_tiles; base += kScanThreads) {
    const int64_t i = base + threadIdx.x;
    const int v = i < n_tiles ? sums[i] : 0;
    int total;
    const int ex = block_exclusive_scan(v, total);
    if (i < n_tiles) sums[i] = carry + ex;
    carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) sums[n_tiles] = carry;
}

__global__ void __launch_bounds__(kScanThreads) scan_apply_kernel(const int32_t *__restrict__ in,
                                                                  int64_t n,
                                                                  const int32_t *__restrict__ sums,
                                                                  int64_t n_tiles,
                                                                  int32_t *__restrict__ out) {
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  int x[kScanItems];
  int v = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    x[i] = base + i < n ? in[base + i] : 0;
    v += x[i];
  }
  int total;
  int run = block_exclusive_scan(v, total) + sums[blockIdx.x];
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if (base + i < n) out[base + i] = run;
    run += x[i];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) out[n] = sums[n_tiles];
}

// ---------------------------------------------------------------- chunk lists

__global__ void long_flags_kernel(int64_t n_rows, const int32_t *__restrict__ row_ptr, int split,
                                  int32_t *__restrict__ flags) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r < n_rows) flags[r] = (row_ptr[r + 1] - row_ptr[r]) > split ? 1 : 0;
}

__global__ void long_compact_kernel(int64_t n_rows, const int32_t *__restrict__ row_ptr, int split,
                                    const int32_t *__restrict__ pos, int32_t *__restrict__ long_rows,
                                    int32_t *__restrict__ counts) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  const int d = row_ptr[r + 1] - row_ptr[r];
  if (d > split) {
    const int j = pos[r];
    long_rows[j] = static_cast<int32_t>(r);
    counts[j] = (d + split - 1) / split;
  }
}

__global__ void chunk_fill_kernel(int64_t n_long, const int32_t *__restrict__ row_ptr, int split,
                                  const int32_t *__restrict__ long_rows,
                                  const int32_t *__restrict__ long_ptr,
                                  int32_t *__restrict__ chunk_row, int32_t *__restrict__ chunk_begin) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= n_long) return;
  const int r = long_rows[j];
  const int b = row_ptr[r];
  for (int c = long_ptr[j], t = 0; c < long_ptr[j + 1]; ++c, ++t) {
    chunk_row[c] = r;
    chunk_begin[c] = b + t * split;
  }
}

// ---------------------------------------------------------------- transpose

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 16;
constexpr int kSortTile = kSortThreads * kSortRounds;

__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(const int32_t *__restrict__ keys,
                                                                  int64_t n, int shift,
                                                                  int64_t n_tiles,
                                                                  int32_t *__restrict__ hist) {
  __shared__ int cnt[256];
  cnt[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
  for (int r = 0; r < kSortRounds; ++r) {
    const int64_t i = base + (int64_t)r * kSortThreads + threadIdx.x;
    if (i < n) atomicAdd(&cnt[(keys[i] >> shift) & 255], 1);
  }
  __syncthreads();
  hist[(int64_t)threadIdx.x * n_tiles + blockIdx.x] = cnt[threadIdx.x];
}

// Stable scatter of one tile: elements keep their order within each digit.
__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(
    const int32_t *__restrict__ keys, const int32_t *__restrict__ vals, int64_t n, int shift,
    int64_t n_tiles, const int32_t *__restrict__ offsets, int32_t *__restrict__ keys_out,
    int32_t *__restrict__ vals_out) {
  __shared__ int wcount[kSortThreads / 32][256];
  __shared__ int run[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned lt = (1u << lane) - 1u;
  run[threadIdx.x] = offsets[(int64_t)threadIdx.x * n_tiles + blockIdx.x];
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
  for (int r = 0; r < kSortRounds; ++r) {
    for (int w = 0; w < kSortThreads / 32; ++w) wcount[w][threadIdx.x] = 0;
    __syncthreads();
    const int64_t i = base + (int64_t)r * kSortThreads + threadIdx.x;
    const bool ok = i < n;
    const int key = ok ? keys[i] : 0;
    const int d = ok ? (key >> shift) & 255 : 256;
    const unsigned peers = __match_any_sync(FULL, d);
    const int rank = __popc(peers & lt);
    if (ok && rank == 0) wcount[warp][d] = __popc(peers);
    __syncthreads();
    {  // thread t turns the per-warp counts of digit t into starting positions
      int x = run[threadIdx.x];
      for (int w = 0; w < kSortThreads / 32; ++w) {
        const int c = wcount[w][threadIdx.x];
        wcount[w][threadIdx.x] = x;
        x += c;
      }
      run[threadIdx.x] = x;
    }
    __syncthreads();
    if (ok) {
      const int dst = wcount[warp][d] + rank;
      keys_out[dst] = key;
      vals_out[dst] = vals[i];
    }
    __syncthreads();
  }
}

__global__ void iota_kernel(int32_t *__restrict__ v, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) v[i] = static_cast<int32_t>(i);
}

__global__ void col_count_kernel(const int32_t *__restrict__ col_idx, int64_t nnz,
                                 int32_t *__restrict__ counts) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < nnz; p += stride)
    atomicAdd(&counts[col_idx[p]], 1);
}

// Row id of every edge (warp per row).
__global__ void expand_rows_kernel(int64_t n_rows, const int32_t *__restrict__ row_ptr,
                                   int32_t *__restrict__ rows) {
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= n_rows) return;
  for (int p = row_ptr[r] + (threadIdx.x & 31); p < row_ptr[r + 1]; p += 32) rows[p] = static_cast<int32_t>(r);
}

__global__ void transpose_gather_kernel(int64_t nnz, const int32_t *__restrict__ order,
                                        const int32_t *__restrict__ rows,
                                        const float *__restrict__ vals,
                                        int32_t *__restrict__ col_idx_t, float *__restrict__ vals_t) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= nnz) return;
  const int p = order[k];
  col_idx_t[k] = rows[p];
  if (vals_t) vals_t[k] = vals[p];
}

// ---------------------------------------------------------------- degree bins

// Sort key of a row for the degree-binned order: 31 - bit_length(degree), so
// an ascending stable sort puts the longest rows first; rows cut into chunks
// (degree > split) get 31 and go last (their row items do no work).
// out[k] = vals[perm[k]]: edge values carried into another edge order
// (grid-stride; perm is read in order, vals gathered).
__global__ void gather_vals_kernel(int64_t nnz, const int32_t *__restrict__ perm, const float *__restrict__ vals,
                                   float *__restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += stride)
    __stcs(out + k, __ldg(vals + __ldcs(perm + k)));
}

// ELL slab of the n rows at positions [pos0, pos0 + n) of a degree-binned
// order (each of degree <= W): col[j * n + e] = column of edge j of row
// order[pos0 + e], -1 past the row's end (column-major: lanes that take
// consecutive rows read consecutive words); start[e] = the row's first edge.
__global__ void ell_build_kernel(int64_t n, int W, const int32_t *__restrict__ order, int64_t pos0,
                                 const int32_t *__restrict__ row_ptr, const int32_t *__restrict__ col_idx,
                                 int32_t *__restrict__ col, int32_t *__restrict__ start) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  const int32_t r = order[pos0 + e];
  const int b = row_ptr[r], d = row_ptr[r + 1] - b;
  start[e] = b;
  for (int j = 0; j < W; ++j) col[(int64_t)j * n + e] = j < d ? col_idx[b + j] : -1;
}

__global__ void degree_key_kernel(int64_t n_rows, const int32_t *__restrict__ row_ptr, int split,
                                  int32_t *__restrict__ keys, int32_t *__restrict__ vals) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= n_rows) return;
  const int d = row_ptr[r + 1] - row_ptr[r];
  int key = 31;
  if (!(split > 0 && d > split)) {
    const int b = d == 0 ? 0 : 32 - __clz(d);
    key = 31 - (b < 31 ? b : 31);
  }
  keys[r] = key;
  vals[r] = static_cast<int32_t>(r);
}

// ---------------------------------------------------------------- typed edges

// combined[p] = edge_type[p] * n_cols + col_idx[p]: the row of Z that edge p
// gathers when the relations' feature blocks are stacked. Types outside
// [0, n_types) are flagged and their index is set to 0.
__global__ void typed_index_kernel(int64_t nnz, int64_t n_cols, int n_types, const int32_t *__restrict__ col_idx,
                                   const int32_t *__restrict__ edge_type, int32_t *__restrict__ combined,
                                   int *__restrict__ err) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < nnz; p += stride) {
    const int r = edge_type[p];
    if (r < 0 || r >= n_types) {
      atomicOr(err, 1);
      combined[p] = 0;
    } else {
      combined[p] = static_cast<int32_t>((int64_t)r * n_cols + col_idx[p]);
    }
  }
}

// ---------------------------------------------------------------- probes

__global__ void fill_probe_kernel(void *__restrict__ p, int64_t n, int bf16, unsigned long long seed) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long z = splitmix64_mix(seed + 0x9E3779B97F4A7C15ull * (unsigned long long)(i + 1));
    const float x = (float)(z >> 40) * (1.0f / 8388608.0f) - 1.0f;  // 24 bits -> [-1, 1)
    if (bf16)
      static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    else
      static_cast<float *>(p)[i] = x;
  }
}

// Gather-rate measurement: gathered row k of a run is a SplitMix64 hash of
// (seed, k), reduced to [0, rows) by a multiply-high (no index array is read,
// so only the table's rows move). One warp per gathered row of `words`
// 16-byte words, S = ceil(words / 32) words a lane: a lane issues all its
// loads of the row before it uses any, so they are in flight together; the
// loaded words are folded into one value per lane, stored only if it hits a
// sentinel, so the loads stay and nothing is written.
template <int S>
__global__ void gather_rate_kernel(const uint4 *__restrict__ table, uint32_t rows, int64_t n, int words,
                                   unsigned long long seed, unsigned *__restrict__ sink) {
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  unsigned acc = 0;
  for (int64_t k = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); k < n; k += warps) {
    const uint32_t h = (uint32_t)(splitmix64_mix(seed + 0x9E3779B97F4A7C15ull * (unsigned long long)(k + 1)) >> 32);
    const uint4 *row = table + (int64_t)__umulhi(h, rows) * words;
    uint4 v[S];
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int w = lane + 32 * j;
      v[j] = w < words ? __ldg(row + w) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < S; ++j) acc ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
  }
  if (acc == 0x9E3779B9u) *sink = acc;
}

__global__ void compare_kernel(const void *__restrict__ a, const void *__restrict__ b, int64_t n,
                               int bf16, float rtol, float atol, unsigned long long *__restrict__ count) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  unsigned long long bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float x, y;
    if (bf16) {
      x = __bfloat162float(static_cast<const __nv_bfloat16 *>(a)[i]);
      y = __bfloat162float(static_cast<const __nv_bfloat16 *>(b)[i]);
    } else {
      x = static_cast<const float *>(a)[i];
      y = static_cast<const float *>(b)[i];
    }
    if (!(fabsf(x - y) <= atol + rtol * fabsf(y))) ++bad;
  }
  for (int off = 16; off > 0; off >>= 1) bad += __shfl_xor_sync(FULL, bad, off);
  if ((threadIdx.x & 31) == 0 && bad) atomicAdd(count, bad);
}

unsigned grid_for(int64_t n, int threads, int64_t cap = 152 * 16) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return static_cast<unsigned>(g);
}

}  // namespace

cudaError_t launch_row_stats(int64_t n_rows, const int32_t *row_ptr, int64_t long_threshold,
                             unsigned long long *ints, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(ints, 0, 40 * sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(ints + 3, 0xff, sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  if (n_rows > 0) {
    row_stats_kernel<<<grid_for(n_rows, 256), 256, 0, s>>>(n_rows, row_ptr, long_threshold, ints);
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t launch_fingerprint(int64_t n_rows, int64_t nnz, const int32_t *row_ptr,
                               const int32_t *col_idx, unsigned long long *out, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(out, 0, sizeof(unsigned long long), s);
  if (err != cudaSuccess) return err;
  fingerprint_kernel<<<grid_for(std::max<int64_t>(n_rows + 1, nnz), 256), 256, 0, s>>>(
      n_rows, nnz, row_ptr, col_idx, out);
  return cudaGetLastError();
}

cudaError_t launch_validate(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *row_ptr,
                            const int32_t *col_idx, int *err_flag, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(err_flag, 0, sizeof(int), s);
  if (err != cudaSuccess) return err;
  validate_kernel<<<grid_for(std::max<int64_t>(n_rows, nnz), 256), 256, 0, s>>>(
      n_rows, n_cols, nnz, row_ptr, col_idx, err_flag);
  return cudaGetLastError();
}

size_t scan_tmp_bytes(int64_t n) {
  const int64_t n_tiles = (n + kScanTile - 1) / kScanTile;
  return sizeof(int32_t) * (size_t)(n_tiles + 1);
}

cudaError_t launch_exclusive_scan(const int32_t *in, int32_t *out, int64_t n, void *tmp,
                                  cudaStream_t s) {
  const int64_t n_tiles = (n + kScanTile - 1) / kScanTile;
  int32_t *sums = static_cast<int32_t *>(tmp);
  if (n_tiles == 0) return cudaMemsetAsync(out, 0, sizeof(int32_t), s);
  scan_tile_sums_kernel<<<(unsigned)n_tiles, kScanThreads, 0, s>>>(in, n, sums);
  scan_sums_kernel<<<1, kScanThreads, 0, s>>>(sums, n_tiles);
  scan_apply_kernel<<<(unsigned)n_tiles, kScanThreads, 0, s>>>(in, n, sums, n_tiles, out);
  return cudaGetLastError();
}

cudaError_t build_chunk_lists(int64_t n_rows, const int32_t *row_ptr, int split, int32_t *flags,
                              int32_t *scan_out, void *scan_tmp, int32_t *long_rows,
                              int32_t *long_ptr, int32_t *chunk_row, int32_t *chunk_begin,
                              int64_t *n_long_out, int64_t *n_chunks_out, cudaStream_t s) {
  const unsigned g = (unsigned)((n_rows + 255) / 256);
  long_flags_kernel<<<g, 256, 0, s>>>(n_rows, row_ptr, split, flags);
  cudaError_t err = launch_exclusive_scan(flags, scan_out, n_rows, scan_tmp, s);
  if (err != cudaSuccess) return err;
  int32_t n_long = 0;
  err = cudaMemcpyAsync(&n_long, scan_out + n_rows, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return err;
  // counts reuse `flags` (the flags are no longer needed after the scan)
  long_compact_kernel<<<g, 256, 0, s>>>(n_rows, row_ptr, split, scan_out, long_rows, flags);
  err = launch_exclusive_scan(flags, long_ptr, n_long, scan_tmp, s);
  if (err != cudaSuccess) return err;
  int32_t n_chunks = 0;
  err = cudaMemcpyAsync(&n_chunks, long_ptr + n_long, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return err;
  if (n_long > 0) {
    chunk_fill_kernel<<<(unsigned)((n_long + 255) / 256), 256, 0, s>>>(n_long, row_ptr, split, long_rows,
                                                                       long_ptr, chunk_row, chunk_begin);
    err = cudaGetLastError();
  }
  *n_long_out = n_long;
  *n_chunks_out = n_chunks;
  return err;
}

cudaError_t csr_transpose(int64_t n_rows, int64_t n_cols, int64_t nnz, const int32_t *row_ptr,
                          const int32_t *col_idx, const float *vals, int32_t *row_ptr_t,
                          int32_t *col_idx_t, float *vals_t, int32_t *perm, cudaStream_t s) {
  cudaError_t err = cudaSuccess;
  // row_ptr_t = exclusive scan of the column counts
  int32_t *counts = nullptr;
  void *scan_tmp = nullptr;
  const int64_t scan_n = std::max<int64_t>(n_cols, 256 * ((nnz + kSortTile - 1) / kSortTile));
  if ((err = cudaMallocAsync(&counts, sizeof(int32_t) * (size_t)std::max<int64_t>(n_cols, 1), s)) != cudaSuccess) return err;
  if ((err = cudaMallocAsync(&scan_tmp, scan_tmp_bytes(scan_n), s)) != cudaSuccess) {
    cudaFreeAsync(counts, s);
    return err;
  }
  cudaMemsetAsync(counts, 0, sizeof(int32_t) * (size_t)std::max<int64_t>(n_cols, 1), s);
  if (nnz > 0) col_count_kernel<<<grid_for(nnz, 256), 256, 0, s>>>(col_idx, nnz, counts);
  err = launch_exclusive_scan(counts, row_ptr_t, n_cols, scan_tmp, s);
  if (err == cudaSuccess && nnz > 0) {
    const int64_t n_tiles = (nnz + kSortTile - 1) / kSortTile;
    int32_t *ka = nullptr, *kb = nullptr, *va = nullptr, *vb = nullptr, *hist = nullptr,
            *offs = nullptr, *rows = nullptr;
    const size_t nb = sizeof(int32_t) * (size_t)nnz;
    const size_t hb = sizeof(int32_t) * (size_t)(256 * n_tiles + 1);
    int32_t **bufs[7] = {&ka, &kb, &va, &vb, &hist, &offs, &rows};
    const size_t sizes[7] = {nb, nb, nb, nb, hb, hb, nb};
    for (int i = 0; i < 7 && err == cudaSuccess; ++i)
      err = cudaMallocAsync(reinterpret_cast<void **>(bufs[i]), sizes[i], s);
    if (err == cudaSuccess) {
      cudaMemcpyAsync(ka, col_idx, nb, cudaMemcpyDeviceToDevice, s);
      iota_kernel<<<(unsigned)((nnz + 255) / 256), 256, 0, s>>>(va, nnz);
      int bits = 0;
      while (bits < 31 && (1ll << bits) < n_cols) ++bits;
      for (int shift = 0; shift < bits; shift += 8) {
        radix_hist_kernel<<<(unsigned)n_tiles, kSortThreads, 0, s>>>(ka, nnz, shift, n_tiles, hist);
        launch_exclusive_scan(hist, offs, 256 * n_tiles, scan_tmp, s);
        radix_scatter_kernel<<<(unsigned)n_tiles, kSortThreads, 0, s>>>(ka, va, nnz, shift, n_tiles,
                                                                         offs, kb, vb);
        std::swap(ka, kb);
        std::swap(va, vb);
      }
      expand_rows_kernel<<<(unsigned)((n_rows + 7) / 8), 256, 0, s>>>(n_rows, row_ptr, rows);
      transpose_gather_kernel<<<(unsigned)((nnz + 255) / 256), 256, 0, s>>>(
          nnz, va, rows, vals, col_idx_t, vals ? vals_t : nullptr);
      err = cudaGetLastError();
      // position k of A^T holds edge va[k] of A
      if (err == cudaSuccess && perm)
        err = cudaMemcpyAsync(perm, va, sizeof(int32_t) * (size_t)nnz, cudaMemcpyDeviceToDevice, s);
    }
    for (int i = 0; i < 7; ++i)
      if (*bufs[i]) cudaFreeAsync(*bufs[i], s);
  }
  cudaFreeAsync(counts, s);
  cudaFreeAsync(scan_tmp, s);
  return err;
}

cudaError_t build_row_order(int64_t n_rows, const int32_t *row_ptr, int split, int32_t *order,
                            int32_t *bucket_start, cudaStream_t s) {
  if (n_rows <= 0) return cudaSuccess;
  const int64_t n_tiles = (n_rows + kSortTile - 1) / kSortTile;
  int32_t *keys = nullptr, *keys_out = nullptr, *vals = nullptr, *hist = nullptr, *offs = nullptr;
  void *scan_tmp = nullptr;
  const size_t nb = sizeof(int32_t) * (size_t)n_rows;
  const size_t hb = sizeof(int32_t) * (size_t)(256 * n_tiles + 1);
  cudaError_t err = cudaSuccess;
  int32_t **bufs[5] = {&keys, &keys_out, &vals, &hist, &offs};
  const size_t sizes[5] = {nb, nb, nb, hb, hb};
  for (int i = 0; i < 5 && err == cudaSuccess; ++i) err = cudaMallocAsync(reinterpret_cast<void **>(bufs[i]), sizes[i], s);
  if (err == cudaSuccess) err = cudaMallocAsync(&scan_tmp, scan_tmp_bytes(256 * n_tiles), s);
  if (err == cudaSuccess) {
    degree_key_kernel<<<(unsigned)((n_rows + 255) / 256), 256, 0, s>>>(n_rows, row_ptr, split, keys, vals);
    // one stable pass over the 5-bit key
    radix_hist_kernel<<<(unsigned)n_tiles, kSortThreads, 0, s>>>(keys, n_rows, 0, n_tiles, hist);
    launch_exclusive_scan(hist, offs, 256 * n_tiles, scan_tmp, s);
    radix_scatter_kernel<<<(unsigned)n_tiles, kSortThreads, 0, s>>>(keys, vals, n_rows, 0, n_tiles, offs, keys_out,
                                                                     order);
    err = cudaGetLastError();
    // where each key starts in the order: the scanned count of tile 0 of its digit
    for (int k = 0; k < 32 && err == cudaSuccess && bucket_start; ++k)
      err = cudaMemcpyAsync(bucket_start + k, offs + (int64_t)k * n_tiles, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (err == cudaSuccess && bucket_start) {
      err = cudaStreamSynchronize(s);
      bucket_start[32] = static_cast<int32_t>(n_rows);
    }
  }
  for (int i = 0; i < 5; ++i)
    if (*bufs[i]) cudaFreeAsync(*bufs[i], s);
  if (scan_tmp) cudaFreeAsync(scan_tmp, s);
  return err;
}

cudaError_t build_ell(int64_t n, int W, const int32_t *order, int64_t pos0, const int32_t *row_ptr,
                      const int32_t *col_idx, int32_t *col, int32_t *start, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  ell_build_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(n, W, order, pos0, row_ptr, col_idx, col, start);
  return cudaGetLastError();
}

cudaError_t launch_gather_vals(int64_t nnz, const int32_t *perm, const float *vals, float *out, cudaStream_t s) {
  if (nnz <= 0) return cudaSuccess;
  gather_vals_kernel<<<grid_for(nnz, 256, 152 * 32), 256, 0, s>>>(nnz, perm, vals, out);
  return cudaGetLastError();
}

cudaError_t launch_typed_index(int64_t nnz, int64_t n_cols, int n_types, const int32_t *col_idx,
                               const int32_t *edge_type, int32_t *combined, int *err, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e != cudaSuccess || nnz <= 0) return e;
  typed_index_kernel<<<grid_for(nnz, 256), 256, 0, s>>>(nnz, n_cols, n_types, col_idx, edge_type, combined, err);
  return cudaGetLastError();
}

cudaError_t fill_probe(void *p, int64_t n_elems, DType dt, uint64_t seed, cudaStream_t s) {
  if (n_elems <= 0) return cudaSuccess;
  fill_probe_kernel<<<grid_for(n_elems, 256), 256, 0, s>>>(p, n_elems, dt == DType::BF16, seed);
  return cudaGetLastError();
}

cudaError_t launch_gather_rate(const void *table, int64_t rows, int64_t n, int row_bytes, int grid,
                               uint64_t seed, unsigned *sink, cudaStream_t s) {
  if (n <= 0 || rows <= 0) return cudaSuccess;
  const uint4 *t = static_cast<const uint4 *>(table);
  const int words = row_bytes / 16;
  const uint32_t r = (uint32_t)rows;
  switch ((words + 31) / 32) {
    case 1: gather_rate_kernel<1><<<grid, 256, 0, s>>>(t, r, n, words, seed, sink); break;
    case 2: gather_rate_kernel<2><<<grid, 256, 0, s>>>(t, r, n, words, seed, sink); break;
    case 3:
    case 4: gather_rate_kernel<4><<<grid, 256, 0, s>>>(t, r, n, words, seed, sink); break;
    default: gather_rate_kernel<8><<<grid, 256, 0, s>>>(t, r, n, words, seed, sink); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_compare(const void *a, const void *b, int64_t n, DType dt, float rtol,
                           float atol, unsigned long long *count, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(count, 0, sizeof(unsigned long long), s);
  if (err != cudaSuccess || n <= 0) return err;
  compare_kernel<<<grid_for(n, 256), 256, 0, s>>>(a, b, n, dt == DType::BF16, rtol, atol, count);
  return cudaGetLastError();
}

}  // namespace autosage
