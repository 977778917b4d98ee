// Row sharding of the aggregation across GPUs (one process per GPU).
//
// Every operation of the library is defined per destination row (AutoSAGE,
// "Input-Aware CUDA Scheduling for Sparse GNN Aggregation (SpMM/SDDMM) and
// CSR Attention", Abstract; benchmark page "fused sparse attention-value
// aggregation", problem statement: an output row per destination node from
// its incoming edges), so contiguous row ranges are independent units. A
// shard is a range of rows with about equal edge counts; it needs the
// feature rows of the columns its edges reference (its halo), which one
// exchange step brings to its GPU; its outputs are its own rows, so nothing
// is reduced afterwards. SpMM with A^T shards the rows of A^T the same way.
//
// This file holds the host-side partition and halo computation (plain C++ on
// host arrays: planning work done once per graph) and the GPU gather that
// packs halo rows into a dense matrix.
#include <algorithm>
#include <vector>

#include "../../include/autosage.h"
#include "internal.h"

namespace autosage {
autosage_status report(autosage_status st, const char *msg);
}

namespace {

// out[k, :] = X[idx[k], :], one warp per output row, W-byte words.
template <typename W>
__global__ void gather_rows_kernel(const char *__restrict__ X, int64_t ldx_bytes, const int32_t *__restrict__ idx,
                                   int64_t n, int64_t words, char *__restrict__ out, int64_t ldo_bytes) {
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  const int lane = threadIdx.x & 31;
  for (int64_t k = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); k < n; k += warps) {
    const W *src = reinterpret_cast<const W *>(X + (int64_t)__ldg(idx + k) * ldx_bytes);
    W *dst = reinterpret_cast<W *>(out + k * ldo_bytes);
    for (int64_t w = lane; w < words; w += 32) dst[w] = __ldg(src + w);
  }
}

}  // namespace

extern "C" {

autosage_status autosage_partition_rows(const int32_t *row_ptr, int64_t n_rows, int parts, int64_t *bounds) {
  if (!row_ptr || !bounds || n_rows < 0 || parts < 1)
    return autosage::report(AUTOSAGE_ERR_INVALID_ARG, "partition: NULL array, negative size or parts < 1");
  if (row_ptr[0] != 0) return autosage::report(AUTOSAGE_ERR_INVALID_CSR, "partition: row_ptr[0] != 0");
  for (int64_t i = 0; i < n_rows; ++i)
    if (row_ptr[i + 1] < row_ptr[i]) return autosage::report(AUTOSAGE_ERR_INVALID_CSR, "partition: row_ptr decreases");
  const int64_t nnz = row_ptr[n_rows];
  bounds[0] = 0;
  bounds[parts] = n_rows;
  for (int k = 1; k < parts; ++k) {
    // the first row whose start reaches k / parts of the edges; a cut never
    // moves backwards, so parts may be empty but never overlap
    const int64_t target = (nnz * k + parts - 1) / parts;
    const int32_t *r = std::lower_bound(row_ptr, row_ptr + n_rows + 1, (int32_t)target);
    bounds[k] = std::max<int64_t>(bounds[k - 1], std::min<int64_t>(r - row_ptr, n_rows));
  }
  return AUTOSAGE_OK;
}

autosage_status autosage_shard_halo(const int32_t *row_ptr, const int32_t *col_idx, int64_t n_cols,
                                    int64_t row_begin, int64_t row_end, int32_t *halo, int64_t *n_halo,
                                    int32_t *local_col) {
  if (!row_ptr || !halo || !n_halo || n_cols < 0 || row_begin < 0 || row_end < row_begin)
    return autosage::report(AUTOSAGE_ERR_INVALID_ARG, "shard halo: NULL array or bad row range");
  const int64_t b = row_ptr[row_begin], e = row_ptr[row_end];
  if (e < b) return autosage::report(AUTOSAGE_ERR_INVALID_CSR, "shard halo: row_ptr decreases");
  if (e > b && (!col_idx || !local_col)) return autosage::report(AUTOSAGE_ERR_INVALID_ARG, "shard halo: NULL edges");
  // mark the referenced columns, number them in increasing order, renumber the edges
  std::vector<int32_t> pos((size_t)n_cols, -1);
  for (int64_t p = b; p < e; ++p) {
    const int32_t c = col_idx[p];
    if (c < 0 || c >= n_cols) return autosage::report(AUTOSAGE_ERR_INVALID_CSR, "shard halo: column out of range");
    pos[(size_t)c] = 0;
  }
  int64_t h = 0;
  for (int64_t c = 0; c < n_cols; ++c)
    if (pos[(size_t)c] == 0) {
      pos[(size_t)c] = (int32_t)h;
      halo[h++] = (int32_t)c;
    }
  *n_halo = h;
  for (int64_t p = b; p < e; ++p) local_col[p - b] = pos[(size_t)col_idx[p]];
  return AUTOSAGE_OK;
}

autosage_status autosage_gather_rows(const void *X, int64_t ldx, const int32_t *idx, int64_t n, int64_t F,
                                     autosage_dtype dt, void *out, int64_t ldo, void *stream) {
  if (n < 0 || F < 1 || ldx < F || ldo < F || (dt != AUTOSAGE_F32 && dt != AUTOSAGE_BF16))
    return autosage::report(AUTOSAGE_ERR_INVALID_ARG, "gather rows: bad sizes or dtype");
  if (n == 0) return AUTOSAGE_OK;
  if (!X || !idx || !out) return autosage::report(AUTOSAGE_ERR_INVALID_ARG, "gather rows: NULL pointer");
  const int64_t es = dt == AUTOSAGE_F32 ? 4 : 2;
  const int64_t row = F * es, lx = ldx * es, lo = ldo * es;
  // the widest word that every address and row length allow
  int wb = 2;
  for (int cand : {16, 8, 4}) {
    if (((uintptr_t)X | (uintptr_t)out | (uint64_t)lx | (uint64_t)lo | (uint64_t)row) % cand == 0) {
      wb = cand;
      break;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t blocks = std::min<int64_t>((n + 7) / 8, 152 * 16);
  const char *x = static_cast<const char *>(X);
  char *o = static_cast<char *>(out);
  switch (wb) {
    case 16: gather_rows_kernel<uint4><<<(unsigned)blocks, 256, 0, s>>>(x, lx, idx, n, row / 16, o, lo); break;
    case 8: gather_rows_kernel<uint2><<<(unsigned)blocks, 256, 0, s>>>(x, lx, idx, n, row / 8, o, lo); break;
    case 4: gather_rows_kernel<uint32_t><<<(unsigned)blocks, 256, 0, s>>>(x, lx, idx, n, row / 4, o, lo); break;
    default: gather_rows_kernel<uint16_t><<<(unsigned)blocks, 256, 0, s>>>(x, lx, idx, n, row / 2, o, lo); break;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return autosage::report(AUTOSAGE_ERR_CUDA, cudaGetErrorString(e));
  return AUTOSAGE_OK;
}

}  // extern "C"
