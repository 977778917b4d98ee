// Unfused CSR attention for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocator) from inside their
// work loop: a serving process that reserved all device memory for its own
// pool up front, or a latency-critical loop where a driver allocation may
// synchronise the device and take unbounded time. The unfused attention
// needs an fp32 score array of nnz * heads elements; this variant keeps it in
// a fixed array in device memory that the library owns, so a call allocates
// nothing. The array lives from the library's load until the process exits,
// on every GPU the library is loaded on.
#include <mutex>

#include "../../include/autosage.h"
#include "internal.h"

namespace autosage {
autosage_status check_attention_args(const autosage_csr *A, const void *Q, const void *K, const void *V, int heads,
                                     int64_t D, autosage_dtype dt, const void *out);
autosage_status attention_unfused_with_scores(const autosage_csr *A, const void *Q, const void *K,
                                              const void *V, int heads, int64_t D, autosage_dtype dt,
                                              float scale, void *out, float *scores, cudaStream_t s);
autosage_status report(autosage_status st, const char *msg);
}

namespace {

// The score scratch: AUTOSAGE_NOALLOC_MAX_SCORES fp32 elements (16 MiB).
static __device__ __align__(256) float g_noalloc_scores[AUTOSAGE_NOALLOC_MAX_SCORES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device. The host-side symbol
// is only a stand-in for the device array, so the address is looked up once
// per device (with that device current) and cached.
autosage_status scratch_address(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return autosage::report(AUTOSAGE_ERR_CUDA, "no current CUDA device");
  if (dev < 0 || dev >= kMaxDevices) return autosage::report(AUTOSAGE_ERR_UNSUPPORTED, "device index above 63");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scores);
    if (e != cudaSuccess || !p)
      return autosage::report(AUTOSAGE_ERR_CUDA, "cannot get the device address of the score scratch");
    g_addr[dev] = static_cast<float *>(p);
  }
  *out = g_addr[dev];
  return AUTOSAGE_OK;
}

}  // namespace

extern "C" autosage_status autosage_csr_attention_unfused_noalloc(const autosage_csr *A, const void *Q,
                                                                  const void *K, const void *V, int heads,
                                                                  int64_t D, autosage_dtype dt, float scale,
                                                                  void *out, void *stream) {
  // every argument is checked on the host before the device is touched
  autosage_status st = autosage::check_attention_args(A, Q, K, V, heads, D, dt, out);
  if (st != AUTOSAGE_OK) return st;
  if ((uint64_t)A->nnz * (uint64_t)heads > (uint64_t)AUTOSAGE_NOALLOC_MAX_SCORES)
    return autosage::report(AUTOSAGE_ERR_UNSUPPORTED,
                            "nnz * heads exceeds the fixed score scratch (AUTOSAGE_NOALLOC_MAX_SCORES = 4194304 "
                            "fp32 elements); use autosage_csr_attention instead");
  float *scores = nullptr;
  st = scratch_address(&scores);
  if (st != AUTOSAGE_OK) return st;
  // every score the softmax and the SpMM read is written by the SDDMM first,
  // so nothing in the scratch has to start at zero
  return autosage::attention_unfused_with_scores(A, Q, K, V, heads, D, dt, scale, out, scores,
                                                 static_cast<cudaStream_t>(stream));
}
