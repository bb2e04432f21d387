// dsa_select_noalloc: the fused select call with its scratch in a static device
// array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// selection: code recorded inside a CUDA stream capture (cudaMalloc is not a
// capturable operation), plugins hosted by a framework that owns every device
// allocation, and latency-critical serving loops that forbid allocation after
// start-up.  For them this entry point keeps its only scratch - one 4096-bin
// score histogram per query - in a file-scope __device__ array of fixed size.
// The caller still passes every input and output buffer.
//
// Limits and sharing rules:
//  * at most kNoAllocMaxQ queries per call (larger Q returns DSA_ERR_UNSUPPORTED);
//  * every GPU that loads the library keeps the array (1 MiB) until the process
//    exits;
//  * all calls on a device share the one array, which keeps what the last call
//    left in it: each call clears the part it uses before the scoring kernel
//    runs, and calls that overlap on the GPU (different streams, no ordering
//    between them) race on it and must not be issued;
//  * the first call on each device with at least one query looks up the
//    array's device address (cudaGetSymbolAddress, with that device current),
//    whatever its geometry; make that first call before any stream capture.
//    The address is kept for the life of the process, which assumes the
//    device's primary context lives as long (no cudaDeviceReset in between).
#include <cmath>
#include <mutex>

#include "dsa_internal.cuh"

namespace {

constexpr int kNoAllocMaxQ = 64;
constexpr int kHistBins = 4096;
constexpr int kMaxDevices = 64;

// The scratch itself: Q x 4096 uint32 histogram bins (zero at module load).
static __device__ __align__(256) uint32_t g_select_scratch[kNoAllocMaxQ * kHistBins];

// In host code `g_select_scratch` only names a host-side stand-in; kernels must
// be given the device address, looked up once per device.
uint32_t* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return DSA_OK;
}

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" int dsa_select_noalloc(const void* q, const float* weights, float scale,
                                  const void* pool_keys, int pool_rows,
                                  const int32_t* pool_start,
                                  const uint8_t* pool_valid, const int32_t* n_pools,
                                  const int32_t* cu_pool_cap, const int32_t* q_seq,
                                  const int32_t* q_pos, int Q, int B, int H, int D, int kpool,
                                  int P_ld, int select_k, int out_width, int dtype, float* scores,
                                  int32_t* pool_ids, int32_t* token_ids, int32_t* status_dev,
                                  void* stream) {
  if (Q < 0 || B < 0 || H < 1 || P_ld < 1 || select_k < 1 || out_width < 1 || pool_rows < 1)
    return DSA_ERR_INVALID_ARG;
  if (kpool < 1 || kpool > DSA_KPOOL_MAX) return DSA_ERR_INVALID_ARG;
  if ((long long)out_width < (long long)select_k * kpool) return DSA_ERR_INVALID_ARG;
  if ((dtype != DSA_BF16 && dtype != DSA_F32) || !(scale > 0.f) || !std::isfinite(scale))
    return DSA_ERR_INVALID_ARG;
  if ((D != 32 && D != 64 && D != 128 && D != 256) || H > 64 || select_k > DSA_SELECT_K_MAX)
    return DSA_ERR_UNSUPPORTED;
  if (Q > kNoAllocMaxQ) return DSA_ERR_UNSUPPORTED;  // the static scratch holds 64 queries
  if (Q == 0) return DSA_OK;
  if (B == 0) return DSA_ERR_INVALID_ARG;
  if (!q || !weights || !pool_keys || !pool_start || !pool_valid || !n_pools || !cu_pool_cap ||
      !scores || !pool_ids || !token_ids)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(weights, 16) || !aligned(pool_keys, 16) || !aligned(scores, 4) ||
      !aligned(n_pools, 4) || !aligned(cu_pool_cap, 4) || !aligned(pool_start, 4) ||
      !aligned(pool_ids, 4) || !aligned(token_ids, 4) || (q_seq && !aligned(q_seq, 4)) ||
      (q_pos && !aligned(q_pos, 4)) || (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the address is looked up on every device's first call, whatever the
  // geometry, so that no later call does it inside a stream capture
  uint32_t* scratch = nullptr;
  int r = scratch_for_current_device(&scratch);
  if (r != DSA_OK) return r;
  uint32_t* hist = nullptr;
  if (dsa::index_fills_histogram(Q, q_seq, H, D, dtype)) {
    hist = scratch;
    // the histogram must start at zero: clear this call's share of the array
    if (cudaMemsetAsync(hist, 0, (size_t)Q * kHistBins * sizeof(uint32_t), st) != cudaSuccess)
      return DSA_ERR_CUDA;
  }
  // without the scoring kernel's histogram the selection kernel builds its
  // own on chip: no scratch is touched
  r = dsa::launch_index_scores(q, weights, scale, pool_keys, pool_rows, pool_start, pool_valid,
                               n_pools, cu_pool_cap, q_seq, q_pos, Q, B, H, D, kpool, P_ld, dtype,
                               scores, hist, status_dev, st);
  if (r != DSA_OK) return r;
  return dsa::launch_select_after_index(scores, Q, P_ld, select_k, pool_ids, hist, pool_start,
                                        cu_pool_cap, q_seq, B, kpool, out_width, token_ids,
                                        status_dev, st);
}
