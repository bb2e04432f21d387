// topk_pools and expand_selection.
//
// Module glm5next_dsa::tp, "Why the indexer is REPLICATED": the selection order
// is pinned - higher score first, then the smaller pool index.  Module
// glm5next_dsa, "Shape of the pipeline" ([Q, select_k] pool ids; [Q, out_width]
// token ids with -1 = invalid) and "Traps carried from Slice 8" (the -1
// destination is written in full).
//
// Every candidate gets a unique 64-bit key (order-preserving score bits << 32 |
// ~pool), so "score descending, pool ascending" is plain key-descending order
// and the selected set and its order are unique.
//
// Top-k is a radix select spread over C CTAs per query row:
//   1. histogram of the top 12 key bits over the row (C CTAs, one global
//      histogram per query);
//   2. each CTA finds the threshold bin (the bin where the count from the top
//      reaches select_k), appends keys above it to a "sure" list and keys in it
//      to a "tie" list; the last CTA to finish the row (atomic ticket, no
//      waiting) picks the exact remaining keys from the tie list by rank or by
//      a radix select on the remaining 52 key bits, sorts the select_k keys and
//      writes the row.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kBins = 4096;           // top 12 bits of the 32-bit score key
constexpr int kBinShift = 20;
constexpr int kTieCap = 4096;         // tie-list capacity per query (overflow: slow exact path)
constexpr int kThreads = 512;
constexpr int kSmallSort = 1024;      // rank sort up to this many keys, bitonic above

struct TopkWs {
  uint32_t* hist;     // [Q][kBins]
  uint32_t* ctr;      // [Q][4]: n_sure, n_tie, done, spare
  uint64_t* sure;     // [Q][K]
  uint64_t* tie;      // [Q][kTieCap]
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t ws_header_bytes(int Q) {
  return align256((size_t)Q * kBins * 4) + align256((size_t)Q * 16);
}

__host__ __device__ inline TopkWs carve(void* ws, int Q, int K) {
  char* p = static_cast<char*>(ws);
  TopkWs w;
  w.hist = reinterpret_cast<uint32_t*>(p);
  p += align256((size_t)Q * kBins * 4);
  w.ctr = reinterpret_cast<uint32_t*>(p);
  p += align256((size_t)Q * 16);
  w.sure = reinterpret_cast<uint64_t*>(p);
  p += align256((size_t)Q * K * 8);
  w.tie = reinterpret_cast<uint64_t*>(p);
  return w;
}

__device__ __forceinline__ uint64_t full_key(float s, int p) {
  return ((uint64_t)score_key(s) << 32) | (uint64_t)(0xffffffffu - (uint32_t)p);
}
__device__ __forceinline__ int key_pool(uint64_t key) {
  return (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu));
}

__global__ void __launch_bounds__(kThreads)
    topk_hist_kernel(const float* __restrict__ scores, int P_ld, int chunks, TopkWs ws) {
  __shared__ uint32_t h[kBins];
  pdl_wait();
  for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
  __syncthreads();
  const int q = blockIdx.y;
  const long long lo = (long long)P_ld * blockIdx.x / chunks;
  const long long hi = (long long)P_ld * (blockIdx.x + 1) / chunks;
  const float* row = scores + (long long)q * P_ld;
  for (long long i = lo + threadIdx.x; i < hi; i += kThreads) {
    const float s = row[i];
    if (is_candidate(s)) atomicAdd(&h[score_key(s) >> kBinShift], 1u);
  }
  __syncthreads();
  uint32_t* gh = ws.hist + (size_t)q * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (h[i]) atomicAdd(&gh[i], h[i]);
}

// Block-wide: threshold bin for select_k over hist (smem).  Sets *thr (-1 when
// every candidate fits) and *above (count strictly above the bin).
__device__ void find_threshold(const uint32_t* h, int K, int* s_thr, uint32_t* s_above,
                               uint32_t* s_scan) {
  constexpr int kPer = kBins / kThreads;  // 8 bins per thread
  const int tid = threadIdx.x;
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) local += h[tid * kPer + i];
  s_scan[tid] = local;
  __syncthreads();
  // suffix sums over threads (Hillis-Steele on kThreads entries)
  for (int o = 1; o < kThreads; o <<= 1) {
    uint32_t v = s_scan[tid] + ((tid + o < kThreads) ? s_scan[tid + o] : 0u);
    __syncthreads();
    s_scan[tid] = v;
    __syncthreads();
  }
  const uint32_t total = s_scan[0];
  if (tid == 0) { *s_thr = -1; *s_above = total; }
  __syncthreads();
  if (total > (uint32_t)K) {
    const uint32_t incl = s_scan[tid];                     // bins >= tid*kPer
    const uint32_t excl = incl - local;                    // bins > tid*kPer+kPer-1
    if (excl < (uint32_t)K && incl >= (uint32_t)K) {
      uint32_t run = excl;
      for (int i = kPer - 1; i >= 0; --i) {
        const uint32_t c = h[tid * kPer + i];
        if (run + c >= (uint32_t)K) {
          *s_thr = tid * kPer + i;
          *s_above = run;
          break;
        }
        run += c;
      }
    }
  }
  __syncthreads();
}

// Warp-aggregated append of `key` (when `take`) into list[ctr++], capped.
__device__ __forceinline__ void append(bool take, uint64_t key, uint32_t* ctr, uint64_t* list,
                                       uint32_t cap) {
  const unsigned mask = __ballot_sync(0xffffffffu, take);
  if (!mask) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(ctr, (uint32_t)__popc(mask));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (take) {
    const uint32_t slot = base + __popc(mask & ((1u << lane) - 1u));
    if (slot < cap) list[slot] = key;
  }
}

// Exact R-th largest key (1-based) among keys given by get(i) (i < n, present
// flag), by 8-bit radix passes from the top.  Block-wide; smem hist[256].
template <typename Get>
__device__ uint64_t radix_kth(int n, uint32_t R, Get get, uint32_t* sh, uint64_t* s_res,
                              uint32_t* s_r) {
  uint64_t prefix = 0;
  uint64_t mask = 0;
  if (threadIdx.x == 0) *s_r = R;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) sh[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) {
      uint64_t key;
      if (get(i, key) && (key & mask) == prefix) atomicAdd(&sh[(key >> shift) & 255], 1u);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t r = *s_r, run = 0;
      int d = 255;
      for (; d > 0; --d) {
        if (run + sh[d] >= r) break;
        run += sh[d];
      }
      *s_r = r - run;
      *s_res = prefix | ((uint64_t)d << shift);
    }
    __syncthreads();
    prefix = *s_res;
    mask |= (uint64_t)255 << shift;
    __syncthreads();
  }
  return prefix;
}

// Sort n (<= cap) keys in smem descending; keys[n..cap) are scratch.
__device__ void sort_desc(uint64_t* keys, int n, uint64_t* tmp) {
  if (n <= kSmallSort) {
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint64_t k = keys[i];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += keys[j] > k;
      tmp[rank] = k;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += kThreads) keys[i] = tmp[i];
    __syncthreads();
    return;
  }
  int N = 1;
  while (N < n) N <<= 1;
  for (int i = n + threadIdx.x; i < N; i += kThreads) keys[i] = 0;
  __syncthreads();
  for (int k = 2; k <= N; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < N; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) { keys[i] = b; keys[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    topk_select_kernel(const float* __restrict__ scores, int P_ld, int K, int chunks, TopkWs ws,
                       int32_t* __restrict__ pool_ids) {
  extern __shared__ __align__(16) unsigned char smem[];
  uint32_t* h = reinterpret_cast<uint32_t*>(smem);                 // kBins
  uint32_t* s_scan = h + kBins;                                    // kThreads
  // final-phase buffers reuse the same dynamic smem after the filter pass
  __shared__ int s_thr;
  __shared__ uint32_t s_above, s_last, s_r, s_nsel;
  __shared__ uint64_t s_res;
  pdl_wait();
  const int q = blockIdx.y;
  const uint32_t* gh = ws.hist + (size_t)q * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = __ldcg(gh + i);
  __syncthreads();
  find_threshold(h, K, &s_thr, &s_above, s_scan);
  const int thr = s_thr;
  uint32_t* ctr = ws.ctr + (size_t)q * 4;
  uint64_t* sure = ws.sure + (size_t)q * K;
  uint64_t* tie = ws.tie + (size_t)q * kTieCap;
  const float* row = scores + (long long)q * P_ld;
  const long long lo = (long long)P_ld * blockIdx.x / chunks;
  const long long hi = (long long)P_ld * (blockIdx.x + 1) / chunks;
  for (long long base = lo; base < hi; base += kThreads) {
    const long long i = base + threadIdx.x;
    bool in_sure = false, in_tie = false;
    uint64_t key = 0;
    if (i < hi) {
      const float s = row[i];
      if (is_candidate(s)) {
        key = full_key(s, (int)i);
        const int bin = (int)(key >> (32 + kBinShift));
        in_sure = bin > thr;
        in_tie = bin == thr;
      }
    }
    append(in_sure, key, &ctr[0], sure, (uint32_t)K);
    append(in_tie, key, &ctr[1], tie, (uint32_t)kTieCap);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&ctr[2], 1u) == (uint32_t)(chunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- final phase: this CTA owns the row now.
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem);              // up to 2*max(K, kTieCap) keys
  uint64_t* tmp = sel + (K > kTieCap ? K : kTieCap);
  const uint32_t n_sure = __ldcg(&ctr[0]);
  const uint32_t n_tie = __ldcg(&ctr[1]);
  uint32_t n_sel;
  if (thr < 0) {
    n_sel = n_sure;  // every candidate is in the sure list (<= K of them)
    for (uint32_t i = threadIdx.x; i < n_sel; i += kThreads) sel[i] = __ldcg(sure + i);
    __syncthreads();
  } else {
    const uint32_t R = (uint32_t)K - n_sure;                      // keys still needed, >= 1
    n_sel = (uint32_t)K;
    for (uint32_t i = threadIdx.x; i < n_sure; i += kThreads) sel[i] = __ldcg(sure + i);
    if (threadIdx.x == 0) s_nsel = n_sure;
    __syncthreads();
    if (n_tie <= (uint32_t)kSmallSort) {
      for (uint32_t i = threadIdx.x; i < n_tie; i += kThreads) tmp[i] = __ldcg(tie + i);
      __syncthreads();
      for (uint32_t i = threadIdx.x; i < n_tie; i += kThreads) {
        const uint64_t k = tmp[i];
        uint32_t rank = 0;
        for (uint32_t j = 0; j < n_tie; ++j) rank += tmp[j] > k;
        if (rank < R) sel[n_sure + rank] = k;
      }
      __syncthreads();
    } else {
      uint64_t T;
      uint32_t* sh = reinterpret_cast<uint32_t*>(tmp);
      if (n_tie <= (uint32_t)kTieCap) {
        auto get = [&](int i, uint64_t& k) { k = __ldcg(tie + i); return true; };
        T = radix_kth((int)n_tie, R, get, sh, &s_res, &s_r);
        for (uint32_t i = threadIdx.x; i < n_tie; i += kThreads) {
          const uint64_t k = __ldcg(tie + i);
          if (k >= T) {
            const uint32_t slot = atomicAdd(&s_nsel, 1u);
            if (slot < (uint32_t)K) sel[slot] = k;
          }
        }
      } else {  // tie list overflowed: exact select straight from the row
        auto get = [&](int i, uint64_t& k) {
          const float s = row[i];
          if (!is_candidate(s)) return false;
          k = full_key(s, i);
          return (int)(k >> (32 + kBinShift)) == thr;
        };
        T = radix_kth(P_ld, R, get, sh, &s_res, &s_r);
        for (int i = threadIdx.x; i < P_ld; i += kThreads) {
          uint64_t k;
          if (get(i, k) && k >= T) {
            const uint32_t slot = atomicAdd(&s_nsel, 1u);
            if (slot < (uint32_t)K) sel[slot] = k;
          }
        }
      }
      __syncthreads();
    }
  }
  sort_desc(sel, (int)n_sel, tmp);
  int32_t* out = pool_ids + (long long)q * K;
  for (int j = threadIdx.x; j < K; j += kThreads)
    out[j] = j < (int)n_sel ? key_pool(sel[j]) : -1;
  pdl_launch_dependents();
}

__global__ void expand_kernel(const int32_t* __restrict__ pool_ids,
                              const int32_t* __restrict__ pool_start,
                              const int32_t* __restrict__ cu_pool_cap,
                              const int32_t* __restrict__ q_seq, int B, int K, int kpool, int W,
                              int32_t* __restrict__ token_ids, int32_t* status) {
  pdl_wait();
  const int q = blockIdx.y;
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= W) return;
  const int b = q_seq ? q_seq[q] : 0;
  int tok = -1;
  if (b < 0 || b >= B) {
    if (c == 0) flag(status, DSA_DEV_BAD_QSEQ);
  } else if (c < K * kpool) {
    const int j = c / kpool, s = c - j * kpool;
    const int p = pool_ids[(long long)q * K + j];
    const long long base = cu_pool_cap[b];
    const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
    if (p >= cap) {
      if (s == 0) flag(status, DSA_DEV_BAD_POOL_ID);
    } else if (p >= 0) {
      const int st = pool_start[base + p];
      if (st >= 0) tok = st + s;
    }
  }
  token_ids[(long long)q * W + c] = tok;
  pdl_launch_dependents();
}

int chunks_for(int Q, int P_ld) {
  const int target = 2 * kNumSMs;
  int c = (target + Q - 1) / Q;
  const int max_c = (P_ld + 1023) / 1024;
  if (c > max_c) c = max_c;
  return c < 1 ? 1 : c;
}

}  // namespace

size_t topk_workspace_size(int Q, int P_ld, int select_k) {
  (void)P_ld;
  return ws_header_bytes(Q) + align256((size_t)Q * select_k * 8) +
         align256((size_t)Q * kTieCap * 8);
}

int launch_topk_pools(const float* scores, int Q, int P_ld, int select_k, int32_t* pool_ids,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  (void)ws_bytes;
  TopkWs ws = carve(workspace, Q, select_k);
  if (cudaMemsetAsync(workspace, 0, ws_header_bytes(Q), stream) != cudaSuccess)
    return DSA_ERR_CUDA;
  const int chunks = chunks_for(Q, P_ld);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks, Q, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 0;  // follows a memset, not a kernel: plain stream order
  if (cudaLaunchKernelEx(&cfg, topk_hist_kernel, scores, P_ld, chunks, ws) != cudaSuccess)
    return DSA_ERR_CUDA;
  cfg.numAttrs = 1;
  const int kmax = select_k > kTieCap ? select_k : kTieCap;
  size_t smem = (size_t)kBins * 4 + kThreads * 4;
  const size_t final_smem = 2 * (size_t)kmax * 8;
  if (final_smem > smem) smem = final_smem;
  cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  cfg.dynamicSmemBytes = smem;
  if (cudaLaunchKernelEx(&cfg, topk_select_kernel, scores, P_ld, select_k, chunks, ws,
                         pool_ids) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}

int launch_expand_selection(const int32_t* pool_ids, const int32_t* pool_start,
                            const int32_t* cu_pool_cap, const int32_t* q_seq, int Q, int B,
                            int select_k, int kpool, int out_width, int32_t* token_ids,
                            int32_t* status_dev, cudaStream_t stream) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((out_width + 255) / 256, Q, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, expand_kernel, pool_ids, pool_start, cu_pool_cap, q_seq,
                                     B, select_k, kpool, out_width, token_ids, status_dev);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
