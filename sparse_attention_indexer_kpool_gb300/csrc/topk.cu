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
// A thread-block cluster of C CTAs per query row (C <= 16), everything on chip:
//   1. a 4096-bin histogram of the top 12 key bits (built by the scoring kernel
//      on the fused path; else each CTA counts its slice and every CTA sums the
//      C slice histograms through distributed shared memory);
//   2. the threshold bin, where the count from the top reaches select_k;
//   3. each CTA scans its slice of the row (8 loads in flight per thread): keys
//      above the bin go to its "sure" list, keys in it to its "tie" list;
//   4. every CTA all-gathers the cluster's lists over distributed shared
//      memory and places its own keys exactly: a sure key's output slot is the
//      number of larger sure keys; a tie key is selected when fewer than
//      select_k - #sure tie keys are larger, and sits after all sure keys (keys
//      are distinct, so these counts are the sorted positions; no sort runs);
//      if the tie lists overflow their on-chip capacity, rank 0 falls back to
//      an exact radix select over the row and a shared-memory sort;
//   5. pool ids written, and optionally expanded to token ids in place.
#include <cooperative_groups.h>

#include <map>
#include <mutex>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kBins = 4096;           // top 12 bits of the 32-bit score key
constexpr int kBinShift = 20;
constexpr int kTieCap = 4096;         // on-chip tie-list capacity (overflow: exact slow path)
constexpr int kThreads = 1024;
constexpr int kSmallSort = 1024;      // general path: rank sort up to this many keys

struct ExpandArgs {   // optional fused expand_selection (token_ids == nullptr: off)
  const int32_t* pool_start;
  const int32_t* cu_pool_cap;
  const int32_t* q_seq;
  int B, kpool, W;
  int32_t* token_ids;
  int32_t* status;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__device__ __forceinline__ uint64_t full_key(float s, int p) {
  return ((uint64_t)score_key(s) << 32) | (uint64_t)(0xffffffffu - (uint32_t)p);
}
__device__ __forceinline__ int key_pool(uint64_t key) {
  return (int)(0xffffffffu - (uint32_t)(key & 0xffffffffu));
}

// Block-wide (kThreads): threshold bin for K over hist h (smem).  *thr = -1
// when every candidate fits.
__device__ void find_threshold(const uint32_t* h, int K, int* s_thr, uint32_t* s_wtot) {
  constexpr int kPer = kBins / kThreads;  // 4 bins per thread
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) local += h[tid * kPer + i];
  uint32_t x = local;  // inclusive suffix sum inside the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) s_wtot[warp] = x;
  if (tid == 0) *s_thr = -1;
  __syncthreads();
  if (warp == 0) {  // exclusive suffix over warps
    const uint32_t v = s_wtot[lane];
    uint32_t z = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, z, o);
      if (lane + o < 32) z += y;
    }
    s_wtot[32 + lane] = z - v;
  }
  __syncthreads();
  const uint32_t incl = x + s_wtot[32 + warp];   // candidates in bins >= tid*kPer
  const uint32_t excl = incl - local;            // candidates in bins > tid*kPer + kPer-1
  const uint32_t total = s_wtot[32] + s_wtot[0];
  if (total > (uint32_t)K && excl < (uint32_t)K && incl >= (uint32_t)K) {
    uint32_t run = excl;
    for (int i = kPer - 1; i >= 0; --i) {
      const uint32_t c = h[tid * kPer + i];
      if (run + c >= (uint32_t)K) {
        *s_thr = tid * kPer + i;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
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

// Sort n keys in smem descending (general path); tmp has room for n keys.
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

// Shared-memory layout of the select kernel (dynamic).  Region A holds the
// per-slice state and is reused as sort scratch on the slow path; region B the
// gathered lists and the output ids.
//   A: h[kBins] | hsum[kBins] | own_sure[K] | own_tie[kTieCap]     (>= 2*max(K,kTieCap) keys)
//   B: all_sure[K] | all_tie[kTieCap] | ids[K]
struct SelLayout {
  size_t hsum, own_sure, own_tie, a_end, all_sure, all_tie, ids, total;
  __host__ __device__ SelLayout(int K) {
    const size_t kmax = (size_t)(K > kTieCap ? K : kTieCap);
    hsum = align256((size_t)kBins * 4);
    own_sure = hsum + align256((size_t)kBins * 4);
    own_tie = own_sure + align256((size_t)K * 8);
    a_end = own_tie + align256((size_t)kTieCap * 8);
    if (a_end < 2 * kmax * 8) a_end = align256(2 * kmax * 8);
    all_sure = a_end;
    all_tie = all_sure + align256((size_t)K * 8);
    ids = all_tie + align256((size_t)kTieCap * 8);
    total = ids + align256((size_t)K * 4);
  }
};

constexpr int kBatch = 8;  // row elements in flight per thread

namespace cg = cooperative_groups;

// Number of keys in list[0..n) larger than x, computed by `parts` cooperating
// lanes (a power of two <= 32, aligned in the warp); every lane gets the total.
__device__ __forceinline__ uint32_t count_larger(const uint64_t* list, uint32_t n, uint64_t x,
                                                 int part, int parts) {
  uint32_t c = 0;
  uint32_t j = part;
  for (; j + 3 * parts < n; j += 4 * parts)
    c += (list[j] > x) + (list[j + parts] > x) + (list[j + 2 * parts] > x) +
         (list[j + 3 * parts] > x);
  for (; j < n; j += parts) c += list[j] > x;
  for (int o = parts >> 1; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  return c;
}

__global__ void __launch_bounds__(kThreads, 1)
    topk_select_kernel(const float* __restrict__ scores, int P_ld, int K,
                       uint32_t* __restrict__ hist_in, int32_t* __restrict__ pool_ids,
                       ExpandArgs ex) {
  extern __shared__ __align__(256) unsigned char smem[];
  const SelLayout lay(K);
  uint32_t* h = reinterpret_cast<uint32_t*>(smem);
  uint32_t* hsum = reinterpret_cast<uint32_t*>(smem + lay.hsum);
  uint64_t* own_sure = reinterpret_cast<uint64_t*>(smem + lay.own_sure);
  uint64_t* own_tie = reinterpret_cast<uint64_t*>(smem + lay.own_tie);
  uint64_t* all_sure = reinterpret_cast<uint64_t*>(smem + lay.all_sure);
  uint64_t* all_tie = reinterpret_cast<uint64_t*>(smem + lay.all_tie);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + lay.ids);
  __shared__ int s_thr;
  __shared__ uint32_t s_nsure, s_ntie, s_r, s_nsel;
  __shared__ uint32_t s_wtot[64];
  __shared__ uint32_t s_cnt[2][17];  // per-rank sure / tie counts, exclusive prefix in [.][r]
  __shared__ uint64_t s_res;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int C = (int)cluster.num_blocks();
  const int q = blockIdx.y;
  const float* row = scores + (long long)q * P_ld;
  const int lo = (int)((long long)P_ld * rank / C);
  const int hi = (int)((long long)P_ld * (rank + 1) / C);
  if (threadIdx.x == 0) { s_nsure = 0; s_ntie = 0; }
  pdl_wait();
  pdl_launch_dependents();  // the next kernel may start its own prologue

  // The histogram (when the scoring kernel counted it), the first batch of this
  // CTA's slice and the expansion's sequence index are requested together, so
  // their latencies overlap; the sequence's cache slice, a load that depends on
  // that index and that only the placement needs, comes after the slice scan.
  uint32_t* gh = hist_in ? hist_in + (size_t)q * kBins : nullptr;
  constexpr int kHistPer = kBins / kThreads;  // 4 bins per thread
  uint32_t hv[kHistPer];
  if (gh) {
#pragma unroll
    for (int u = 0; u < kHistPer; ++u) hv[u] = __ldcg(gh + u * kThreads + threadIdx.x);
  }
  float v_first[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int i = lo + u * kThreads + threadIdx.x;
    v_first[u] = i < hi ? row[i] : -INFINITY;
  }
  const int b = ex.token_ids ? (ex.q_seq ? ex.q_seq[q] : 0) : 0;
  const bool seq_ok = !ex.token_ids || (b >= 0 && b < ex.B);
  // slice element i of the pass starting at `base` (the first batch is in registers)
  auto slice = [&](int base, int u) -> float {
    const int i = base + u * kThreads + threadIdx.x;
    return base == lo ? v_first[u] : (i < hi ? row[i] : -INFINITY);
  };

  // ---- 1. histogram of the top 12 key bits
  uint32_t* hh = h;
  if (gh) {
#pragma unroll
    for (int u = 0; u < kHistPer; ++u) h[u * kThreads + threadIdx.x] = hv[u];
    __syncthreads();
  } else {
    for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
    __syncthreads();
    for (int base = lo; base < hi; base += kThreads * kBatch) {
      float v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) v[u] = slice(base, u);
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (is_candidate(v[u])) atomicAdd(&h[score_key(v[u]) >> kBinShift], 1u);
    }
    if (C > 1) {
      cluster.sync();  // every slice histogram is complete
      for (int i = threadIdx.x; i < kBins; i += kThreads) {
        uint32_t t = 0;
        for (int r = 0; r < C; ++r) t += cluster.map_shared_rank(h, r)[i];
        hsum[i] = t;
      }
      hh = hsum;
    }
    __syncthreads();
  }
  // ---- 2. threshold bin
  find_threshold(hh, K, &s_thr, s_wtot);
  const int thr = s_thr;
  // ---- 3. this CTA's slice: sure and tie lists
  // A thread marks its batch's keys above and in the threshold bin; a scan
  // over the warp's counts and one shared atomic per warp and list reserve the
  // slots, so no atomic result is waited for per element.
  for (int base = lo; base < hi; base += kThreads * kBatch) {
    float v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) v[u] = slice(base, u);
    uint32_t sure_bits = 0, tie_bits = 0;  // bit u: element u goes to that list
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (is_candidate(v[u])) {
        const int bin = (int)(score_key(v[u]) >> kBinShift);
        sure_bits |= (uint32_t)(bin > thr) << u;
        tie_bits |= (uint32_t)(bin == thr) << u;
      }
    }
    const int lane = threadIdx.x & 31;
    const uint32_t cs = __popc(sure_bits), ct = __popc(tie_bits);
    uint32_t incl_s = cs, incl_t = ct;  // inclusive prefix inside the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t ys = __shfl_up_sync(0xffffffffu, incl_s, o);
      const uint32_t yt = __shfl_up_sync(0xffffffffu, incl_t, o);
      if (lane >= o) {
        incl_s += ys;
        incl_t += yt;
      }
    }
    const uint32_t warp_s = __shfl_sync(0xffffffffu, incl_s, 31);
    const uint32_t warp_t = __shfl_sync(0xffffffffu, incl_t, 31);
    uint32_t base_s = 0, base_t = 0;
    if (lane == 31) {
      if (warp_s) base_s = atomicAdd(&s_nsure, warp_s);
      if (warp_t) base_t = atomicAdd(&s_ntie, warp_t);
    }
    uint32_t slot_s = __shfl_sync(0xffffffffu, base_s, 31) + incl_s - cs;
    uint32_t slot_t = __shfl_sync(0xffffffffu, base_t, 31) + incl_t - ct;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (((sure_bits | tie_bits) >> u) & 1u) {
        const uint64_t key = full_key(v[u], base + u * kThreads + threadIdx.x);
        if ((sure_bits >> u) & 1u) {
          if (slot_s < (uint32_t)K) own_sure[slot_s] = key;
          ++slot_s;
        } else {
          if (slot_t < (uint32_t)kTieCap) own_tie[slot_t] = key;
          ++slot_t;
        }
      }
    }
  }
  const long long cap_base = (ex.token_ids && seq_ok) ? ex.cu_pool_cap[b] : 0;
  const int cap = (ex.token_ids && seq_ok) ? ex.cu_pool_cap[b + 1] - ex.cu_pool_cap[b] : 0;
  cluster.sync();  // every slice's lists and counts are final
  // ---- 4. all-gather the cluster's lists
  if (threadIdx.x < 2 * C) {
    const int r = threadIdx.x % C, which = threadIdx.x / C;
    s_cnt[which][r + 1] = *cluster.map_shared_rank(which ? &s_ntie : &s_nsure, r);
  }
  __syncthreads();
  if (threadIdx.x < 2) {
    s_cnt[threadIdx.x][0] = 0;
    for (int r = 0; r < C; ++r) s_cnt[threadIdx.x][r + 1] += s_cnt[threadIdx.x][r];
  }
  __syncthreads();
  const uint32_t n_sure = s_cnt[0][C], n_tie = s_cnt[1][C];
  const bool ties_fit = n_tie <= (uint32_t)kTieCap;
  {
    // one flat pass over (rank, element): every remote load is issued before any
    // local store, so the copy costs a single distributed-shared-memory round trip
    const uint32_t n_s = n_sure < (uint32_t)K ? n_sure : (uint32_t)K;
    const uint32_t n_all = n_s + (ties_fit ? n_tie : 0u);
    constexpr int kPer = 4;
    for (uint32_t base = 0; base < n_all; base += kThreads * kPer) {
      uint64_t v[kPer];
      uint32_t dst[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const uint32_t f = base + u * kThreads + threadIdx.x;
        dst[u] = 0xffffffffu;
        v[u] = 0;
        if (f < n_all) {
          const bool is_tie = f >= n_s;
          const uint32_t g = is_tie ? f - n_s : f;
          int r = 0;
          while (r + 1 < C && s_cnt[is_tie][r + 1] <= g) ++r;
          const uint64_t* src = cluster.map_shared_rank(is_tie ? own_tie : own_sure, r);
          v[u] = src[g - s_cnt[is_tie][r]];
          dst[u] = f;
        }
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        if (dst[u] == 0xffffffffu) continue;
        if (dst[u] < n_s) all_sure[dst[u]] = v[u];
        else all_tie[dst[u] - n_s] = v[u];
      }
    }
  }
  cluster.sync();  // every CTA has its copy: the others' shared memory may go away
  const int32_t* pstart = ex.pool_start;
  int32_t* out = pool_ids + (long long)q * K;
  int32_t* tok = ex.token_ids ? ex.token_ids + (long long)q * ex.W : nullptr;
  // writes one selected key's pool id and token ids at output slot `pos`
  // start of a selected pool's tokens (-1 when it cannot be expanded)
  auto pool_first_token = [&](uint64_t key) -> int {
    const int p = key_pool(key);
    return (tok && seq_ok && p < cap) ? pstart[cap_base + p] : -1;
  };
  // writes one selected key's pool id and token ids at output slot `pos`
  auto emit_with = [&](uint32_t pos, uint64_t key, int st) {
    const int p = key_pool(key);
    out[pos] = p;
    if (tok) {
      if (seq_ok && p >= cap) flag(ex.status, DSA_DEV_BAD_POOL_ID);
      for (int s = 0; s < ex.kpool; ++s) tok[pos * ex.kpool + s] = (st >= 0) ? st + s : -1;
    }
  };
  auto emit = [&](uint32_t pos, uint64_t key) { emit_with(pos, key, pool_first_token(key)); };
  // The lists are exactly the selection only if they agree with the histogram
  // (a workspace that was not zero-filled breaks that); otherwise rank 0 runs an
  // exact select that never looks at the histogram.
  const bool consistent = thr < 0 ? n_sure <= (uint32_t)K
                                  : (n_sure < (uint32_t)K && n_sure + n_tie >= (uint32_t)K);
  if (consistent && ties_fit) {
    const uint32_t n_sel = thr < 0 ? n_sure : (uint32_t)K;
    if (rank == 0) {  // the -1 tail of both outputs
      for (int j = n_sel + threadIdx.x; j < K; j += kThreads) out[j] = -1;
      if (tok)
        for (int c = n_sel * ex.kpool + threadIdx.x; c < ex.W; c += kThreads) tok[c] = -1;
      if (tok && !seq_ok && threadIdx.x == 0) flag(ex.status, DSA_DEV_BAD_QSEQ);
    }
    // ---- 5. place this CTA's own keys by counting larger keys
    const uint32_t my_s0 = s_cnt[0][rank], my_ns = s_cnt[0][rank + 1] - my_s0;
    const uint32_t my_t0 = s_cnt[1][rank], my_nt = thr < 0 ? 0 : s_cnt[1][rank + 1] - my_t0;
    const uint32_t n_own = my_ns + my_nt;
    const uint32_t R = thr < 0 ? 0 : (uint32_t)K - n_sure;
    int parts = 1;
    while (parts < 32 && (uint32_t)parts * 2 * n_own <= (uint32_t)kThreads) parts *= 2;
    for (uint32_t base = 0; base < n_own * parts; base += kThreads) {
      const uint32_t w = base + threadIdx.x;
      const uint32_t i = w / parts;
      const int part = (int)(w % parts);
      const bool act = i < n_own;
      const bool is_tie = i >= my_ns;
      uint64_t x = 0;
      if (act) x = is_tie ? all_tie[my_t0 + (i - my_ns)] : all_sure[my_s0 + i];
      // lanes of one key share a warp (parts divides 32); inactive lanes count
      // nothing; one call site, so every lane runs the same shuffles
      const uint64_t* lst = is_tie ? all_tie : all_sure;
      const uint32_t nl = act ? (is_tie ? n_tie : n_sure) : 0u;
      // the pool's first token is fetched before the count, so the two overlap
      const int st = (act && part == 0) ? pool_first_token(x) : -1;
      const uint32_t c = count_larger(lst, nl, x, part, parts);
      if (act && part == 0) {
        if (!is_tie) emit_with(c, x, st);
        else if (c < R) emit_with(n_sure + c, x, st);
      }
    }
  } else if (rank == 0) {
    // ---- 5'. exact select straight from the row (tie lists overflowed, or the
    // histogram did not describe these scores)
    if (!consistent && threadIdx.x == 0) flag(ex.status, DSA_DEV_HIST_MISMATCH);
    if (tok && !seq_ok && threadIdx.x == 0) flag(ex.status, DSA_DEV_BAD_QSEQ);
    uint64_t* sel = reinterpret_cast<uint64_t*>(smem);               // region A as scratch
    const int kmax = K > kTieCap ? K : kTieCap;
    uint64_t* tmp = sel + kmax;
    uint32_t* sh = reinterpret_cast<uint32_t*>(tmp);
    if (threadIdx.x == 0) s_nsel = 0;
    __syncthreads();
    uint32_t cnt = 0;
    for (int i = threadIdx.x; i < P_ld; i += kThreads) cnt += is_candidate(row[i]);
    atomicAdd(&s_nsel, cnt);
    __syncthreads();
    const uint32_t n_cand = s_nsel;
    const uint32_t n_sel = n_cand < (uint32_t)K ? n_cand : (uint32_t)K;
    __syncthreads();
    if (threadIdx.x == 0) s_nsel = 0;
    __syncthreads();
    if (n_sel > 0) {
      auto get = [&](int i, uint64_t& k) {
        const float sc = row[i];
        if (!is_candidate(sc)) return false;
        k = full_key(sc, i);
        return true;
      };
      const uint64_t T = radix_kth(P_ld, n_sel, get, sh, &s_res, &s_r);
      for (int i = threadIdx.x; i < P_ld; i += kThreads) {
        uint64_t k;
        if (get(i, k) && k >= T) {
          const uint32_t slot = atomicAdd(&s_nsel, 1u);
          if (slot < (uint32_t)K) sel[slot] = k;
        }
      }
      __syncthreads();
      sort_desc(sel, (int)n_sel, tmp);
    }
    for (int j = threadIdx.x; j < (int)n_sel; j += kThreads) emit(j, sel[j]);
    for (int j = n_sel + threadIdx.x; j < K; j += kThreads) out[j] = -1;
    if (tok)
      for (int c = n_sel * ex.kpool + threadIdx.x; c < ex.W; c += kThreads) tok[c] = -1;
  }
  if (gh && rank == 0)  // leave the histogram the scoring kernel filled zeroed for the next call
    for (int i = threadIdx.x; i < kBins; i += kThreads) gh[i] = 0;
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

// How many clusters of 16 top-k CTAs can be resident at once (per shared
// memory size; asked once).
int clusters16_resident(size_t smem) {
  static std::mutex mu;
  static std::map<size_t, int> known;
  std::lock_guard<std::mutex> lock(mu);
  const auto it = known.find(smem);
  if (it != known.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) == cudaSuccess &&
      cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) == cudaSuccess) {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeClusterDimension;
    a.val.clusterDim.x = 16;
    a.val.clusterDim.y = 1;
    a.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = &a;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, topk_select_kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();  // a refused query leaves no error behind
  known[smem] = n;
  return n;
}

int launch_select(const float* scores, int Q, int P_ld, int select_k, int32_t* pool_ids,
                  uint32_t* hist, const ExpandArgs& ex, cudaStream_t stream) {
  // cluster size: enough CTAs to spread a few rows over the SMs, a slice of at
  // least 4096 scores per CTA, at most 16 (16 is a non-portable size, taken
  // only when all Q clusters of 16 can be resident at once; measured on the
  // 4-query 262k step: 8 -> 16 CTAs per row, 0.459 -> 0.451 ms)
  const size_t smem = SelLayout(select_k).total;
  if (smem > 227 * 1024) return DSA_ERR_UNSUPPORTED;
  int C = 1;
  while (C < 16 && Q * C * 2 <= num_sms() && (long long)P_ld >= (long long)C * 2 * 4096) C *= 2;
  if (C == 16 && clusters16_resident(smem) < Q) C = 8;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, Q, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  cfg.dynamicSmemBytes = smem;
  return launch_kernel(&cfg, topk_select_kernel, scores, P_ld, select_k, hist, pool_ids,
                       ex) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

// Standalone top-k needs no workspace: the histogram lives on chip.  The fused
// select path keeps a [Q][4096] histogram in its workspace.
size_t topk_workspace_size(int Q, int P_ld, int select_k) {
  (void)Q; (void)P_ld; (void)select_k;
  return 0;
}
size_t select_workspace_size(int Q, int P_ld, int select_k) {
  (void)P_ld; (void)select_k;
  return align256((size_t)Q * kBins * 4);  // the per-query histograms
}

uint32_t* topk_workspace_hist(void* workspace) { return static_cast<uint32_t*>(workspace); }

int launch_topk_pools(const float* scores, int Q, int P_ld, int select_k, int32_t* pool_ids,
                      void* workspace, size_t ws_bytes, cudaStream_t stream) {
  (void)workspace; (void)ws_bytes;
  ExpandArgs ex = {};
  return launch_select(scores, Q, P_ld, select_k, pool_ids, nullptr, ex, stream);
}

int launch_select_after_index(const float* scores, int Q, int P_ld, int select_k,
                              int32_t* pool_ids, void* workspace, const int32_t* pool_start,
                              const int32_t* cu_pool_cap, const int32_t* q_seq, int B, int kpool,
                              int out_width, int32_t* token_ids, int32_t* status_dev,
                              cudaStream_t stream) {
  ExpandArgs ex = {pool_start, cu_pool_cap, q_seq, B, kpool, out_width, token_ids, status_dev};
  return launch_select(scores, Q, P_ld, select_k, pool_ids,
                       static_cast<uint32_t*>(workspace), ex, stream);
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
  cudaError_t e = launch_kernel(&cfg, expand_kernel, pool_ids, pool_start, cu_pool_cap, q_seq,
                                B, select_k, kpool, out_width, token_ids, status_dev);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
