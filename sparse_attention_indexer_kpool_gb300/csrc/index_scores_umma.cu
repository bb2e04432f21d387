// index_scores on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// score[q, p] = sum_h w[q, h] * max(0, scale * <q[q, h, :], key[p, :]>)   (module
// glm5next_dsa::tp, "Why the indexer is REPLICATED": a plain sum over heads of
// weights[h] * relu(scale * dot); module glm5next_dsa, "Shape of the pipeline":
// [Q, P] scores, -inf where a pool is not a candidate).  Geometry: bf16 keys and
// queries, 32 heads, head_dim 128.
//
// Swap-AB contraction: A = 128 pool keys (M = 128 -> TMEM lanes), B = G queries
// x 32 heads (N = 32 G -> TMEM columns), K = 128 channels in 8 steps of 16.
// G = 1 serves decode (one query per sequence, any q_seq); G = 8 serves a chunk
// of queries on one sequence (q_seq absent), the dense [Q*32, 128] x [128, P]
// prefill contraction, where one key tile feeds eight queries.
//
// One persistent CTA per SM owns a balanced contiguous range of the flattened
// (query group, 128-pool tile) space.  Warp roles:
//   warp 0     TMA producer: per query group, the query block (B, two 64-channel
//              boxes, 128-byte swizzle) and its head weights; then the group's
//              key tiles (A, two boxes of 128 rows x 64 channels) into a ring;
//   warp 1     MMA issuer: one thread issues 8 tcgen05.mma per tile into one of
//              two TMEM accumulators, then commits to the ring slot's "empty"
//              barrier and the accumulator's "full" barrier;
//   warps 2-9  epilogue: tcgen05.ld of the accumulator rows (a warp reads the 32
//              TMEM lanes of its quarter), relu / weight / head sum in registers
//              (scale folded into the weights once per query group),
//              -0 -> +0, candidate mask, coalesced score stores and (decode) a
//              4096-bin histogram of the score keys' top 12 bits for the top-k
//              that follows.  For G = 1 the two halves of the epilogue take
//              alternate tiles (one accumulator each); for G = 8 each half takes
//              four of the eight queries of every tile;
//   warp 10    (fused decode call only) the call's compress of one new pool per
//              sequence, with the compress kernels' own per-pool code; the
//              producer and the epilogue wait for it, on an in-CTA barrier,
//              only at the tile that holds the new pool.
// Every mbarrier wait is bounded.  On a timeout the kernel flags DSA_DEV_TIMEOUT,
// stops issuing work, waits (bounded) for its own copies and MMAs in flight and
// frees its TMEM before it returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "compress_pool.cuh"
#include "dsa_internal.cuh"
#include "umma.cuh"

namespace dsa {
namespace {

constexpr int kD = 128, kH = 32;
constexpr int kBM = 128;                       // pools per tile (MMA M)
constexpr int kABytes = kBM * kD * 2;          // 32 KB key tile
constexpr int kHalfA = kBM * 64 * 2;           // one 64-channel box of it
constexpr int kEpiWarps = 8;
constexpr int kCompressWarp = 2 + kEpiWarps;  // the decode compress, when the call fuses it
constexpr int kThreadsU = (3 + kEpiWarps) * 32;
constexpr int kHistBins = 4096;
constexpr int kSmemMax = 227 * 1024;
constexpr int kBaseCache = 4096;               // groups whose cache base is kept on chip

template <int G>
struct Cfg {
  static constexpr int N = 32 * G;                         // MMA N: queries x heads
  // key tile ring; decode step measured with 2 / 3 / 4 / 5 stages: 0.428 /
  // 0.414 / 0.418 / 0.429 ms (more tiles in flight per SM do not stream faster)
  static constexpr int kStages = 3;
  static constexpr int kBSlots = G == 1 ? 2 : 1;           // query blocks in flight
  static constexpr int kBBytes = N * kD * 2;
  static constexpr int kTmemCols = 2 * N < 32 ? 32 : 2 * N;  // two accumulators
  static constexpr int kTileWarps = G == 1 ? 4 : 8;        // epilogue warps per tile
  static_assert((2 * N & (2 * N - 1)) == 0, "TMEM allocation must be a power of two");
};

struct Ctl {
  uint64_t full[4], empty[4];      // key tile ring
  uint64_t bfull[2], bempty[2];    // query block slots
  uint64_t tfull[2], tempty[2];    // TMEM accumulators
  uint64_t done;                   // all MMAs of the CTA retired
  uint64_t cdone;                  // the compress warp's pools are written
  uint32_t tmem_base;
  int abort;
  int scan_warp[kThreadsU / 32];   // tile prefix scan: per-warp totals and carry
  int scan_carry;
};

// Shared-memory layout (offsets from a 1 KB-aligned base): the swizzled tiles
// first, each on a 1 KB boundary as the 128-byte swizzle atoms require.
template <int G>
struct Layout {
  static constexpr size_t a = 0;
  static constexpr size_t b = (size_t)Cfg<G>::kStages * kABytes;
  static constexpr size_t ctl = b + (size_t)Cfg<G>::kBSlots * Cfg<G>::kBBytes;
  static constexpr size_t w = ctl + ((sizeof(Ctl) + 15) & ~size_t(15));
  static constexpr size_t hist = w + (size_t)Cfg<G>::kBSlots * G * kH * 4;
  static constexpr size_t base = hist + (G == 1 ? (size_t)kHistBins * 4 : 0);
  // cache bases, then (early start) the safe tile counts and the pool counts
  // found from the compress's inputs, then the tile prefix
  __host__ __device__ static size_t cached(int n_groups) {
    return (size_t)(n_groups < kBaseCache ? n_groups : kBaseCache);
  }
  __host__ __device__ static size_t prefix(int n_groups, bool early) {
    return base + cached(n_groups) * 4 * (early ? 3 : 1);
  }
  static size_t bytes(int n_groups, bool early) {
    return 1024 + prefix(n_groups, early) + (size_t)(n_groups + 1) * 4;
  }
};

struct QMeta {
  long long base;  // first cache row of the query's sequence
  int n_cand;      // pools [0, n_cand) may be candidates
  int pos;         // query position (causal rule) or INT_MAX
  int valid;       // the query exists and its sequence id is in range
};

// Candidate range of query qi (as the other index kernels define it).
// np_known >= 0 stands in for n_pools[b] (the same value, found before the
// kernel that writes n_pools has ended).
__device__ __forceinline__ QMeta qmeta(int qi, int Q, const int32_t* q_seq, const int32_t* q_pos,
                                       const int32_t* n_pools, const int32_t* cu_pool_cap,
                                       const int32_t* pool_start, int B, int kpool, int P_ld,
                                       int32_t* status, bool report, int np_known = -1) {
  QMeta m{0, 0, 0x7fffffff, 0};
  if (qi >= Q) return m;
  const int b = q_seq ? q_seq[qi] : 0;
  if (b < 0 || b >= B) {
    if (report) flag(status, DSA_DEV_BAD_QSEQ);
    return m;
  }
  m.valid = 1;
  m.base = cu_pool_cap[b];
  const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
  const int np = np_known >= 0 ? np_known : n_pools[b];
  int P = min(np, min(cap, P_ld));
  if (np > P && report) flag(status, DSA_DEV_POOL_RANGE);
  P = max(P, 0);
  if (q_pos != nullptr && P > 0) {
    // pool p is complete at pos when t0 + p*kpool + kpool - 1 <= pos
    m.pos = q_pos[qi];
    const long long t0 = pool_start[m.base];
    const long long nv = (m.pos - t0 + 1) >= 0 ? (m.pos - t0 + 1) / kpool : 0;
    P = (int)min((long long)P, nv);
  }
  m.n_cand = P;
  return m;
}

// The pool count that the compress of the same call writes for sequence b:
// min((T - t0) / kpool, cap), t0 its first valid token (T when it has none).
// Found when t0 lies among the first kScanTokens tokens or the sequence is no
// longer than that, else -1.  Called by a whole warp; every lane gets the value.
constexpr int kScanTokens = 256;
__device__ __forceinline__ int early_pool_count(const EarlyStart& es, int b, int cap, int kpool,
                                                int lane) {
  const long long lo = es.cu_seqlens[b];
  const int T = es.cu_seqlens[b + 1] - es.cu_seqlens[b];
  if (es.k != nullptr)  // the call's compress is in this kernel: scan the whole sequence
    return min((T - first_valid_warp(es.valid, lo, T, lane)) / kpool, cap);
  const int lim = min(T, kScanTokens);
  uint32_t nz[kScanTokens / 32];
#pragma unroll
  for (int j = 0; j < kScanTokens / 32; ++j) {  // every load first, then the votes
    const int t = j * 32 + lane;
    nz[j] = t < lim ? es.valid[lo + t] : 0u;
  }
  int t0 = -1;
#pragma unroll
  for (int j = 0; j < kScanTokens / 32; ++j) {
    const uint32_t m = __ballot_sync(0xffffffffu, nz[j] != 0u);
    if (t0 < 0 && m != 0u) t0 = j * 32 + __ffs((int)m) - 1;
  }
  if (t0 < 0 && T <= kScanTokens) t0 = T;
  return t0 < 0 ? -1 : min((T - t0) / kpool, cap);
}

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}
// Bounded wait that also gives up at once after another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              int32_t* status, unsigned long long limit_ns) {
  if (*abort) return false;
  if (mbar_wait_bounded(bar, parity, limit_ns)) return true;
  flag(status, DSA_DEV_TIMEOUT);
  *abort = 1;
  return false;
}

template <int G>
__global__ void __launch_bounds__(kThreadsU, 1)
    index_scores_umma_kernel(const __grid_constant__ CUtensorMap tmap_keys,
                             const __grid_constant__ CUtensorMap tmap_q,
                             const float* __restrict__ wts, float scale,
                             const int32_t* __restrict__ pool_start,
                             const uint8_t* __restrict__ pool_valid,
                             const int32_t* __restrict__ n_pools,
                             const int32_t* __restrict__ cu_pool_cap,
                             const int32_t* __restrict__ q_seq, const int32_t* __restrict__ q_pos,
                             int Q, int B, int kpool, int P_ld, float* __restrict__ scores,
                             uint32_t* __restrict__ hist, const EarlyStart es, int drill,
                             int32_t* status) {
  using C = Cfg<G>;
  using LY = Layout<G>;
  constexpr int N = C::N;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sbase = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Ctl& ctl = *reinterpret_cast<Ctl*>(sbase + LY::ctl);
  float* s_w = reinterpret_cast<float*>(sbase + LY::w);
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(sbase + LY::hist);
  const int n_groups = (Q + G - 1) / G;
  // Early start (decode, inside one call after the compress of pools
  // [es.pool_begin[b], ...)): the tile plan comes from the call's inputs only;
  // the key tiles below pool_begin[b], which that compress does not write, are
  // streamed and scored before the compress has finished, with the pool count
  // found from the compress's own inputs.  Fused (es.k set), that compress is
  // warp 10 of this kernel, which is then the call's first kernel.
  const bool early = G == 1 && es.pool_begin != nullptr;
  // the compress of the call runs in this kernel (see EarlyStart)
  const bool fused = early && es.k != nullptr;
  int* s_base = reinterpret_cast<int*>(sbase + LY::base);  // first cache row of group gi
  int* s_safe = s_base + LY::cached(n_groups);             // early: tiles readable at once
  int* s_np = s_safe + LY::cached(n_groups);               // early: pool count, or -1
  int* s_prefix = reinterpret_cast<int*>(sbase + LY::prefix(n_groups, early));
  volatile int* abort = &ctl.abort;
  const bool use_hist = G == 1 && hist != nullptr;
  // a failure drill loads nothing and arms no barrier: the first waits run out
  const unsigned long long wait_ns = drill ? kDrillWaitNs : kWaitNs;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return wait_or_abort(bar, parity, abort, status, wait_ns);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&ctl.bfull[j], 1);
      mbar_init(&ctl.bempty[j], 1 + kEpiWarps);  // the MMA commit + every epilogue warp
      mbar_init(&ctl.tfull[j], 1);
      mbar_init(&ctl.tempty[j], C::kTileWarps);
    }
    mbar_init(&ctl.done, 1);
    mbar_init(&ctl.cdone, 1);
    fence_mbar_init();
    ctl.abort = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_keys))
                 : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_q))
                 : "memory");
  }
  if (warp == 1) {  // two accumulators of N fp32 columns
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl.tmem_base)),
                 "n"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  if (use_hist)
    for (int i = threadIdx.x; i < kHistBins; i += kThreadsU) s_hist[i] = 0;
  if (!early || fused) {
    pdl_wait();  // the pool cache may come from the kernel just before
    pdl_launch_dependents();
  }

  // ---- tiles per query group (its widest candidate range) and their prefix sum
  {
    int* s_warp = ctl.scan_warp;
    int& s_carry = ctl.scan_carry;
    if (threadIdx.x == 0) {
      s_prefix[0] = 0;
      s_carry = 0;
    }
    __syncthreads();
    for (int c0 = 0; c0 < n_groups; c0 += kThreadsU) {
      const int gi = c0 + threadIdx.x;
      int n = 0;
      if (gi < n_groups && early) {
        // every pool of the sequence's slice that a score row can hold
        const int b = q_seq ? q_seq[gi] : 0;
        int nt = 0, safe = 0;
        long long base = 0;
        if (b >= 0 && b < B) {
          base = cu_pool_cap[b];
          const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
          nt = (max(0, min(cap, P_ld)) + kBM - 1) / kBM;
          safe = min(nt, max(0, es.pool_begin[b]) / kBM);
        } else if (blockIdx.x == 0) {
          flag(status, DSA_DEV_BAD_QSEQ);
        }
        s_base[gi] = (int)base;
        s_safe[gi] = safe;
        n = nt;
      } else if (gi < n_groups) {
        int mx = 0;
        for (int u = 0; u < G; ++u) {
          const QMeta m = qmeta(gi * G + u, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B,
                                kpool, P_ld, status, blockIdx.x == 0);
          mx = max(mx, m.n_cand);
          if (u == 0 && gi < kBaseCache) s_base[gi] = (int)m.base;
        }
        n = (mx + kBM - 1) / kBM;
      }
      int x = n;  // inclusive warp scan
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) s_warp[warp] = x;
      __syncthreads();
      int off = s_carry;
      for (int w = 0; w < warp; ++w) off += s_warp[w];
      if (gi < n_groups) s_prefix[gi + 1] = off + x;
      __syncthreads();
      if (threadIdx.x == kThreadsU - 1) s_carry = off + x;
      __syncthreads();
    }
  }
  tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const long long NT = s_prefix[n_groups];
  const long long t_lo = NT * blockIdx.x / gridDim.x;
  const long long t_hi = NT * (blockIdx.x + 1) / gridDim.x;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0 && drill == 0) {
      // decode reads every key once: keep the call's other data in L2 instead; in a
      // chunk every query group rereads every key tile, so there the keys stay
      const uint64_t keys_policy = G == 1 ? l2_policy_evict_first() : l2_policy_evict_last();
      uint32_t a_par = 0, a_used = 0;  // per ring slot: parity of its next fill, ever filled
      uint32_t b_par = 0, b_used = 0;  // the same for the query block slots
      int stage = 0, gi = 0, seg = 0;
      bool waited = !early;            // the compress before this kernel is complete
      for (long long t = t_lo; t < t_hi && !*abort; ++seg) {
        while (s_prefix[gi + 1] <= t) ++gi;
        const long long seg_hi = min(t_hi, (long long)s_prefix[gi + 1]);
        const int slot = seg % C::kBSlots;
        if (((b_used >> slot) & 1) &&
            !wait(&ctl.bempty[slot], ((b_par >> slot) & 1) ^ 1))
          break;
        const long long base0 =
            gi < kBaseCache ? (long long)s_base[gi]
                            : qmeta(gi * G, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B,
                                    kpool, P_ld, status, false).base;
        const int nq = min(G, Q - gi * G);
        unsigned char* bt = sbase + LY::b + (size_t)slot * C::kBBytes;
        mbar_arrive_expect_tx(&ctl.bfull[slot], C::kBBytes + nq * kH * 4);
        tma_load_2d(bt, &tmap_q, 0, gi * N, &ctl.bfull[slot]);
        tma_load_2d(bt + N * 128, &tmap_q, 64, gi * N, &ctl.bfull[slot]);
        bulk_g2s(s_w + slot * G * kH, wts + (long long)gi * G * kH, nq * kH * 4,
                 &ctl.bfull[slot]);
        b_par ^= 1u << slot;
        b_used |= 1u << slot;
        for (; t < seg_hi; ++t) {
          if (((a_used >> stage) & 1) &&
              !wait(&ctl.empty[stage], ((a_par >> stage) & 1) ^ 1))
            break;
          if (!waited && t - s_prefix[gi] >= s_safe[gi]) {
            // this tile may hold a pool the compress rewrites
            if (fused) {
              if (!wait(&ctl.cdone, 0)) break;
            } else {
              pdl_wait();
            }
            waited = true;
          }
          const int row = (int)(base0 + (t - s_prefix[gi]) * kBM);
          unsigned char* at = sbase + LY::a + (size_t)stage * kABytes;
          mbar_arrive_expect_tx(&ctl.full[stage], kABytes);
          tma_load_2d_hint(at, &tmap_keys, 0, row, &ctl.full[stage], keys_policy);
          tma_load_2d_hint(at + kHalfA, &tmap_keys, 64, row, &ctl.full[stage], keys_policy);
          a_par ^= 1u << stage;
          a_used |= 1u << stage;
          stage = stage + 1 == C::kStages ? 0 : stage + 1;
        }
        if (t < seg_hi) break;  // aborted inside the segment
      }
      // Never leave a copy in flight: wait for the last fill of every slot.
      for (int s = 0; s < C::kStages; ++s)
        if ((a_used >> s) & 1) mbar_wait_bounded(&ctl.full[s], ((a_par >> s) & 1) ^ 1);
      for (int s = 0; s < C::kBSlots; ++s)
        if ((b_used >> s) & 1) mbar_wait_bounded(&ctl.bfull[s], ((b_par >> s) & 1) ^ 1);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kBM, N, false);
      uint32_t a_par = 0;  // per ring slot: parity of its next "full" phase
      int stage = 0, gi = 0, seg = 0;
      long long tc = 0;    // tiles issued by this CTA
      for (long long t = t_lo; t < t_hi && !*abort; ++seg) {
        while (s_prefix[gi + 1] <= t) ++gi;
        const long long seg_hi = min(t_hi, (long long)s_prefix[gi + 1]);
        const int slot = seg % C::kBSlots;
        if (!wait(&ctl.bfull[slot], (seg / C::kBSlots) & 1)) break;
        const uint32_t b_lo = smem_u32(sbase + LY::b + (size_t)slot * C::kBBytes);
        const uint32_t b_hi = b_lo + N * 128;
        for (; t < seg_hi; ++t, ++tc) {
          const int acc = (int)(tc & 1);
          if (!wait(&ctl.full[stage], (a_par >> stage) & 1)) break;
          a_par ^= 1u << stage;
          if (tc >= 2 &&  // the epilogue has drained this accumulator's previous tile
              !wait(&ctl.tempty[acc], (uint32_t)((tc >> 1) - 1) & 1))
            break;
          tc_fence_after();
          const uint32_t a_lo = smem_u32(sbase + LY::a + (size_t)stage * kABytes);
          const uint32_t a_hi = a_lo + kHalfA;
          const uint32_t d = tmem + (uint32_t)(acc * N);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (uint32_t)(kk & 3) * 32;  // 16 channels = 32 bytes
            umma_bf16(d, sw128_desc((kk < 4 ? a_lo : a_hi) + off),
                      sw128_desc((kk < 4 ? b_lo : b_hi) + off), idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&ctl.empty[stage]);  // the key tile may be refilled
          umma_commit(&ctl.tfull[acc]);    // the accumulator is ready
          stage = stage + 1 == C::kStages ? 0 : stage + 1;
        }
        if (t < seg_hi) break;
        umma_commit(&ctl.bempty[slot]);  // no more MMAs read this query block
      }
      umma_commit(&ctl.done);  // retire every MMA before TMEM is freed
      mbar_wait_bounded(&ctl.done, 0);
    }
  } else if (warp < kCompressWarp) {
    // ================= epilogue =================
    constexpr int GH = G == 1 ? 1 : G / 2;  // queries per warp of each tile
    const int ew = warp - 2;                // 0..7
    const int quarter = warp & 3;           // the TMEM lanes this warp may read
    const int half = ew >> 2;
    const int r = quarter * 32 + lane;      // pool row within the tile
    const int qw0 = G == 1 ? 0 : half * GH; // this warp's first query of the group
    bool waited = !early;  // the compress of this call has ended
    if (early) {
      // A kernel after the first of its call may let its dependents launch
      // before its own wait: it was itself launched by the trigger of a kernel
      // that had waited, so nothing enqueued before the call is still running.
      pdl_launch_dependents();
      // the pool count of every sequence this CTA scores: with it, the tiles
      // below pool_begin need nothing that the compress writes
      if (t_lo < t_hi) {
        int g_lo = 0;
        while (s_prefix[g_lo + 1] <= t_lo) ++g_lo;
        int g_hi = g_lo;
        while (g_hi + 1 < n_groups && s_prefix[g_hi + 1] < t_hi) ++g_hi;
        for (int g = g_lo + ew; g <= g_hi; g += kEpiWarps) {
          const int b = q_seq ? q_seq[g] : 0;
          const int np = (b >= 0 && b < B) ? early_pool_count(es, b,
                                                              cu_pool_cap[b + 1] - cu_pool_cap[b],
                                                              kpool, lane)
                                           : -1;
          if (lane == 0) s_np[g] = np;
        }
      }
      epi_bar();
    }
    int gi = 0, seg = 0;
    long long tc = 0;
    for (long long t = t_lo; t < t_hi; ++seg) {
      while (s_prefix[gi + 1] <= t) ++gi;
      const long long seg_hi = min(t_hi, (long long)s_prefix[gi + 1]);
      const int slot = seg % C::kBSlots;
      int np_known = -1;
      if (early) {
        np_known = s_np[gi];
        if (np_known < 0 && !waited) {  // not found from the inputs: read what the compress wrote
          pdl_wait();
          waited = true;
        }
      }
      QMeta mq[GH];
      int ncmax = 0;
#pragma unroll
      for (int u = 0; u < GH; ++u) {
        mq[u] = qmeta(gi * G + qw0 + u, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B,
                      kpool, P_ld, status, false, np_known);
        ncmax = max(ncmax, mq[u].n_cand);
      }
      const long long base = mq[0].base;  // every query of a group reads one sequence
      const bool b_ok = wait(&ctl.bfull[slot], (seg / C::kBSlots) & 1);
      float* wq = s_w + slot * G * kH;
      // fold scale into the weights once per group: w * max(0, scale * dot) equals
      // (w * scale) * max(0, dot) for scale > 0 (up to rounding)
      if (b_ok && ew * 32 + lane < G * kH) wq[ew * 32 + lane] *= scale;
      epi_bar();
      for (; t < seg_hi; ++t, ++tc) {
        const int acc = (int)(tc & 1);
        if (G == 1 && acc != half) continue;  // the other half's tile
        if (!waited && t - s_prefix[gi] >= s_safe[gi]) {  // a tile the compress may rewrite
          if (fused)
            (void)wait(&ctl.cdone, 0);
          else
            pdl_wait();
          waited = true;
        }
        const int p = (int)(t - s_prefix[gi]) * kBM + r;
        // candidate metadata first: its latency hides behind the accumulator wait
        uint8_t pv = 0;
        int ps = 0;
        if (p < ncmax) {
          pv = pool_valid[base + p];
          if (q_pos != nullptr) ps = pool_start[base + p];
        }
        if (!b_ok || !wait(&ctl.tfull[acc], (uint32_t)(tc >> 1) & 1))
          continue;  // keep walking so that every warp meets the same barriers
        tc_fence_after();
        const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * N);
        // the score of query u at this row: sum over the heads in order
        auto put = [&](int u, float sc) {
          if (sc == 0.f) sc = 0.f;  // -0 -> +0
          const QMeta& m = mq[u];
          if (m.valid && p < P_ld) {
            bool cand = p < m.n_cand && pv != 0;
            if (cand && q_pos != nullptr) cand = ps + kpool - 1 <= m.pos;
            scores[(long long)(gi * G + qw0 + u) * P_ld + p] = cand ? sc : -INFINITY;
            if (use_hist && cand) atomicAdd(&s_hist[score_key(sc) >> 20], 1u);
          }
        };
        if constexpr (GH % 2 == 0) {
          // two queries at a time: both loads before one wait, two independent
          // sums (each in head order, as below)
#pragma unroll
          for (int u = 0; u < GH; u += 2) {
            float va[32], vb[32];
            tmem_ld32x2(tb + (uint32_t)((qw0 + u) * kH), tb + (uint32_t)((qw0 + u + 1) * kH), va,
                        vb);
            const float4* wa4 = reinterpret_cast<const float4*>(wq + (qw0 + u) * kH);
            const float4* wb4 = reinterpret_cast<const float4*>(wq + (qw0 + u + 1) * kH);
            // packed fp32 FMA: even and odd heads in the two halves, added last
            unsigned long long sa2 = 0ull, sb2 = 0ull;
            auto ffma2 = [](unsigned long long acc, float w0, float w1, float x0, float x1) {
              unsigned long long w, x, d;
              asm("mov.b64 %0, {%1, %2};" : "=l"(w) : "f"(w0), "f"(w1));
              asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
              asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(w), "l"(x), "l"(acc));
              return d;
            };
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 wa = wa4[i], wb = wb4[i];
              sa2 = ffma2(sa2, wa.x, wa.y, fmaxf(va[4 * i + 0], 0.f), fmaxf(va[4 * i + 1], 0.f));
              sb2 = ffma2(sb2, wb.x, wb.y, fmaxf(vb[4 * i + 0], 0.f), fmaxf(vb[4 * i + 1], 0.f));
              sa2 = ffma2(sa2, wa.z, wa.w, fmaxf(va[4 * i + 2], 0.f), fmaxf(va[4 * i + 3], 0.f));
              sb2 = ffma2(sb2, wb.z, wb.w, fmaxf(vb[4 * i + 2], 0.f), fmaxf(vb[4 * i + 3], 0.f));
            }
            float a0, a1, b0, b1;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(sa2));
            asm("mov.b64 {%0, %1}, %2;" : "=f"(b0), "=f"(b1) : "l"(sb2));
            put(u, a0 + a1);
            put(u + 1, b0 + b1);
          }
        } else {
#pragma unroll
          for (int u = 0; u < GH; ++u) {
            float v[32];
            tmem_ld32(tb + (uint32_t)((qw0 + u) * kH), v);
            const float4* w4 = reinterpret_cast<const float4*>(wq + (qw0 + u) * kH);
            float sc = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 w = w4[i];
              sc = fmaf(w.x, fmaxf(v[4 * i + 0], 0.f), sc);
              sc = fmaf(w.y, fmaxf(v[4 * i + 1], 0.f), sc);
              sc = fmaf(w.z, fmaxf(v[4 * i + 2], 0.f), sc);
              sc = fmaf(w.w, fmaxf(v[4 * i + 3], 0.f), sc);
            }
            put(u, sc);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive1(&ctl.tempty[acc]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive1(&ctl.bempty[slot]);  // done with this query block's weights
      if (use_hist) {  // flush this query's histogram
        epi_bar();
        uint32_t* gh = hist + (size_t)gi * kHistBins;
        // 16 bins per thread as four 16-byte reads, all issued before any add
        static_assert(kHistBins == 16 * kEpiWarps * 32, "four 16-byte groups of bins per thread");
        const int et = ew * 32 + lane;
        uint4 hv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          hv[k] = reinterpret_cast<const uint4*>(s_hist)[k * kEpiWarps * 32 + et];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i0 = 4 * (k * kEpiWarps * 32 + et);
          if (hv[k].x) atomicAdd(&gh[i0], hv[k].x);
          if (hv[k].y) atomicAdd(&gh[i0 + 1], hv[k].y);
          if (hv[k].z) atomicAdd(&gh[i0 + 2], hv[k].z);
          if (hv[k].w) atomicAdd(&gh[i0 + 3], hv[k].w);
          if (hv[k].x | hv[k].y | hv[k].z | hv[k].w)
            reinterpret_cast<uint4*>(s_hist)[k * kEpiWarps * 32 + et] = make_uint4(0, 0, 0, 0);
        }
        epi_bar();
      }
    }
    if (early) {
      // every CTA ends after the compress, so that the end of this kernel
      // implies the end of the compress for whatever waits on it (a fused
      // compress is part of this CTA)
      if (!waited && !fused) pdl_wait();
      if (blockIdx.x == 0 && !fused)  // the range checks the tile plan skipped
        for (int qi = ew * 32 + lane; qi < Q; qi += kEpiWarps * 32)
          qmeta(qi, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool, P_ld, status,
                true);
      if (blockIdx.x == 0 && fused)  // the same, with the pool counts found from the inputs
        for (int qi = ew; qi < Q; qi += kEpiWarps) {
          const int b = q_seq ? q_seq[qi] : 0;
          const int np = (b >= 0 && b < B)
                             ? early_pool_count(es, b, cu_pool_cap[b + 1] - cu_pool_cap[b],
                                                kpool, lane)
                             : 0;
          if (lane == 0)
            qmeta(qi, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool, P_ld, status,
                  true, np);
        }
    }
  } else if (fused) {
    // ================= compress warp (the call's one new pool per sequence) =================
    // Sequences of the tiles in this CTA's range that may hold a rewritten
    // pool, and every gridDim.x-th sequence that no query's tiles cover (its
    // cache is updated all the same).  Two CTAs that share a sequence write
    // the same bytes.
    auto compress_seq = [&](int b) {
      const long long lo = es.cu_seqlens[b];
      const int Tb = es.cu_seqlens[b + 1] - es.cu_seqlens[b];
      const long long cap_lo = cu_pool_cap[b];
      const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
      const int begin = es.pool_begin[b];
      const int end = (int)min((long long)begin + 1, (long long)cap);
      const int t0 = first_valid_warp(es.valid, lo, Tb, lane);
      const int P = (Tb - t0) / kpool;
      const int P_eff = min(P, cap);
      if (lane == 0) {
        es.n_pools_out[b] = P_eff;
        if (P > cap) flag(status, DSA_DEV_POOL_OVERFLOW);
        if (P_eff > end) flag(status, DSA_DEV_POOL_UNCOVERED);
      }
      const int p = begin;
      if (p < 0 || p >= end) return;
      __nv_bfloat16* out = es.pool_keys_out + (cap_lo + p) * kD + lane * 4;
      if (p >= P_eff)
        compress_sentinel_warp<__nv_bfloat16, 4>(lane, out, es.pool_start_out + cap_lo + p,
                                                 es.pool_valid_out + cap_lo + p);
      else
        compress_pool_warp<__nv_bfloat16, 4>(es.k, es.gate, es.valid, es.ape, es.ln_gamma,
                                             es.ln_beta, es.ln_eps,
                                             lo + t0 + (long long)p * kpool, kpool, lane, out,
                                             t0 + p * kpool, es.pool_start_out + cap_lo + p,
                                             es.pool_valid_out + cap_lo + p);
    };
    for (int gi = 0; gi < n_groups; ++gi) {
      const long long u0 = (long long)s_prefix[gi] + s_safe[gi], u1 = s_prefix[gi + 1];
      const int b = q_seq ? q_seq[gi] : 0;
      if (u0 < u1 && max(u0, t_lo) < min(u1, t_hi) && b >= 0 && b < B) compress_seq(b);
    }
    for (int b = blockIdx.x; b < B; b += gridDim.x) {
      bool covered = false;
      for (int gi = 0; gi < n_groups && !covered; ++gi)
        covered = (q_seq ? q_seq[gi] : 0) == b && s_safe[gi] < s_prefix[gi + 1] - s_prefix[gi];
      if (!covered) compress_seq(b);
    }
    // the writes above are read by this CTA's TMA loads and by its epilogue
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence_block();
    __syncwarp();
    if (lane == 0) mbar_arrive1(&ctl.cdone);
  }

  // Fill the rest of each row (pools past every tile of its group) with -inf.
  if (n_groups >= (int)gridDim.x) {
    for (int gi = blockIdx.x; gi < n_groups; gi += gridDim.x) {
      const long long start = (long long)(s_prefix[gi + 1] - s_prefix[gi]) * kBM;
      for (int u = 0; u < G && gi * G + u < Q; ++u) {
        float* row = scores + (long long)(gi * G + u) * P_ld;
        for (long long i = start + threadIdx.x; i < P_ld; i += kThreadsU) row[i] = -INFINITY;
      }
    }
  } else {
    const long long gtid = (long long)blockIdx.x * kThreadsU + threadIdx.x;
    const long long gstride = (long long)gridDim.x * kThreadsU;
    for (int gi = 0; gi < n_groups; ++gi) {
      const long long start = (long long)(s_prefix[gi + 1] - s_prefix[gi]) * kBM;
      for (int u = 0; u < G && gi * G + u < Q; ++u) {
        float* row = scores + (long long)(gi * G + u) * P_ld;
        for (long long i = start + gtid; i < P_ld; i += gstride) row[i] = -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(C::kTmemCols)
                 : "memory");
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// [rows, 128] bf16 row-major matrix, boxes of 64 channels x box_rows rows,
// 128-byte swizzle; rows at or beyond `rows` read as zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int G>
int launch_g(const void* q, const float* weights, float scale, const void* pool_keys,
             int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
             const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
             const int32_t* q_pos, int Q, int B, int kpool, int P_ld, float* scores,
             uint32_t* hist, const EarlyStart& es, int32_t* status, cudaStream_t stream,
             int busy_ctas) {
  const size_t smem = Layout<G>::bytes((Q + G - 1) / G, es.pool_begin != nullptr);
  if (smem > (size_t)kSmemMax) return DSA_ERR_UNSUPPORTED;
  CUtensorMap mk, mq;
  if (!make_map(&mk, pool_keys, (uint64_t)pool_rows, kBM)) return DSA_ERR_CUDA;
  if (!make_map(&mq, q, (uint64_t)Q * kH, 32 * G)) return DSA_ERR_CUDA;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(index_scores_umma_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemMax);
  });
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  // A scoring CTA cannot share an SM with a CTA of the compress kernel still
  // running beside an early start (measured: those CTAs begin ~2 us late and
  // finish last), so a few busy SMs are left out of the grid; the fused form
  // (the compress in this kernel) keeps that grid, which measured faster.
  const int sms = num_sms();
  const int grid = (busy_ctas > 0 && busy_ctas <= sms / 8) ? sms - busy_ctas : sms;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreadsU, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  const cudaError_t e = launch_kernel(&cfg, index_scores_umma_kernel<G>, mk, mq, weights,
                                           scale, pool_start, pool_valid, n_pools, cu_pool_cap,
                                           q_seq, q_pos, Q, B, kpool, P_ld, scores, hist,
                                           es, failure_drill(), status);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

int umma_index_group(int Q, const int32_t* q_seq) {
  // eight queries share every key tile when they all read one sequence
  const int G = (q_seq == nullptr && Q >= 64) ? 8 : 1;
  const size_t smem = G == 8 ? Layout<8>::bytes((Q + 7) / 8, false) : Layout<1>::bytes(Q, false);
  return smem <= (size_t)kSmemMax ? G : 0;
}

bool umma_index_early_ok(int Q, const int32_t* q_seq, const int32_t* q_pos) {
  return umma_index_group(Q, q_seq) == 1 && q_pos == nullptr && Q <= kBaseCache &&
         Layout<1>::bytes(Q, true) <= (size_t)kSmemMax;
}

int launch_index_scores_umma(const void* q, const float* weights, float scale,
                             const void* pool_keys, int pool_rows, const int32_t* pool_start,
                             const uint8_t* pool_valid, const int32_t* n_pools,
                             const int32_t* cu_pool_cap, const int32_t* q_seq,
                             const int32_t* q_pos, int Q, int B, int kpool, int P_ld,
                             float* scores, uint32_t* hist, EarlyStart es,
                             int32_t* status_dev, cudaStream_t stream, int busy_ctas) {
  const int G = umma_index_group(Q, q_seq);
  if (G == 8)
    return launch_g<8>(q, weights, scale, pool_keys, pool_rows, pool_start, pool_valid, n_pools,
                       cu_pool_cap, q_seq, q_pos, Q, B, kpool, P_ld, scores, nullptr,
                       EarlyStart{}, status_dev, stream, 0);
  if (G == 1) {
    const bool early = es.pool_begin != nullptr && es.valid != nullptr &&
                       es.cu_seqlens != nullptr && umma_index_early_ok(Q, q_seq, q_pos);
    return launch_g<1>(q, weights, scale, pool_keys, pool_rows, pool_start, pool_valid, n_pools,
                       cu_pool_cap, q_seq, q_pos, Q, B, kpool, P_ld, scores, hist,
                       early ? es : EarlyStart{}, status_dev, stream, early ? busy_ctas : 0);
  }
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
