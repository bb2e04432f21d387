// index_scores: score[q, p] = sum_h w[q, h] * max(0, scale * <q[q, h, :], key[p, :]>).
//
// Module glm5next_dsa::tp, "Why the indexer is REPLICATED, not sharded": a plain
// sum over heads of weights[h] * relu(scale * dot); module glm5next_dsa, "Shape
// of the pipeline": [Q, P] scores with candidate validity (-inf here).
//
// Decode kernel (bf16, H = 32, D = 128).  Each pool key costs 32 x 128 MACs
// for 256 bytes (32 flop/B), which at HBM speed is far above what fp32 FMA
// units deliver, so the contraction runs on the tensor cores with warp-level
// mma.sync m16n8k16 in swap-AB form: A = 16 pool keys (rows), B = 8 heads
// (columns), K = 16 channels.  A warp owns 16 pools per step: 4 head tiles x 8
// channel steps = 32 MMAs.  Pool keys go straight from HBM into the A
// registers with coalesced 128-bit loads: the channel axis is permuted
// identically on A and B (a dot product does not care about channel order), so
// the four lanes of a quad read one contiguous 64-byte run of a key row per
// load.  The 32-head query block (8 KB) and its weights are staged once per
// query segment in shared memory by a TMA bulk copy, then held in registers as
// B fragments (64 registers).  The head sum is done in registers across the
// four head tiles and with two xor-shuffles inside each quad.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kH = 32, kD = 128;
constexpr int kTile = 16;              // pools per warp step
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct QInfo {
  long long base;  // first cache entry of the query's sequence
  int n_cand;      // pools [0, n_cand) may be candidates
  int pos;         // query position (causal) or INT_MAX
};

// Candidate range of query qi; flags bad sequence ids and pool ranges.
__device__ __forceinline__ QInfo query_info(int qi, const int32_t* q_seq, const int32_t* q_pos,
                                            const int32_t* n_pools, const int32_t* cu_pool_cap,
                                            const int32_t* pool_start, int B, int kpool,
                                            int P_ld, int32_t* status, bool report) {
  QInfo r{0, 0, 0x7fffffff};
  const int b = q_seq ? q_seq[qi] : 0;
  if (b < 0 || b >= B) {
    if (report) flag(status, DSA_DEV_BAD_QSEQ);
    return r;
  }
  r.base = cu_pool_cap[b];
  const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
  const int np = n_pools[b];
  int P = min(np, min(cap, P_ld));
  if (np > P && report) flag(status, DSA_DEV_POOL_RANGE);
  P = max(P, 0);
  if (q_pos != nullptr && P > 0) {
    r.pos = q_pos[qi];
    // pool p is complete at pos when t0 + p*kpool + kpool - 1 <= pos
    const long long t0 = pool_start[r.base];
    const long long nv = (r.pos - t0 + 1) >= 0 ? (r.pos - t0 + 1) / kpool : 0;
    P = (int)min((long long)P, nv);
  }
  r.n_cand = P;
  return r;
}

// Per-CTA prefix over queries of "heavy" 16-pool tiles (tiles holding at
// least one pool below n_cand).  Block-wide; ends with __syncthreads.
__device__ void tile_prefix(int* s_prefix, int Q, const int32_t* q_seq, const int32_t* q_pos,
                            const int32_t* n_pools, const int32_t* cu_pool_cap,
                            const int32_t* pool_start, int B, int kpool, int P_ld,
                            int32_t* status) {
  __shared__ int s_warp[32];
  __shared__ int s_carry;
  const int nthr = blockDim.x, nwarp = (nthr + 31) >> 5;
  if (threadIdx.x == 0) { s_prefix[0] = 0; s_carry = 0; }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int c = 0; c < Q; c += nthr) {
    const int qi = c + threadIdx.x;
    int n = 0;
    if (qi < Q) {
      QInfo in = query_info(qi, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool, P_ld,
                            status, blockIdx.x == 0);
      n = (in.n_cand + kTile - 1) / kTile;
    }
    int x = n;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    int off = s_carry;
    for (int w = 0; w < warp; ++w) off += s_warp[w];
    if (qi < Q) s_prefix[qi + 1] = off + x;
    __syncthreads();
    if (threadIdx.x == nthr - 1) s_carry = off + x;
    __syncthreads();
  }
  (void)nwarp;
}

// ---------------------------------------------------------------------------
// Tensor-core decode kernel.  Warp-specialised: warp 8 is the producer (one
// lane issues TMA bulk copies of 128-pool chunks, 32 KB each, into a 4-stage
// shared-memory ring guarded by full/empty mbarriers); warps 0..7 consume, one
// 16-pool tile each per chunk.  Each CTA owns a balanced, contiguous range of
// the flattened (query, 16-pool tile) space; the query block of each query it
// meets is staged by a bulk copy and held as B fragments in registers.
// Optionally every candidate score is counted in a 4096-bin histogram of its
// top 12 key bits (shared memory, flushed to hist[q] per query segment) for the
// radix top-k that follows.
// ---------------------------------------------------------------------------
constexpr int kConsumers = 8;
constexpr int kIdxThreads = (kConsumers + 1) * 32;
constexpr int kChunk = kConsumers * kTile;        // 128 pools per stage
constexpr int kChunkBytes = kChunk * kD * 2;      // 32 KB
constexpr int kStages = 4;
constexpr int kHistBins = 4096;

struct IdxSmem {
  __nv_bfloat16 stage[kStages][kChunk * kD];
  __nv_bfloat16 q[kH * kD];
  float w[kH];
  uint64_t full[kStages], empty[kStages], qfull, qempty;
  uint32_t hist[kHistBins];
};

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__global__ void __launch_bounds__(kIdxThreads, 1)
    index_scores_mma_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ wts,
                            float scale, const __nv_bfloat16* __restrict__ pool_keys,
                            const int32_t* __restrict__ pool_start,
                            const uint8_t* __restrict__ pool_valid,
                            const int32_t* __restrict__ n_pools,
                            const int32_t* __restrict__ cu_pool_cap,
                            const int32_t* __restrict__ q_seq, const int32_t* __restrict__ q_pos,
                            int Q, int B, int kpool, int P_ld, float* __restrict__ scores,
                            uint32_t* __restrict__ hist, int32_t* status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  IdxSmem& sm = *reinterpret_cast<IdxSmem*>(smem_raw);
  int* s_prefix = reinterpret_cast<int*>(smem_raw + sizeof(IdxSmem));
  __shared__ int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool producer = warp == kConsumers;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsumers);
    }
    mbar_init(&sm.qfull, 1);
    mbar_init(&sm.qempty, kConsumers);
    fence_mbar_init();
    s_abort = 0;
  }
  if (hist)
    for (int i = threadIdx.x; i < kHistBins; i += kIdxThreads) sm.hist[i] = 0;
  pdl_wait();  // the pool cache may come from the kernel just before
  pdl_launch_dependents();  // the selection kernel may start its prologue
  tile_prefix(s_prefix, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool, P_ld,
              status);
  const int NT = s_prefix[Q];
  const long long t_lo = (long long)NT * blockIdx.x / gridDim.x;
  const long long t_hi = (long long)NT * (blockIdx.x + 1) / gridDim.x;
  const int g = lane >> 2, t = lane & 3;

  uint32_t full_phase = 0, empty_phase = 0;  // one parity bit per stage
  uint32_t uses = 0;                         // producer: stage uses so far (first lap: no wait)
  int stage = 0, qi = 0, seg = 0;
  for (long long seg_lo = t_lo; seg_lo < t_hi; ++seg) {
    while (s_prefix[qi + 1] <= seg_lo) ++qi;
    const long long seg_hi = min(t_hi, (long long)s_prefix[qi + 1]);
    const QInfo in = query_info(qi, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool,
                                P_ld, status, false);
    const long long tile_q0 = s_prefix[qi];
    const int p_seg0 = (int)(seg_lo - tile_q0) * kTile;
    const int p_seg1 = min((int)(seg_hi - tile_q0) * kTile, in.n_cand);
    const int n_chunks = (p_seg1 - p_seg0 + kChunk - 1) / kChunk;
    const __nv_bfloat16* keys = pool_keys + in.base * kD;

    if (producer) {
      if (lane == 0) {
        if (seg > 0 && !mbar_wait_bounded(&sm.qempty, (seg - 1) & 1)) {
          flag(status, DSA_DEV_TIMEOUT);
          s_abort = 1;
        }
        mbar_arrive_expect_tx(&sm.qfull, kH * kD * 2 + kH * 4);
        bulk_g2s(sm.q, q + (long long)qi * kH * kD, kH * kD * 2, &sm.qfull);
        bulk_g2s(sm.w, wts + (long long)qi * kH, kH * 4, &sm.qfull);
        for (int c = 0; c < n_chunks && !s_abort; ++c) {
          const int r0 = p_seg0 + c * kChunk, r1 = min(r0 + kChunk, p_seg1);
          if (uses >= (uint32_t)kStages) {
            if (!mbar_wait_bounded(&sm.empty[stage], (empty_phase >> stage) & 1)) {
              flag(status, DSA_DEV_TIMEOUT);
              s_abort = 1;
              break;
            }
            empty_phase ^= 1u << stage;
          }
          ++uses;
          const uint32_t bytes = (uint32_t)(r1 - r0) * kD * 2;
          mbar_arrive_expect_tx(&sm.full[stage], bytes);
          bulk_g2s(sm.stage[stage], keys + (long long)r0 * kD, bytes, &sm.full[stage]);
          stage = (stage + 1) % kStages;
        }
      }
    } else {
      if (!mbar_wait_bounded(&sm.qfull, seg & 1)) {
        flag(status, DSA_DEV_TIMEOUT);
        return;
      }
      uint4 bq[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m)
          bq[i][m] = *reinterpret_cast<const uint4*>(sm.q + (8 * i + g) * kD + 8 * (4 * m + t));
      float wv[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wv[i][0] = sm.w[8 * i + 2 * t];
        wv[i][1] = sm.w[8 * i + 2 * t + 1];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.qempty);
      const long long row0 = (long long)qi * P_ld;
      for (int c = 0; c < n_chunks; ++c) {
        const int r0 = p_seg0 + c * kChunk;
        const int p0 = r0 + warp * kTile;  // this warp's 16 pools
        // candidate metadata first: its latency hides behind the chunk wait
        const int pm = p0 + lane;
        bool cand = lane < kTile && pm < in.n_cand && pool_valid[in.base + pm] != 0;
        if (cand && q_pos != nullptr) cand = pool_start[in.base + pm] + kpool - 1 <= in.pos;
        if (!mbar_wait_bounded(&sm.full[stage], (full_phase >> stage) & 1)) {
          flag(status, DSA_DEV_TIMEOUT);
          return;
        }
        full_phase ^= 1u << stage;
        if (p0 < p_seg1) {
          const __nv_bfloat16* a = sm.stage[stage] + warp * kTile * kD;
          float acc[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][r] = 0.f;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint4 lo4 = *reinterpret_cast<const uint4*>(a + g * kD + 8 * (4 * m + t));
            const uint4 hi4 = *reinterpret_cast<const uint4*>(a + (g + 8) * kD + 8 * (4 * m + t));
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // channel step j = 2m + h
              const uint32_t a0 = h ? lo4.z : lo4.x, a2 = h ? lo4.w : lo4.y;
              const uint32_t a1 = h ? hi4.z : hi4.x, a3 = h ? hi4.w : hi4.y;
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t b0 = h ? bq[i][m].z : bq[i][m].x;
                const uint32_t b1 = h ? bq[i][m].w : bq[i][m].y;
                mma_bf16_16816(acc[i], a0, a1, a2, a3, b0, b1);
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[stage]);  // smem reads of this warp are done
          float lo = 0.f, hi = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            lo += wv[i][0] * fmaxf(scale * acc[i][0], 0.f) + wv[i][1] * fmaxf(scale * acc[i][1], 0.f);
            hi += wv[i][0] * fmaxf(scale * acc[i][2], 0.f) + wv[i][1] * fmaxf(scale * acc[i][3], 0.f);
          }
          lo += __shfl_xor_sync(0xffffffffu, lo, 1);
          hi += __shfl_xor_sync(0xffffffffu, hi, 1);
          lo += __shfl_xor_sync(0xffffffffu, lo, 2);
          hi += __shfl_xor_sync(0xffffffffu, hi, 2);
          const float v_lo = __shfl_sync(0xffffffffu, lo, 4 * (lane & 7));
          const float v_hi = __shfl_sync(0xffffffffu, hi, 4 * (lane & 7));
          const int p = pm;
          if (lane < kTile && p < P_ld) {
            float sc = (lane < 8) ? v_lo : v_hi;
            if (sc == 0.f) sc = 0.f;  // -0 -> +0
            scores[row0 + p] = cand ? sc : -INFINITY;
            if (cand && hist) atomicAdd(&sm.hist[score_key(sc) >> 20], 1u);
          }
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[stage]);
        }
        stage = (stage + 1) % kStages;
      }
      if (hist) {  // flush this query segment's histogram
        consumer_bar();
        uint32_t* gh = hist + (size_t)qi * kHistBins;
        for (int i = threadIdx.x; i < kHistBins; i += kConsumers * 32) {
          const uint32_t v = sm.hist[i];
          if (v) {
            atomicAdd(&gh[i], v);
            sm.hist[i] = 0;
          }
        }
        consumer_bar();
      }
    }
    // the producer's lane 0 and every consumer warp advance `stage` once per chunk
    seg_lo = seg_hi;
  }

  // Fill the rest of each row (whole tiles past n_cand) with -inf.
  const long long gtid = (long long)blockIdx.x * kIdxThreads + threadIdx.x;
  const long long gstride = (long long)gridDim.x * kIdxThreads;
  for (int r = 0; r < Q; ++r) {
    const long long start = (long long)(s_prefix[r + 1] - s_prefix[r]) * kTile;
    const long long n = (long long)P_ld - start;
    for (long long i = gtid; i < n; i += gstride) scores[(long long)r * P_ld + start + i] = -INFINITY;
  }
}

// Generic SIMT kernel: any H <= 64, D in {32..256}, fp32 or bf16.  One thread
// per pool; the query block sits in shared memory as fp32.
template <typename T>
__global__ void __launch_bounds__(128)
    index_scores_simt_kernel(const T* __restrict__ q, const float* __restrict__ wts, float scale,
                             const T* __restrict__ pool_keys, const int32_t* __restrict__ pool_start,
                             const uint8_t* __restrict__ pool_valid,
                             const int32_t* __restrict__ n_pools,
                             const int32_t* __restrict__ cu_pool_cap,
                             const int32_t* __restrict__ q_seq, const int32_t* __restrict__ q_pos,
                             int B, int H, int D, int kpool, int P_ld, float* __restrict__ scores,
                             int32_t* status) {
  extern __shared__ float s_qf[];  // [H][D] then [H] weights
  pdl_wait();
  const int qi = blockIdx.y;
  for (int i = threadIdx.x; i < H * D; i += blockDim.x)
    s_qf[i] = Act<T>::to_f(q[(long long)qi * H * D + i]);
  for (int i = threadIdx.x; i < H; i += blockDim.x) s_qf[H * D + i] = wts[(long long)qi * H + i];
  __syncthreads();
  const QInfo in = query_info(qi, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool, P_ld,
                              status, blockIdx.x == 0 && threadIdx.x == 0);
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= P_ld) return;
  bool cand = p < in.n_cand && pool_valid[in.base + p] != 0;
  if (cand && q_pos != nullptr) cand = pool_start[in.base + p] + kpool - 1 <= in.pos;
  float s = -INFINITY;
  if (cand) {
    const T* key = pool_keys + (in.base + p) * D;
    s = 0.f;
    for (int h = 0; h < H; ++h) {
      float dot = 0.f;
      for (int d = 0; d < D; ++d) dot = fmaf(Act<T>::to_f(key[d]), s_qf[h * D + d], dot);
      s += s_qf[H * D + h] * fmaxf(scale * dot, 0.f);
    }
    if (s == 0.f) s = 0.f;
  }
  scores[(long long)qi * P_ld + p] = s;
}

cudaLaunchAttribute pdl_attr() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

}  // namespace

bool index_uses_tensor_cores(int H, int D, int dtype) {
  return dtype == DSA_BF16 && H == kH && D == kD;
}

int launch_index_scores(const void* q, const float* weights, float scale, const void* pool_keys,
                        const int32_t* pool_start, const uint8_t* pool_valid,
                        const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                        const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                        int dtype, float* scores, uint32_t* score_hist, int32_t* status_dev,
                        cudaStream_t stream) {
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (dtype == DSA_BF16 && H == kH && D == kD) {
    const size_t smem = sizeof(IdxSmem) + (size_t)(Q + 1) * 4;
    if (smem > 227 * 1024) return DSA_ERR_UNSUPPORTED;
    cudaFuncSetAttribute(index_scores_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    // One CTA per SM; each streams a balanced share of the pool tiles.
    cfg.gridDim = dim3(kNumSMs, 1, 1);
    cfg.blockDim = dim3(kIdxThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaError_t e = cudaLaunchKernelEx(&cfg, index_scores_mma_kernel,
                                       (const __nv_bfloat16*)q, weights, scale,
                                       (const __nv_bfloat16*)pool_keys, pool_start, pool_valid,
                                       n_pools, cu_pool_cap, q_seq, q_pos, Q, B, kpool, P_ld,
                                       scores, score_hist, status_dev);
    return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  if (H < 1 || H > 64 || (D != 32 && D != 64 && D != 128 && D != 256)) return DSA_ERR_UNSUPPORTED;
  const size_t smem = ((size_t)H * D + H) * 4;
  cfg.gridDim = dim3((P_ld + 127) / 128, Q, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaError_t e;
  if (dtype == DSA_BF16) {
    cudaFuncSetAttribute(index_scores_simt_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
    e = cudaLaunchKernelEx(&cfg, index_scores_simt_kernel<__nv_bfloat16>,
                           (const __nv_bfloat16*)q, weights, scale,
                           (const __nv_bfloat16*)pool_keys, pool_start, pool_valid, n_pools,
                           cu_pool_cap, q_seq, q_pos, B, H, D, kpool, P_ld, scores, status_dev);
  } else {
    cudaFuncSetAttribute(index_scores_simt_kernel<float>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
    e = cudaLaunchKernelEx(&cfg, index_scores_simt_kernel<float>, (const float*)q, weights, scale,
                           (const float*)pool_keys, pool_start, pool_valid, n_pools, cu_pool_cap,
                           q_seq, q_pos, B, H, D, kpool, P_ld, scores, status_dev);
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
