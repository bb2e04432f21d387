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
// least one pool below n_cand).
__device__ void tile_prefix(int* s_prefix, int Q, const int32_t* q_seq, const int32_t* q_pos,
                            const int32_t* n_pools, const int32_t* cu_pool_cap,
                            const int32_t* pool_start, int B, int kpool, int P_ld,
                            int32_t* status) {
  __shared__ int s_warp[kWarps];
  __shared__ int s_carry;
  if (threadIdx.x == 0) { s_prefix[0] = 0; s_carry = 0; }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int c = 0; c < Q; c += kThreads) {
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
    if (threadIdx.x == kThreads - 1) s_carry = off + x;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    index_scores_mma_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ wts,
                            float scale, const __nv_bfloat16* __restrict__ pool_keys,
                            const int32_t* __restrict__ pool_start,
                            const uint8_t* __restrict__ pool_valid,
                            const int32_t* __restrict__ n_pools,
                            const int32_t* __restrict__ cu_pool_cap,
                            const int32_t* __restrict__ q_seq, const int32_t* __restrict__ q_pos,
                            int Q, int B, int kpool, int P_ld, float* __restrict__ scores,
                            int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // layout: q block [32][128] bf16 (8 KB) | weights [32] fp32 | mbarrier | prefix [Q+1]
  __nv_bfloat16* s_q = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  float* s_w = reinterpret_cast<float*>(smem_raw + kH * kD * 2);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem_raw + kH * kD * 2 + kH * 4);
  int* s_prefix = reinterpret_cast<int*>(smem_raw + kH * kD * 2 + kH * 4 + 16);

  pdl_wait();
  if (threadIdx.x == 0) {
    mbar_init(s_bar, 1);
    fence_mbar_init();
  }
  tile_prefix(s_prefix, Q, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool, P_ld,
              status);  // ends with __syncthreads
  const int NT = s_prefix[Q];
  const long long t_lo = (long long)NT * blockIdx.x / gridDim.x;
  const long long t_hi = (long long)NT * (blockIdx.x + 1) / gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  int qi = 0;
  uint32_t phase = 0;
  for (long long seg_lo = t_lo; seg_lo < t_hi;) {
    while (s_prefix[qi + 1] <= seg_lo) ++qi;  // query owning tile seg_lo
    const long long seg_hi = min(t_hi, (long long)s_prefix[qi + 1]);
    const QInfo in = query_info(qi, q_seq, q_pos, n_pools, cu_pool_cap, pool_start, B, kpool,
                                P_ld, status, false);
    // Stage the query block and its weights with the TMA engine.
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(s_bar, kH * kD * 2 + kH * 4);
      bulk_g2s(s_q, q + (long long)qi * kH * kD, kH * kD * 2, s_bar);
      bulk_g2s(s_w, wts + (long long)qi * kH, kH * 4, s_bar);
    }
    if (!mbar_wait_bounded(s_bar, phase)) {
      flag(status, DSA_DEV_TIMEOUT);
      return;
    }
    phase ^= 1;
    // B fragments: head 8i+g, channels {8(4m+t) + e}, as uint4 per (i, m).
    uint4 bq[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int m = 0; m < 4; ++m)
        bq[i][m] = *reinterpret_cast<const uint4*>(s_q + (8 * i + g) * kD + 8 * (4 * m + t));
    float wv[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      wv[i][0] = s_w[8 * i + 2 * t];
      wv[i][1] = s_w[8 * i + 2 * t + 1];
    }
    const __nv_bfloat16* keys = pool_keys + in.base * kD;
    const long long row0 = (long long)qi * P_ld;
    const long long tile_q0 = s_prefix[qi];

    auto load_tile = [&](long long tile, uint4 (&a_lo)[4], uint4 (&a_hi)[4]) {
      const int p0 = (int)(tile - tile_q0) * kTile;
      const int r0 = p0 + g, r1 = p0 + g + 8;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        a_lo[m] = r0 < in.n_cand ? ld_stream_v4(keys + (long long)r0 * kD + 8 * (4 * m + t))
                                 : make_uint4(0, 0, 0, 0);
        a_hi[m] = r1 < in.n_cand ? ld_stream_v4(keys + (long long)r1 * kD + 8 * (4 * m + t))
                                 : make_uint4(0, 0, 0, 0);
      }
    };

    long long tile = seg_lo + warp;
    uint4 a_lo[4], a_hi[4];
    if (tile < seg_hi) load_tile(tile, a_lo, a_hi);
    for (; tile < seg_hi; tile += kWarps) {
      uint4 n_lo[4], n_hi[4];
      const long long nxt = tile + kWarps;
      if (nxt < seg_hi) load_tile(nxt, n_lo, n_hi);
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[i][r] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = j >> 1;
        const uint32_t a0 = (j & 1) ? a_lo[m].z : a_lo[m].x;
        const uint32_t a2 = (j & 1) ? a_lo[m].w : a_lo[m].y;
        const uint32_t a1 = (j & 1) ? a_hi[m].z : a_hi[m].x;
        const uint32_t a3 = (j & 1) ? a_hi[m].w : a_hi[m].y;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t b0 = (j & 1) ? bq[i][m].z : bq[i][m].x;
          const uint32_t b1 = (j & 1) ? bq[i][m].w : bq[i][m].y;
          mma_bf16_16816(acc[i], a0, a1, a2, a3, b0, b1);
        }
      }
      // Epilogue: rows g and g+8 of the tile; columns = heads 8i+2t, 8i+2t+1.
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
      // lane l < 16 writes pool p0 + l (rows 0..7 from quad l, rows 8..15 from quad l-8)
      const float v_lo = __shfl_sync(0xffffffffu, lo, 4 * (lane & 7));
      const float v_hi = __shfl_sync(0xffffffffu, hi, 4 * (lane & 7));
      const int p0 = (int)(tile - tile_q0) * kTile;
      const int p = p0 + lane;
      if (lane < kTile && p < P_ld) {
        float s = (lane < 8) ? v_lo : v_hi;
        if (s == 0.f) s = 0.f;  // -0 -> +0
        bool cand = p < in.n_cand && pool_valid[in.base + p] != 0;
        if (cand && q_pos != nullptr) cand = pool_start[in.base + p] + kpool - 1 <= in.pos;
        scores[row0 + p] = cand ? s : -INFINITY;
      }
      if (nxt < seg_hi) {
#pragma unroll
        for (int m = 0; m < 4; ++m) { a_lo[m] = n_lo[m]; a_hi[m] = n_hi[m]; }
      }
    }
    __syncthreads();  // all warps done with s_q before the next segment's copy
    seg_lo = seg_hi;
  }

  // Fill the rest of each row (whole tiles past n_cand) with -inf.
  const long long gtid = (long long)blockIdx.x * kThreads + threadIdx.x;
  const long long gstride = (long long)gridDim.x * kThreads;
  for (int r = 0; r < Q; ++r) {
    const long long start = (long long)(s_prefix[r + 1] - s_prefix[r]) * kTile;
    const long long n = (long long)P_ld - start;
    for (long long i = gtid; i < n; i += gstride) scores[(long long)r * P_ld + start + i] = -INFINITY;
  }
  pdl_launch_dependents();
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

int launch_index_scores(const void* q, const float* weights, float scale, const void* pool_keys,
                        const int32_t* pool_start, const uint8_t* pool_valid,
                        const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                        const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                        int dtype, float* scores, int32_t* status_dev, cudaStream_t stream) {
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (dtype == DSA_BF16 && H == kH && D == kD) {
    const size_t smem = kH * kD * 2 + kH * 4 + 16 + (size_t)(Q + 1) * 4;
    if (smem > 200 * 1024) return DSA_ERR_UNSUPPORTED;
    cudaFuncSetAttribute(index_scores_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    // Enough CTAs to cover every SM once; each streams a balanced share of tiles.
    cfg.gridDim = dim3(kNumSMs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaError_t e = cudaLaunchKernelEx(&cfg, index_scores_mma_kernel,
                                       (const __nv_bfloat16*)q, weights, scale,
                                       (const __nv_bfloat16*)pool_keys, pool_start, pool_valid,
                                       n_pools, cu_pool_cap, q_seq, q_pos, Q, B, kpool, P_ld,
                                       scores, status_dev);
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
