// kpool_compress: fused indexer-key LayerNorm + per-channel slot-softmax pooling.
//
// Module glm5next_dsa, "Shape of the pipeline" (k, gate, valid, ape ->
// kpool_compress -> pool keys / indices / valid) and "Traps carried from Slice 8"
// (LayerNorm with bias, softmax over the slot axis per channel, pools start at
// the first valid token, only full all-valid pools count).  Constants,
// LAYERNORM_MODULE: the normalised key is stored in the activation dtype, so it
// is rounded to that dtype in registers before it is pooled.
//
// One warp owns one pool.  Lane l owns channels [l*V, l*V + V) (V = D/32), so a
// token row is read by the warp as one contiguous D-element segment.  The kpool
// (<= 8) slots of the pool stay in registers: LayerNorm statistics are two warp
// reductions per slot, the softmax runs over the slot axis in registers, and
// the pooled key is written with one vector store per lane.  HBM-bound: a full
// build streams 2 * D * sizeof(act) bytes per token and writes D * sizeof(act)
// / kpool bytes per token.
#include <mutex>

#include "compress_pool.cuh"

namespace dsa {
namespace {

constexpr int kWarpsPerCta = 8;
// First valid token of sequence [lo, lo+T): block-wide scan from the front,
// stopping at the first chunk that holds a valid byte.
__device__ int first_valid_token(const uint8_t* valid, long long lo, int T, int* s_min) {
  if (threadIdx.x == 0) *s_min = T;
  __syncthreads();
  for (int base = 0; base < T; base += blockDim.x) {
    int t = base + threadIdx.x;
    bool hit = (t < T) && valid[lo + t] != 0;
    if (hit) atomicMin(s_min, t);
    if (__syncthreads_or(hit)) break;
  }
  int r = *s_min;
  __syncthreads();
  return r;
}

template <typename T, int V>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    kpool_compress_kernel(const T* __restrict__ k, const T* __restrict__ gate,
                          const uint8_t* __restrict__ valid, const float* __restrict__ ape,
                          const T* __restrict__ ln_gamma, const T* __restrict__ ln_beta,
                          float ln_eps, const int32_t* __restrict__ cu_seqlens,
                          const int32_t* __restrict__ cu_pool_cap,
                          const int32_t* __restrict__ pool_begin, int kpool, int max_pools,
                          T* __restrict__ pool_keys, int32_t* __restrict__ pool_start,
                          uint8_t* __restrict__ pool_valid, int32_t* __restrict__ n_pools,
                          int32_t* status) {
  constexpr int D = 32 * V;
  __shared__ int s_min;
  pdl_wait();
  pdl_launch_dependents();  // the next kernel may start its prologue
  const int b = blockIdx.y;
  const long long lo = cu_seqlens[b];
  const int Tb = cu_seqlens[b + 1] - cu_seqlens[b];
  const long long cap_lo = cu_pool_cap[b];
  const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
  const int begin = pool_begin ? pool_begin[b] : 0;
  const long long end_ll = min((long long)begin + max_pools, (long long)cap);
  const int end = (int)end_ll;

  // Nothing of this sequence is in this CTA's pool range: skip the scan.
  const int p_first = begin + blockIdx.x * kWarpsPerCta;
  const bool cta_has_work = p_first < end || blockIdx.x == 0;
  if (!cta_has_work) return;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p = p_first + warp;
  // An incremental call (begin > 0) extends a cache whose first pool starts at
  // the sequence's first valid token.  Warm this warp's token rows in L2 from
  // that start while the scan below confirms it, so the two cold misses overlap
  // instead of following each other.  Only in-range addresses are touched.
  if (begin > 0 && p >= 0 && p < end) {
    const int t0g = pool_start[cap_lo];
    const long long s0 = lo + t0g + (long long)p * kpool;
    if (t0g >= 0 && s0 + kpool <= lo + Tb) {
      constexpr int kLines = (D * (int)sizeof(T) + 127) / 128;   // 128-byte lines per row
      for (int i = lane; i < 2 * kKpoolMax * kLines; i += 32) {
        const int arr = i / (kKpoolMax * kLines), r = i % (kKpoolMax * kLines);
        const int s = r / kLines, l = r % kLines;
        if (s < kpool) {
          const T* row = (arr ? gate : k) + (s0 + s) * D;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(row) + l * 128));
        }
      }
      if (lane == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(valid + s0));
    }
  }
  const int t0 = first_valid_token(valid + 0, lo, Tb, &s_min);
  const int P = (Tb - t0) / kpool;
  const int P_eff = min(P, cap);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    n_pools[b] = P_eff;
    if (P > cap) flag(status, DSA_DEV_POOL_OVERFLOW);
    if (P_eff > end) flag(status, DSA_DEV_POOL_UNCOVERED);
  }

  if (p < 0 || p >= end) return;
  T* out = pool_keys + (cap_lo + p) * D + lane * V;
  if (p >= P_eff) {  // sentinel entry
    compress_sentinel_warp<T, V>(lane, out, pool_start + cap_lo + p, pool_valid + cap_lo + p);
    return;
  }

  compress_pool_warp<T, V>(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps,
                           lo + t0 + (long long)p * kpool, kpool, lane, out,
                           t0 + p * kpool, pool_start + cap_lo + p, pool_valid + cap_lo + p);
}

// Bulk builds (a cache build, a prefill chunk's pools) in bf16 with D = 128.
// Each CTA takes up to kWidePools consecutive pools of one sequence, whose token rows
// are one contiguous stretch of k and one of gate: a producer warp streams them
// with 1-D bulk copies (TMA) into a ring of shared-memory stages of 16 pools,
// while the 16 half-warps of the other eight warps compute one pool each per
// stage (lane j owning channels
// [8j, 8j + 8)) and write 16-byte key pieces.  The metadata loads and the
// first-valid-token scan are shared by the CTA's pools.  The LayerNorm
// statistics are reduced in the order of the warp-per-pool kernel above (lane
// j holds that kernel's lanes 2j and 2j + 1), so the two kernels write
// bit-identical keys.  Waits on the ring are bounded (DSA_DEV_TIMEOUT).
constexpr int kWidePools = 256;   // most pools per CTA (fewer when that leaves SMs idle)
constexpr int kStagePools = 16;   // pools per ring stage (one per half-warp)
constexpr int kWideMin = 32;      // launches covering at least this many pools per sequence
constexpr int kWideConsumers = 256;             // 8 warps, 16 half-warps
constexpr int kWideThreads = kWideConsumers + 32;  // + the producer warp

template <int KP>
struct WideCfg {
  static constexpr int kStageBytes = kStagePools * KP * 128 * 2;  // one array (k or gate)
  static constexpr int kStages = 2;
  static constexpr int kCtasPerSm = KP <= 4 ? 3 : 1;  // 64 KB of ring each at kpool <= 4
  static constexpr size_t kSmem = 128 + (size_t)kStages * 2 * kStageBytes;
};

__device__ __forceinline__ float half_sum(float v, unsigned mask) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(mask, v, o, 16);
  return v;
}

template <int KP>  // slots held per pool (>= kpool)
__global__ void __launch_bounds__(kWideThreads, WideCfg<KP>::kCtasPerSm)
    kpool_compress_wide_kernel(const __nv_bfloat16* __restrict__ k,
                               const __nv_bfloat16* __restrict__ gate,
                               const uint8_t* __restrict__ valid, const float* __restrict__ ape,
                               const __nv_bfloat16* __restrict__ ln_gamma,
                               const __nv_bfloat16* __restrict__ ln_beta, float ln_eps,
                               const int32_t* __restrict__ cu_seqlens,
                               const int32_t* __restrict__ cu_pool_cap,
                               const int32_t* __restrict__ pool_begin, int kpool, int max_pools,
                               int ppc, __nv_bfloat16* __restrict__ pool_keys,
                               int32_t* __restrict__ pool_start,
                               uint8_t* __restrict__ pool_valid, int32_t* __restrict__ n_pools,
                               int32_t* status) {
  constexpr int D = 128;
  using T = __nv_bfloat16;
  using WC = WideCfg<KP>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  static_assert(kWidePools * KP <= 2048, "valid bytes on chip");
  __shared__ int s_min;
  __shared__ __align__(16) float s_ape[KP * D];
  __shared__ uint8_t s_valid[kWidePools * KP];
  __shared__ uint64_t full[4], empty[4];
  pdl_wait();
  pdl_launch_dependents();  // the next kernel may start its prologue
  const int b = blockIdx.y;
  const long long lo = cu_seqlens[b];
  const int Tb = cu_seqlens[b + 1] - cu_seqlens[b];
  const long long cap_lo = cu_pool_cap[b];
  const int cap = cu_pool_cap[b + 1] - cu_pool_cap[b];
  const int begin = pool_begin ? pool_begin[b] : 0;
  const int end = (int)min((long long)begin + max_pools, (long long)cap);
  const int p_first = begin + blockIdx.x * ppc;
  if (!(p_first < end || blockIdx.x == 0)) return;  // nothing of this sequence here
  for (int i = threadIdx.x; i < kpool * D; i += blockDim.x) s_ape[i] = ape[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < WC::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWideConsumers / 32);
    }
    fence_mbar_init();
  }
  const int t0 = first_valid_token(valid + 0, lo, Tb, &s_min);  // (its barriers publish the above)
  const int P = (Tb - t0) / kpool;
  const int P_eff = min(P, cap);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    n_pools[b] = P_eff;
    if (P > cap) flag(status, DSA_DEV_POOL_OVERFLOW);
    if (P_eff > end) flag(status, DSA_DEV_POOL_UNCOVERED);
  }
  // this CTA's pools [pa, pb); the computed ones [pa, pc), sentinels after
  const int pa = max(p_first, 0), pb = min(p_first + ppc, end);
  const int pc = max(pa, min(pb, P_eff));
  const int n_stages_work = (pc - pa + kStagePools - 1) / kStagePools;
  const int half = threadIdx.x >> 4, j = threadIdx.x & 15;
  const unsigned hmask = 0xffffu << (threadIdx.x & 16);
  const size_t row_bytes = (size_t)D * 2;

  if (threadIdx.x >= kWideConsumers) {
    // ---- producer warp (lane 0): the rows of 16 pools per stage, k then gate
    if (threadIdx.x != kWideConsumers) return;
    int i = 0;
    for (; i < n_stages_work; ++i) {
      const int st = i % WC::kStages;
      if (i >= WC::kStages &&
          !mbar_wait_bounded(&empty[st], (uint32_t)((i / WC::kStages) - 1) & 1)) {
        flag(status, DSA_DEV_TIMEOUT);
        break;
      }
      const int p0 = pa + i * kStagePools, np = min(kStagePools, pc - p0);
      const uint32_t bytes = (uint32_t)((size_t)np * kpool * row_bytes);
      const long long row0 = lo + t0 + (long long)p0 * kpool;
      unsigned char* sk = ring + (size_t)st * 2 * WC::kStageBytes;
      mbar_arrive_expect_tx(&full[st], 2 * bytes);
      bulk_g2s(sk, k + row0 * D, bytes, &full[st]);
      bulk_g2s(sk + WC::kStageBytes, gate + row0 * D, bytes, &full[st]);
    }
    // never leave a copy in flight: wait for the last fills issued
    for (int f = max(0, i - WC::kStages); f < i; ++f)
      mbar_wait_bounded(&full[f % WC::kStages], (uint32_t)(f / WC::kStages) & 1);
    return;
  }
  // the valid bytes of every slot of the computed pools, once per CTA
  const long long tok0 = lo + t0 + (long long)pa * kpool;
  for (int i = threadIdx.x; i < (pc - pa) * kpool; i += kWideConsumers) s_valid[i] = valid[tok0 + i];
  asm volatile("bar.sync 1, %0;" ::"n"(kWideConsumers) : "memory");  // the consumer warps
  float g[8], be[8];
  Vec<T, 8>::load(ln_gamma + j * 8, g);
  Vec<T, 8>::load(ln_beta + j * 8, be);
  bool ok = true;
  for (int i = 0; i < n_stages_work; ++i) {
    const int st = i % WC::kStages;
    ok = ok && mbar_wait_bounded(&full[st], (uint32_t)(i / WC::kStages) & 1);
    const int p = pa + i * kStagePools + half;
    if (ok && p < pc) {
      // this pool's slot rows in the stage: k at sk, gate at sk + kStageBytes
      unsigned char* sk = ring + (size_t)st * 2 * WC::kStageBytes +
                          (size_t)half * kpool * row_bytes + j * 16;
      // the slot logits gate + ape of the pool's 8 channels of this lane
      auto logits = [&](int s, float (&l)[8]) {
        const uint4 c4 = *reinterpret_cast<const uint4*>(sk + WC::kStageBytes + s * row_bytes);
        const float4 a0 = *reinterpret_cast<const float4*>(s_ape + s * D + j * 8);
        const float4 a1 = *reinterpret_cast<const float4*>(s_ape + s * D + j * 8 + 4);
        l[0] = bf16lo(c4.x) + a0.x;
        l[1] = bf16hi(c4.x) + a0.y;
        l[2] = bf16lo(c4.y) + a0.z;
        l[3] = bf16hi(c4.y) + a0.w;
        l[4] = bf16lo(c4.z) + a1.x;
        l[5] = bf16hi(c4.z) + a1.y;
        l[6] = bf16lo(c4.w) + a1.z;
        l[7] = bf16hi(c4.w) + a1.w;
      };
      // 1. the per-channel maximum of the logits over the slots
      float m[8], den[8], acc[8];
      logits(0, m);
#pragma unroll
      for (int s = 1; s < KP; ++s) {
        if (s < kpool) {
          float l[8];
          logits(s, l);
#pragma unroll
          for (int c = 0; c < 8; ++c) m[c] = fmaxf(m[c], l[c]);
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) den[c] = acc[c] = 0.f;
      // 2. per slot: the LayerNorm of the k row (statistics in the warp-per-pool
      // kernel's order: lane j holds its lanes 2j and 2j + 1), rounded to bf16,
      // weighed by the softmax weight (the logits are formed again)
#pragma unroll
      for (int s = 0; s < KP; ++s) {
        if (s < kpool) {
          float x[8], dx[8], l[8];
          const uint4 a = *reinterpret_cast<const uint4*>(sk + s * row_bytes);
          const uint32_t av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            x[2 * u] = bf16lo(av[u]);
            x[2 * u + 1] = bf16hi(av[u]);
          }
          const float mean =
              half_sum(lane_sum<4>(x) + lane_sum<4>(x + 4), hmask) * (1.0f / D);
#pragma unroll
          for (int c = 0; c < 8; ++c) dx[c] = x[c] - mean;
          const float var = half_sum(lane_sq<4>(dx) + lane_sq<4>(dx + 4), hmask) * (1.0f / D);
          const float rstd = rsqrtf(var + ln_eps);
          logits(s, l);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            // the normalised pair rounded to bf16 (round to nearest even)
            const uint32_t yy = pack_bf16(fmaf(dx[2 * u] * rstd, g[2 * u], be[2 * u]),
                                          fmaf(dx[2 * u + 1] * rstd, g[2 * u + 1], be[2 * u + 1]));
            const float y[2] = {bf16lo(yy), bf16hi(yy)};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = 2 * u + h;
              const float e = exp2_approx((l[c] - m[c]) * kLog2e);
              den[c] += e;
              acc[c] = fmaf(e, y[h], acc[c]);
            }
          }
        }
      }
      float res[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) res[c] = __fdividef(acc[c], den[c]);  // den in [1, kpool]
      Vec<T, 8>::store(pool_keys + (cap_lo + p) * D + j * 8, res);
      if (j == 0) {
        bool all_valid = true;
        for (int s = 0; s < kpool; ++s) all_valid &= s_valid[(p - pa) * kpool + s] != 0;
        pool_start[cap_lo + p] = t0 + p * kpool;
        pool_valid[cap_lo + p] = all_valid ? 1 : 0;
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive1(&empty[st]);  // this warp is done with the stage
  }
  if (!ok && (threadIdx.x & 31) == 0) flag(status, DSA_DEV_TIMEOUT);
  // sentinels: pools of the range past the complete ones
  for (int p = pc + half; p < pb; p += kWideConsumers / 16) {
    *reinterpret_cast<uint4*>(pool_keys + (cap_lo + p) * D + j * 8) = make_uint4(0u, 0u, 0u, 0u);
    if (j == 0) {
      pool_start[cap_lo + p] = -1;
      pool_valid[cap_lo + p] = 0;
    }
  }
}

// Pools per CTA of the bulk kernel: kWidePools, or fewer (a multiple of the
// 16-pool stage) when that many would leave SMs without a CTA.
int wide_pools_per_cta(int B, int max_pools, int ctas_per_sm) {
  const long long slots = (long long)num_sms() * ctas_per_sm;
  const long long want = ((long long)B * max_pools + slots - 1) / slots;
  const int ppc = (int)((want + kStagePools - 1) / kStagePools * kStagePools);
  return max(kStagePools, min(kWidePools, ppc));
}

template <int KP>
int launch_wide(const void* k, const void* gate, const uint8_t* valid, const float* ape,
                const void* g, const void* be, float eps, const int32_t* cu, const int32_t* cap,
                const int32_t* begin, int B, int kpool, int max_pools, void* pk, int32_t* ps,
                uint8_t* pv, int32_t* np, int32_t* st, cudaStream_t stream) {
  using T = __nv_bfloat16;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(kpool_compress_wide_kernel<KP>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)WideCfg<KP>::kSmem);
  });
  cudaLaunchConfig_t cfg = {};
  const int ppc = wide_pools_per_cta(B, max_pools, WideCfg<KP>::kCtasPerSm);
  cfg.gridDim = dim3((max_pools + ppc - 1) / ppc, B, 1);
  cfg.blockDim = dim3(kWideThreads, 1, 1);
  cfg.dynamicSmemBytes = WideCfg<KP>::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = launch_kernel(
      &cfg, kpool_compress_wide_kernel<KP>, (const T*)k, (const T*)gate, valid, ape, (const T*)g,
      (const T*)be, eps, cu, cap, begin, kpool, max_pools, ppc, (T*)pk, ps, pv, np, st);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

bool uses_wide(int D, int max_pools, int dtype) {
  return dtype == DSA_BF16 && D == 128 && max_pools >= kWideMin;
}

template <typename T, int V>
int launch_t(const void* k, const void* gate, const uint8_t* valid, const float* ape,
             const void* g, const void* be, float eps, const int32_t* cu, const int32_t* cap,
             const int32_t* begin, int B, int kpool, int max_pools, void* pk, int32_t* ps,
             uint8_t* pv, int32_t* np, int32_t* st, cudaStream_t stream) {
  const int gx = max(1, (max_pools + kWarpsPerCta - 1) / kWarpsPerCta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, B, 1);
  cfg.blockDim = dim3(kWarpsPerCta * 32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = launch_kernel(
      &cfg, kpool_compress_kernel<T, V>, (const T*)k, (const T*)gate, valid, ape, (const T*)g,
      (const T*)be, eps, cu, cap, begin, kpool, max_pools, (T*)pk, ps, pv, np, st);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

int kpool_compress_ctas(int B, int kpool, int max_pools) {
  if (max_pools >= kWideMin) {
    const int ppc = wide_pools_per_cta(B, max_pools, kpool <= 4 ? WideCfg<4>::kCtasPerSm
                                                                : WideCfg<8>::kCtasPerSm);
    return (max_pools + ppc - 1) / ppc * B;
  }
  return max(1, (max_pools + kWarpsPerCta - 1) / kWarpsPerCta) * B;
}

int launch_kpool_compress(const void* k, const void* gate, const uint8_t* valid, const float* ape,
                          const void* ln_gamma, const void* ln_beta, float ln_eps,
                          const int32_t* cu_seqlens, const int32_t* cu_pool_cap,
                          const int32_t* pool_begin, int B, int D, int kpool, int max_pools,
                          int dtype, void* pool_keys, int32_t* pool_start, uint8_t* pool_valid,
                          int32_t* n_pools, int32_t* status_dev, cudaStream_t stream) {
  if (uses_wide(D, max_pools, dtype)) {
    if (kpool <= 4)
      return launch_wide<4>(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens,
                            cu_pool_cap, pool_begin, B, kpool, max_pools, pool_keys, pool_start,
                            pool_valid, n_pools, status_dev, stream);
    return launch_wide<8>(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens, cu_pool_cap,
                          pool_begin, B, kpool, max_pools, pool_keys, pool_start, pool_valid,
                          n_pools, status_dev, stream);
  }
#define DSA_COMPRESS_CASE(TT, VV)                                                            \
  return launch_t<TT, VV>(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens,        \
                          cu_pool_cap, pool_begin, B, kpool, max_pools, pool_keys, pool_start, \
                          pool_valid, n_pools, status_dev, stream)
  if (dtype == DSA_BF16) {
    switch (D) {
      case 32: DSA_COMPRESS_CASE(__nv_bfloat16, 1);
      case 64: DSA_COMPRESS_CASE(__nv_bfloat16, 2);
      case 128: DSA_COMPRESS_CASE(__nv_bfloat16, 4);
      case 256: DSA_COMPRESS_CASE(__nv_bfloat16, 8);
    }
  } else {
    switch (D) {
      case 32: DSA_COMPRESS_CASE(float, 1);
      case 64: DSA_COMPRESS_CASE(float, 2);
      case 128: DSA_COMPRESS_CASE(float, 4);
      case 256: DSA_COMPRESS_CASE(float, 8);
    }
  }
#undef DSA_COMPRESS_CASE
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
