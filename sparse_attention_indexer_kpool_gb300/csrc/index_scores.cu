// index_scores: score[q, p] = sum_h w[q, h] * max(0, scale * <q[q, h, :], key[p, :]>).
//
// Module glm5next_dsa::tp, "Why the indexer is REPLICATED, not sharded": a plain
// sum over heads of weights[h] * relu(scale * dot); module glm5next_dsa, "Shape
// of the pipeline": [Q, P] scores with candidate validity (-inf here).
//
// Dispatch: the bf16 / 32-head / 128-channel geometry of the indexer runs on
// the tcgen05 kernel (index_scores_umma.cu); every other geometry (fp32, other
// head counts or head dims) runs on the SIMT kernel below.
#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kH = 32, kD = 128;  // the tensor-core geometry

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

bool index_fills_histogram(int Q, const int32_t* q_seq, int H, int D, int dtype) {
  return index_uses_tensor_cores(H, D, dtype) && umma_index_group(Q, q_seq) == 1;
}

bool index_early_start(const EarlyStart& es, int Q, const int32_t* q_seq, const int32_t* q_pos,
                       int H, int D, int dtype) {
  return es.pool_begin != nullptr && es.valid != nullptr && es.cu_seqlens != nullptr &&
         index_uses_tensor_cores(H, D, dtype) && umma_index_group(Q, q_seq) == 1 &&
         umma_index_early_ok(Q, q_seq, q_pos);
}

int launch_index_scores(const void* q, const float* weights, float scale, const void* pool_keys,
                        int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
                        const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                        const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                        int dtype, float* scores, uint32_t* score_hist, int32_t* status_dev,
                        cudaStream_t stream, EarlyStart early, int busy_ctas) {
  if (index_uses_tensor_cores(H, D, dtype) && umma_index_group(Q, q_seq) != 0)
    return launch_index_scores_umma(q, weights, scale, pool_keys, pool_rows, pool_start,
                                    pool_valid, n_pools, cu_pool_cap, q_seq, q_pos, Q, B, kpool,
                                    P_ld, scores, score_hist, early, status_dev, stream,
                                    busy_ctas);
  // the SIMT kernel fills no histogram; callers ask index_fills_histogram first
  cudaLaunchAttribute attr = pdl_attr();
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (H < 1 || H > 64 || (D != 32 && D != 64 && D != 128 && D != 256)) return DSA_ERR_UNSUPPORTED;
  const size_t smem = ((size_t)H * D + H) * 4;
  cfg.gridDim = dim3((P_ld + 127) / 128, Q, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaError_t e;
  if (dtype == DSA_BF16) {
    cudaFuncSetAttribute(index_scores_simt_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
    e = launch_kernel(&cfg, index_scores_simt_kernel<__nv_bfloat16>,
                      (const __nv_bfloat16*)q, weights, scale,
                      (const __nv_bfloat16*)pool_keys, pool_start, pool_valid, n_pools,
                      cu_pool_cap, q_seq, q_pos, B, H, D, kpool, P_ld, scores, status_dev);
  } else {
    cudaFuncSetAttribute(index_scores_simt_kernel<float>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, 80 * 1024);
    e = launch_kernel(&cfg, index_scores_simt_kernel<float>, (const float*)q, weights, scale,
                      (const float*)pool_keys, pool_start, pool_valid, n_pools, cu_pool_cap,
                      q_seq, q_pos, B, H, D, kpool, P_ld, scores, status_dev);
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
