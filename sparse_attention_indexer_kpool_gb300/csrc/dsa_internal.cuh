// Internal helpers shared by the libdsa kernels (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/dsa.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libdsa is built for sm_103a only"
#endif

namespace dsa {

constexpr int kKpoolMax = DSA_KPOOL_MAX;

// SMs of the current device (cudaDevAttrMultiProcessorCount, read once per
// device), for launch shapes; 152, the GB300's count, when no device answers.
int num_sms();

// Bounded waits.  A wait on an mbarrier gives up after kWaitNs of the GPU's
// global timer; the kernel then flags DSA_DEV_TIMEOUT, issues nothing more,
// waits (bounded again) for the copies and MMAs it already issued and frees
// its tensor memory before it returns.  Under a failure drill (tests only:
// dsa_set_failure_drill) the tensor-core kernels skip arming the barrier of
// their first wait, and every wait of those launches gives up after
// kDrillWaitNs.
constexpr unsigned long long kWaitNs = 1000000000ull;  // 1 s
constexpr unsigned long long kDrillWaitNs = 1000000ull;  // 1 ms
int failure_drill();  // the drill armed for the launches that follow (0: none)

// ---------------------------------------------------------------- launches
// Every kernel of the library is launched through launch_kernel, which counts
// the launches that succeed (dsa_kernel_launches reports the count).
std::atomic<unsigned long long>& launch_counter();
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(const cudaLaunchConfig_t* cfg, void (*kernel)(KArgs...),
                          Args&&... args) {
  const cudaError_t e = cudaLaunchKernelEx(cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) launch_counter().fetch_add(1, std::memory_order_relaxed);
  return e;
}

// ---------------------------------------------------------------- status
__device__ __forceinline__ void flag(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- dtypes
template <typename T> struct Act;
template <> struct Act<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
  static __device__ __forceinline__ float round(float x) { return x; }
};
template <> struct Act<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static __device__ __forceinline__ float round(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
  }
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits)
  return *reinterpret_cast<uint32_t*>(&p);
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ---------------------------------------------------------------- warp
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- mma.sync
// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// ---------------------------------------------------------------- cp.async (16 B)
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g, bool pred) {
  int n = pred ? 16 : 0;  // src-size 0 zero-fills the destination
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(g), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N));
}
// The same with a count known only after unrolling (0..7; more waits for all).
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  switch (n) {
    case 7: cp_async_wait<7>(); break;
    case 6: cp_async_wait<6>(); break;
    case 5: cp_async_wait<5>(); break;
    case 4: cp_async_wait<4>(); break;
    case 3: cp_async_wait<3>(); break;
    case 2: cp_async_wait<2>(); break;
    case 1: cp_async_wait<1>(); break;
    default: cp_async_wait<0>(); break;
  }
}

// ---------------------------------------------------------------- mbarrier + bulk copy
// 2^x on the special-function unit (ex2.approx, relative error below 2^-22;
// 2^-inf = +0).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: gives up after about `limit_ns` nanoseconds and reports false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;");
}

// ---------------------------------------------------------------- score keys
// Order-preserving map of an fp32 score to uint32 (bigger float -> bigger key);
// -0 is mapped like +0 so the two compare equal.
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ bool is_candidate(float s) { return s > -INFINITY; }

}  // namespace dsa

// ---------------------------------------------------------------- host launchers
namespace dsa {
// CTAs of one launch of the compress kernel (they stay resident while a
// scoring kernel of the same call starts early)
int kpool_compress_ctas(int B, int kpool, int max_pools);
// The compress of the same call, for a scoring kernel that starts before that
// compress has ended: it rewrites pools [pool_begin[b], ...) of sequence b, and
// the pool count it writes follows from the first valid token of the sequence.
struct EarlyStart {
  const int32_t* pool_begin = nullptr;  // nullptr: no early start
  const uint8_t* valid = nullptr;
  const int32_t* cu_seqlens = nullptr;
  // Set (k != nullptr) when the scoring kernel does the compress of its call
  // itself (bf16, D = 128, one pool per sequence from pool_begin[b]): it is
  // then the first kernel of the call, and no compress kernel is launched.
  const __nv_bfloat16* k = nullptr;
  const __nv_bfloat16* gate = nullptr;
  const float* ape = nullptr;
  const __nv_bfloat16* ln_gamma = nullptr;
  const __nv_bfloat16* ln_beta = nullptr;
  float ln_eps = 0.f;
  __nv_bfloat16* pool_keys_out = nullptr;
  int32_t* pool_start_out = nullptr;
  uint8_t* pool_valid_out = nullptr;
  int32_t* n_pools_out = nullptr;
};
// whether launch_index_scores starts the scoring kernel early with es
bool index_early_start(const EarlyStart& es, int Q, const int32_t* q_seq, const int32_t* q_pos,
                       int H, int D, int dtype);
int launch_kpool_compress(const void* k, const void* gate, const uint8_t* valid, const float* ape,
                          const void* ln_gamma, const void* ln_beta, float ln_eps,
                          const int32_t* cu_seqlens, const int32_t* cu_pool_cap,
                          const int32_t* pool_begin, int B, int D, int kpool, int max_pools,
                          int dtype, void* pool_keys, int32_t* pool_start, uint8_t* pool_valid,
                          int32_t* n_pools, int32_t* status_dev, cudaStream_t stream);
int launch_index_scores(const void* q, const float* weights, float scale, const void* pool_keys,
                        int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
                        const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                        const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                        int dtype, float* scores, uint32_t* score_hist, int32_t* status_dev,
                        cudaStream_t stream, EarlyStart early = {}, int busy_ctas = 0);
// tcgen05 index kernel: queries per key tile (1 or 8), 0 when Q does not fit it
int umma_index_group(int Q, const int32_t* q_seq);
int launch_index_scores_umma(const void* q, const float* weights, float scale,
                             const void* pool_keys, int pool_rows, const int32_t* pool_start,
                             const uint8_t* pool_valid, const int32_t* n_pools,
                             const int32_t* cu_pool_cap, const int32_t* q_seq,
                             const int32_t* q_pos, int Q, int B, int kpool, int P_ld,
                             float* scores, uint32_t* hist, EarlyStart early,
                             int32_t* status_dev, cudaStream_t stream, int busy_ctas = 0);
// whether the decode kernel can start streaming before the compress of its call ends
bool umma_index_early_ok(int Q, const int32_t* q_seq, const int32_t* q_pos);
// true when launch_index_scores also counts the per-query score histogram
bool index_fills_histogram(int Q, const int32_t* q_seq, int H, int D, int dtype);
size_t topk_workspace_size(int Q, int P_ld, int select_k);
size_t select_workspace_size(int Q, int P_ld, int select_k);
uint32_t* topk_workspace_hist(void* workspace);
int launch_select_after_index(const float* scores, int Q, int P_ld, int select_k,
                              int32_t* pool_ids, void* workspace, const int32_t* pool_start,
                              const int32_t* cu_pool_cap, const int32_t* q_seq, int B, int kpool,
                              int out_width, int32_t* token_ids, int32_t* status_dev,
                              cudaStream_t stream);
bool index_uses_tensor_cores(int H, int D, int dtype);
int launch_topk_pools(const float* scores, int Q, int P_ld, int select_k, int32_t* pool_ids,
                      void* workspace, size_t ws_bytes, cudaStream_t stream);
int launch_expand_selection(const int32_t* pool_ids, const int32_t* pool_start,
                            const int32_t* cu_pool_cap, const int32_t* q_seq, int Q, int B,
                            int select_k, int kpool, int out_width, int32_t* token_ids,
                            int32_t* status_dev, cudaStream_t stream);
size_t mla_workspace_size(int Q, int Hm, int L, int out_width, int dtype);
// A paged latent cache (dsa_paged_kv after validation).
struct PagedKv {
  const void* pages;
  const float* row_scale;      // E4M3 only
  const int32_t* block_table;  // [B, max_pages]
  const int32_t* seq_lens;     // [B]
  int n_pages, page_size, max_pages, kv_dtype;
};
// tcgen05 attention (bf16, 64 heads, latent 512): one CTA per 128 selected rows
bool mla_umma_ok(int Q, int Hm, int L, int out_width, int dtype);
bool mla_umma_shape_ok(int Hm, int L, int dtype);  // the geometry alone, any number of queries
int mla_umma_splits(int out_width);
// paged: NULL for the contiguous cache (kv + cu_seqlens)
int launch_mla_umma(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                    const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int out_width,
                    float sm_scale, void* out, float* lse, float* part_o, float* part_ml,
                    bool early, int32_t* status_dev, cudaStream_t stream,
                    const PagedKv* paged = nullptr);
// streaming tcgen05 attention (same geometry, many queries): one CTA per query
// and range of 128-row tiles, all 64 heads, online softmax; splits of the tiles
int mla_stream_splits(int Q, int out_width);
int launch_mla_stream(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                      const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int out_width,
                      float sm_scale, void* out, float* lse, float* part_o, float* part_ml,
                      int32_t* status_dev, cudaStream_t stream, const PagedKv* paged = nullptr);
// the paged attention: the tcgen05 kernel for its geometry (any number of
// queries) and bf16 or E4M3 rows, else the generic kernel
size_t mla_paged_workspace_size(int Q, int Hm, int L, int out_width, int dtype, int kv_dtype);
int launch_mla_paged_decode(const void* q_lat, const PagedKv& kv, const int32_t* q_seq,
                            const int32_t* token_ids, int Q, int B, int Hm, int L, int out_width,
                            float sm_scale, int dtype, void* out, float* lse, void* workspace,
                            size_t ws_bytes, int32_t* status_dev, cudaStream_t stream);
// early: the caller guarantees that only the token ids come from kernels still in
// flight (the attention of a fused decode call), so the rest is read before the wait
int launch_mla_selected_decode(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                               const int32_t* q_seq, const int32_t* token_ids, int Q, int B,
                               int Hm, int L, int out_width, float sm_scale, int dtype, void* out,
                               float* lse, void* workspace, size_t ws_bytes, int32_t* status_dev,
                               cudaStream_t stream, bool early = false);
}  // namespace dsa

#define DSA_LAUNCH_CHECK()                          \
  do {                                              \
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA; \
  } while (0)
