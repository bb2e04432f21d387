// C ABI of libdsa: host-side validation, then dispatch to the kernels.
// Nothing is launched and no output is touched when validation fails.
#include <math.h>

#include "dsa_internal.cuh"

namespace {

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
inline bool dtype_ok(int dtype) { return dtype == DSA_BF16 || dtype == DSA_F32; }
inline bool d_ok(int D) { return D == 32 || D == 64 || D == 128 || D == 256; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

constexpr int kNoWork = -1;  // valid call with nothing to do

int check_compress(const void* k, const void* gate, const uint8_t* valid, const float* ape,
                   const void* ln_gamma, const void* ln_beta, float ln_eps,
                   const int32_t* cu_seqlens, const int32_t* cu_pool_cap,
                   const int32_t* pool_begin, int B, int D, int kpool, int max_pools, int dtype,
                   void* pool_keys, int32_t* pool_start, uint8_t* pool_valid, int32_t* n_pools,
                   int32_t* status_dev) {
  if (B < 0 || max_pools < 0) return DSA_ERR_INVALID_ARG;
  if (kpool < 1 || kpool > DSA_KPOOL_MAX) return DSA_ERR_INVALID_ARG;  // refuse, never truncate
  if (!dtype_ok(dtype) || !(ln_eps >= 0.f) || !isfinite(ln_eps)) return DSA_ERR_INVALID_ARG;
  if (!d_ok(D)) return DSA_ERR_UNSUPPORTED;
  if (B == 0) return kNoWork;
  if (!k || !gate || !valid || !ape || !ln_gamma || !ln_beta || !cu_seqlens || !cu_pool_cap ||
      !pool_keys || !pool_start || !pool_valid || !n_pools)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(gate, 16) || !aligned(pool_keys, 16) || !aligned(ln_gamma, 16) ||
      !aligned(ln_beta, 16) || !aligned(ape, 4) || !aligned(cu_seqlens, 4) ||
      !aligned(cu_pool_cap, 4) || !aligned(pool_start, 4) || !aligned(n_pools, 4) ||
      (pool_begin && !aligned(pool_begin, 4)) || (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  if (B > 65535) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

int check_select(const void* q, const float* weights, float scale, const void* pool_keys,
                 int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
                 const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                 const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                 int select_k, int out_width, int dtype, float* scores, int32_t* pool_ids,
                 int32_t* token_ids, void* workspace, size_t ws_bytes, int32_t* status_dev) {
  if (Q < 0 || B < 0 || H < 1 || P_ld < 1 || select_k < 1 || out_width < 1 || pool_rows < 1)
    return DSA_ERR_INVALID_ARG;
  if (kpool < 1 || kpool > DSA_KPOOL_MAX) return DSA_ERR_INVALID_ARG;
  if ((long long)out_width < (long long)select_k * kpool) return DSA_ERR_INVALID_ARG;
  if (!dtype_ok(dtype) || !(scale > 0.f) || !isfinite(scale)) return DSA_ERR_INVALID_ARG;
  if (!d_ok(D) || H > 64 || select_k > DSA_SELECT_K_MAX) return DSA_ERR_UNSUPPORTED;
  if (Q == 0) return kNoWork;
  if (B == 0) return DSA_ERR_INVALID_ARG;
  if (!q || !weights || !pool_keys || !pool_start || !pool_valid || !n_pools || !cu_pool_cap ||
      !scores || !pool_ids || !token_ids)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(weights, 16) || !aligned(pool_keys, 16) || !aligned(scores, 4) ||
      !aligned(n_pools, 4) || !aligned(cu_pool_cap, 4) || !aligned(pool_start, 4) ||
      !aligned(pool_ids, 4) || !aligned(token_ids, 4) || (q_seq && !aligned(q_seq, 4)) ||
      (q_pos && !aligned(q_pos, 4)) || (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  if (!workspace || ws_bytes < dsa::select_workspace_size(Q, P_ld, select_k))
    return DSA_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return DSA_ERR_MISALIGNED;
  if (Q > 65535) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

// index_scores -> top-k (+ expansion); early: see dsa::EarlyStart
int run_select(const void* q, const float* weights, float scale, const void* pool_keys,
               int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
               const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
               const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
               int select_k, int out_width, int dtype, float* scores, int32_t* pool_ids,
               int32_t* token_ids, void* workspace, int32_t* status_dev, cudaStream_t st,
               dsa::EarlyStart early = {}, int busy_ctas = 0) {
  // Decode geometry: the scoring kernel also counts each query's score
  // histogram into the workspace and the selection starts from it.  Otherwise
  // the selection kernel builds the histogram itself.
  const bool hist = dsa::index_fills_histogram(Q, q_seq, H, D, dtype);
  int r = dsa::launch_index_scores(q, weights, scale, pool_keys, pool_rows, pool_start,
                                   pool_valid, n_pools, cu_pool_cap, q_seq, q_pos, Q, B, H, D,
                                   kpool, P_ld, dtype, scores,
                                   hist ? dsa::topk_workspace_hist(workspace) : nullptr,
                                   status_dev, st, early, busy_ctas);
  if (r != DSA_OK) return r;
  return dsa::launch_select_after_index(scores, Q, P_ld, select_k, pool_ids,
                                        hist ? workspace : nullptr, pool_start, cu_pool_cap,
                                        q_seq, B, kpool, out_width, token_ids, status_dev, st);
}

int check_mla(const void* q_lat, const void* kv_latent, const int32_t* cu_seqlens,
              const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int Hm, int L,
              int out_width, float sm_scale, int dtype, void* out, float* lse, void* workspace,
              size_t ws_bytes, int32_t* status_dev) {
  if (Q < 0 || B < 0 || Hm < 1 || L < 1 || out_width < 1) return DSA_ERR_INVALID_ARG;
  if (!dtype_ok(dtype) || !isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  if (L % 8 != 0 || L > 1024 || Hm > 128) return DSA_ERR_UNSUPPORTED;
  if (Q == 0) return kNoWork;
  if (B == 0) return DSA_ERR_INVALID_ARG;
  if (!q_lat || !kv_latent || !cu_seqlens || !token_ids || !out) return DSA_ERR_INVALID_ARG;
  if (!aligned(q_lat, 16) || !aligned(kv_latent, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens, 4) || !aligned(token_ids, 4) || (lse && !aligned(lse, 4)) ||
      (q_seq && !aligned(q_seq, 4)) || (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  const size_t need = dsa::mla_workspace_size(Q, Hm, L, out_width, dtype);
  if (need > 0 && (!workspace || ws_bytes < need)) return DSA_ERR_WORKSPACE;
  if (workspace && !aligned(workspace, 16)) return DSA_ERR_MISALIGNED;
  if (Q > 65535) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int check_mla_paged(const void* q_lat, const dsa_paged_kv* kv, const int32_t* q_seq,
                    const int32_t* token_ids, int Q, int B, int Hm, int L, int out_width,
                    float sm_scale, int dtype, void* out, float* lse, void* workspace,
                    size_t ws_bytes, int32_t* status_dev) {
  if (!kv || Q < 0 || B < 0 || Hm < 1 || L < 1 || out_width < 1) return DSA_ERR_INVALID_ARG;
  if (!dtype_ok(dtype) || !isfinite(sm_scale)) return DSA_ERR_INVALID_ARG;
  const int kd = kv->kv_dtype;
  if (kd != DSA_BF16 && kd != DSA_F32 && kd != DSA_FP8_E4M3) return DSA_ERR_INVALID_ARG;
  if (kv->n_pages < 1 || kv->page_size < 1 || kv->max_pages < 1) return DSA_ERR_INVALID_ARG;
  if ((kd == DSA_FP8_E4M3) != (kv->row_scale != nullptr)) return DSA_ERR_INVALID_ARG;
  if (L % 8 != 0 || L > 1024 || Hm > 128) return DSA_ERR_UNSUPPORTED;
  if ((long long)kv->n_pages * kv->page_size > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  if (Q == 0) return kNoWork;
  if (B == 0) return DSA_ERR_INVALID_ARG;
  if (!q_lat || !kv->pages || !kv->block_table || !kv->seq_lens || !token_ids || !out)
    return DSA_ERR_INVALID_ARG;
  if (!aligned(q_lat, 16) || !aligned(kv->pages, 16) || !aligned(out, 16) ||
      !aligned(kv->block_table, 4) || !aligned(kv->seq_lens, 4) || !aligned(token_ids, 4) ||
      (kv->row_scale && !aligned(kv->row_scale, 4)) || (lse && !aligned(lse, 4)) ||
      (q_seq && !aligned(q_seq, 4)) || (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  const size_t need = dsa::mla_paged_workspace_size(Q, Hm, L, out_width, dtype, kd);
  if (need > 0 && (!workspace || ws_bytes < need)) return DSA_ERR_WORKSPACE;
  if (workspace && !aligned(workspace, 16)) return DSA_ERR_MISALIGNED;
  if (Q > 65535) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

}  // namespace

namespace dsa {
std::atomic<unsigned long long>& launch_counter() {
  static std::atomic<unsigned long long> n{0};
  return n;
}

namespace {
std::atomic<int> g_drill{0};
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
}  // namespace

int failure_drill() { return g_drill.load(std::memory_order_relaxed); }

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 152;
  }
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 152;
  }
  g_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}
}  // namespace dsa

extern "C" {

int dsa_version(void) { return 10000; }

uint64_t dsa_kernel_launches(void) { return dsa::launch_counter().load(); }

int dsa_set_failure_drill(int drill) {
  if (drill != 0 && drill != DSA_DRILL_SKIP_ARM && drill != DSA_DRILL_SKIP_PV_COMMIT)
    return DSA_ERR_INVALID_ARG;
  dsa::g_drill.store(drill, std::memory_order_relaxed);
  return DSA_OK;
}

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: bad size, null pointer or kpool";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED: pointer alignment";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: geometry or dtype";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing or too small";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: kernel launch failed";
    default: return "DSA_ERR_UNKNOWN";
  }
}

int dsa_kpool_compress(const void* k, const void* gate, const uint8_t* valid, const float* ape,
                       const void* ln_gamma, const void* ln_beta, float ln_eps,
                       const int32_t* cu_seqlens, const int32_t* cu_pool_cap,
                       const int32_t* pool_begin, int B, int D, int kpool, int max_pools,
                       int dtype, void* pool_keys, int32_t* pool_start, uint8_t* pool_valid,
                       int32_t* n_pools, int32_t* status_dev, void* stream) {
  const int r = check_compress(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens,
                               cu_pool_cap, pool_begin, B, D, kpool, max_pools, dtype, pool_keys,
                               pool_start, pool_valid, n_pools, status_dev);
  if (r != DSA_OK) return r == kNoWork ? DSA_OK : r;
  return dsa::launch_kpool_compress(k, gate, valid, ape, ln_gamma, ln_beta, ln_eps, cu_seqlens,
                                    cu_pool_cap, pool_begin, B, D, kpool, max_pools, dtype,
                                    pool_keys, pool_start, pool_valid, n_pools, status_dev,
                                    as_stream(stream));
}

int dsa_index_scores(const void* q, const float* weights, float scale, const void* pool_keys,
                     int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
                     const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                     const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                     int dtype, float* scores, int32_t* status_dev, void* stream) {
  if (Q < 0 || B < 0 || H < 1 || P_ld < 1 || pool_rows < 1) return DSA_ERR_INVALID_ARG;
  if (kpool < 1 || kpool > DSA_KPOOL_MAX) return DSA_ERR_INVALID_ARG;
  if (!dtype_ok(dtype) || !(scale > 0.f) || !isfinite(scale)) return DSA_ERR_INVALID_ARG;
  if (!d_ok(D) || H > 64) return DSA_ERR_UNSUPPORTED;
  if (Q == 0) return DSA_OK;
  if (B == 0) return DSA_ERR_INVALID_ARG;
  if (!q || !weights || !pool_keys || !pool_valid || !n_pools || !cu_pool_cap || !scores)
    return DSA_ERR_INVALID_ARG;
  if (q_pos && !pool_start) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(weights, 16) || !aligned(pool_keys, 16) || !aligned(scores, 4) ||
      !aligned(n_pools, 4) || !aligned(cu_pool_cap, 4) || (q_seq && !aligned(q_seq, 4)) ||
      (q_pos && !aligned(q_pos, 4)) || (pool_start && !aligned(pool_start, 4)) ||
      (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  if (Q > 65535) return DSA_ERR_UNSUPPORTED;
  return dsa::launch_index_scores(q, weights, scale, pool_keys, pool_rows, pool_start, pool_valid,
                                  n_pools, cu_pool_cap, q_seq, q_pos, Q, B, H, D, kpool, P_ld,
                                  dtype, scores, nullptr, status_dev, as_stream(stream));
}

size_t dsa_topk_pools_workspace_size(int Q, int P_ld, int select_k) {
  if (Q <= 0 || P_ld <= 0 || select_k <= 0) return 0;
  return dsa::topk_workspace_size(Q, P_ld, select_k);  // 0: the histogram lives on chip
}

int dsa_topk_pools(const float* scores, int Q, int P_ld, int select_k, int32_t* pool_ids,
                   void* workspace, size_t ws_bytes, void* stream) {
  if (Q < 0 || P_ld < 1 || select_k < 1) return DSA_ERR_INVALID_ARG;
  if (select_k > DSA_SELECT_K_MAX) return DSA_ERR_UNSUPPORTED;
  if (Q == 0) return DSA_OK;
  if (Q > 65535) return DSA_ERR_UNSUPPORTED;
  if (!scores || !pool_ids) return DSA_ERR_INVALID_ARG;
  if (!aligned(scores, 4) || !aligned(pool_ids, 4)) return DSA_ERR_MISALIGNED;
  if (ws_bytes < dsa::topk_workspace_size(Q, P_ld, select_k)) return DSA_ERR_WORKSPACE;
  if (workspace && !aligned(workspace, 16)) return DSA_ERR_MISALIGNED;
  return dsa::launch_topk_pools(scores, Q, P_ld, select_k, pool_ids, workspace, ws_bytes,
                                as_stream(stream));
}

int dsa_expand_selection(const int32_t* pool_ids, const int32_t* pool_start,
                         const int32_t* cu_pool_cap, const int32_t* q_seq, int Q, int B,
                         int select_k, int kpool, int out_width, int32_t* token_ids,
                         int32_t* status_dev, void* stream) {
  if (Q < 0 || B < 0 || select_k < 1 || out_width < 1) return DSA_ERR_INVALID_ARG;
  if (kpool < 1 || kpool > DSA_KPOOL_MAX) return DSA_ERR_INVALID_ARG;
  if ((long long)out_width < (long long)select_k * kpool) return DSA_ERR_INVALID_ARG;
  if (Q == 0) return DSA_OK;
  if (B == 0) return DSA_ERR_INVALID_ARG;
  if (!pool_ids || !pool_start || !cu_pool_cap || !token_ids) return DSA_ERR_INVALID_ARG;
  if (!aligned(pool_ids, 4) || !aligned(pool_start, 4) || !aligned(cu_pool_cap, 4) ||
      !aligned(token_ids, 4) || (q_seq && !aligned(q_seq, 4)) ||
      (status_dev && !aligned(status_dev, 4)))
    return DSA_ERR_MISALIGNED;
  if (Q > 65535) return DSA_ERR_UNSUPPORTED;
  return dsa::launch_expand_selection(pool_ids, pool_start, cu_pool_cap, q_seq, Q, B, select_k,
                                      kpool, out_width, token_ids, status_dev, as_stream(stream));
}

size_t dsa_select_workspace_size(int Q, int P_ld, int select_k) {
  if (Q <= 0 || P_ld <= 0 || select_k <= 0) return 0;
  return dsa::select_workspace_size(Q, P_ld, select_k);
}

int dsa_select(const void* q, const float* weights, float scale, const void* pool_keys,
               int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
               const int32_t* n_pools,
               const int32_t* cu_pool_cap, const int32_t* q_seq, const int32_t* q_pos, int Q,
               int B, int H, int D, int kpool, int P_ld, int select_k, int out_width, int dtype,
               float* scores, int32_t* pool_ids, int32_t* token_ids, void* workspace,
               size_t ws_bytes, int32_t* status_dev, void* stream) {
  const int r = check_select(q, weights, scale, pool_keys, pool_rows, pool_start, pool_valid,
                             n_pools, cu_pool_cap, q_seq, q_pos, Q, B, H, D, kpool, P_ld,
                             select_k, out_width, dtype, scores, pool_ids, token_ids, workspace,
                             ws_bytes, status_dev);
  if (r != DSA_OK) return r == kNoWork ? DSA_OK : r;
  return run_select(q, weights, scale, pool_keys, pool_rows, pool_start, pool_valid, n_pools,
                    cu_pool_cap, q_seq, q_pos, Q, B, H, D, kpool, P_ld, select_k, out_width,
                    dtype, scores, pool_ids, token_ids, workspace, status_dev, as_stream(stream));
}

size_t dsa_mla_selected_decode_workspace_size(int Q, int Hm, int L, int out_width, int dtype) {
  if (Q <= 0 || Hm <= 0 || L <= 0 || out_width <= 0 || !dtype_ok(dtype)) return 0;
  return dsa::mla_workspace_size(Q, Hm, L, out_width, dtype);
}

int dsa_mla_selected_decode(const void* q_lat, const void* kv_latent, const int32_t* cu_seqlens,
                            const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int Hm,
                            int L, int out_width, float sm_scale, int dtype, void* out,
                            float* lse, void* workspace, size_t ws_bytes, int32_t* status_dev,
                            void* stream) {
  const int r = check_mla(q_lat, kv_latent, cu_seqlens, q_seq, token_ids, Q, B, Hm, L, out_width,
                          sm_scale, dtype, out, lse, workspace, ws_bytes, status_dev);
  if (r != DSA_OK) return r == kNoWork ? DSA_OK : r;
  return dsa::launch_mla_selected_decode(q_lat, kv_latent, cu_seqlens, q_seq, token_ids, Q, B, Hm,
                                         L, out_width, sm_scale, dtype, out, lse, workspace,
                                         ws_bytes, status_dev, as_stream(stream));
}

size_t dsa_mla_paged_decode_workspace_size(int Q, int Hm, int L, int out_width, int dtype,
                                           int kv_dtype) {
  if (Q <= 0 || Hm <= 0 || L <= 0 || out_width <= 0 || !dtype_ok(dtype)) return 0;
  return dsa::mla_paged_workspace_size(Q, Hm, L, out_width, dtype, kv_dtype);
}

int dsa_mla_paged_decode(const void* q_lat, const dsa_paged_kv* kv, const int32_t* q_seq,
                         const int32_t* token_ids, int Q, int B, int Hm, int L, int out_width,
                         float sm_scale, int dtype, void* out, float* lse, void* workspace,
                         size_t ws_bytes, int32_t* status_dev, void* stream) {
  const int r = check_mla_paged(q_lat, kv, q_seq, token_ids, Q, B, Hm, L, out_width, sm_scale,
                                dtype, out, lse, workspace, ws_bytes, status_dev);
  if (r != DSA_OK) return r == kNoWork ? DSA_OK : r;
  const dsa::PagedKv pk{kv->pages,    kv->row_scale, kv->block_table, kv->seq_lens,
                        kv->n_pages,  kv->page_size, kv->max_pages,   kv->kv_dtype};
  return dsa::launch_mla_paged_decode(q_lat, pk, q_seq, token_ids, Q, B, Hm, L, out_width,
                                      sm_scale, dtype, out, lse, workspace, ws_bytes, status_dev,
                                      as_stream(stream));
}

size_t dsa_decode_layer_workspace_size(const dsa_decode_layer_args* a, size_t* ws_select,
                                       size_t* ws_mla) {
  if (!a) return 0;
  const size_t s = (a->Q > 0 && a->P_ld > 0 && a->select_k > 0)
                       ? dsa::select_workspace_size(a->Q, a->P_ld, a->select_k)
                       : 0;
  const size_t m = (a->Q > 0 && a->Hm > 0 && a->L > 0 && a->out_width > 0 && dtype_ok(a->dtype))
                       ? dsa::mla_workspace_size(a->Q, a->Hm, a->L, a->out_width, a->dtype)
                       : 0;
  if (ws_select) *ws_select = s;
  if (ws_mla) *ws_mla = m;
  return s + m;
}

int dsa_decode_layer(const dsa_decode_layer_args* a, void* stream) {
  if (!a) return DSA_ERR_INVALID_ARG;
  // every stage is checked before anything is launched
  const int rc = check_compress(a->k, a->gate, a->valid, a->ape, a->ln_gamma, a->ln_beta,
                                a->ln_eps, a->cu_seqlens, a->cu_pool_cap, a->pool_begin, a->B,
                                a->D, a->kpool, a->max_pools, a->dtype, a->pool_keys,
                                a->pool_start, a->pool_valid, a->n_pools, a->status_dev);
  if (rc != DSA_OK && rc != kNoWork) return rc;
  const int rs = check_select(a->q, a->weights, a->scale, a->pool_keys, a->pool_rows,
                              a->pool_start, a->pool_valid, a->n_pools, a->cu_pool_cap, a->q_seq,
                              a->q_pos, a->Q, a->B, a->H, a->D, a->kpool, a->P_ld, a->select_k,
                              a->out_width, a->dtype, a->scores, a->pool_ids, a->token_ids,
                              a->ws_select, a->ws_select_bytes, a->status_dev);
  if (rs != DSA_OK && rs != kNoWork) return rs;
  const int rm = check_mla(a->q_lat, a->kv_latent, a->cu_seqlens, a->q_seq, a->token_ids, a->Q,
                           a->B, a->Hm, a->L, a->out_width, a->sm_scale, a->dtype, a->out, a->lse,
                           a->ws_mla, a->ws_mla_bytes, a->status_dev);
  if (rm != DSA_OK && rm != kNoWork) return rm;
  cudaStream_t st = as_stream(stream);
  int r;
  // Inside this call the scoring kernel may stream the key tiles below
  // pool_begin[b] before the compress ends (it does not write them); with no
  // pool_begin the compress rewrites every pool.
  dsa::EarlyStart es = rc == DSA_OK ? dsa::EarlyStart{a->pool_begin, a->valid, a->cu_seqlens}
                                    : dsa::EarlyStart{};
  // A decode step (one new pool per sequence) on the tensor-core scoring path:
  // the scoring kernel does that compress itself and is the call's first kernel.
  const bool fuse = rc == DSA_OK && rs == DSA_OK && a->max_pools == 1 && a->dtype == DSA_BF16 &&
                    a->D == 128 &&
                    dsa::index_early_start(es, a->Q, a->q_seq, a->q_pos, a->H, a->D, a->dtype);
  if (fuse) {
    es.k = static_cast<const __nv_bfloat16*>(a->k);
    es.gate = static_cast<const __nv_bfloat16*>(a->gate);
    es.ape = a->ape;
    es.ln_gamma = static_cast<const __nv_bfloat16*>(a->ln_gamma);
    es.ln_beta = static_cast<const __nv_bfloat16*>(a->ln_beta);
    es.ln_eps = a->ln_eps;
    es.pool_keys_out = static_cast<__nv_bfloat16*>(a->pool_keys);
    es.pool_start_out = a->pool_start;
    es.pool_valid_out = a->pool_valid;
    es.n_pools_out = a->n_pools;
  } else if (rc == DSA_OK) {
    r = dsa::launch_kpool_compress(a->k, a->gate, a->valid, a->ape, a->ln_gamma, a->ln_beta,
                                   a->ln_eps, a->cu_seqlens, a->cu_pool_cap, a->pool_begin, a->B,
                                   a->D, a->kpool, a->max_pools, a->dtype, a->pool_keys,
                                   a->pool_start, a->pool_valid, a->n_pools, a->status_dev, st);
    if (r != DSA_OK) return r;
  }
  if (rs == kNoWork) return DSA_OK;  // no queries: nothing to select or attend
  r = run_select(a->q, a->weights, a->scale, a->pool_keys, a->pool_rows, a->pool_start,
                 a->pool_valid, a->n_pools, a->cu_pool_cap, a->q_seq, a->q_pos, a->Q, a->B, a->H,
                 a->D, a->kpool, a->P_ld, a->select_k, a->out_width, a->dtype, a->scores,
                 a->pool_ids, a->token_ids, a->ws_select, a->status_dev, st, es,
                 // SMs the scoring grid leaves to the compress kernel beside it; the
                 // fused form keeps the same grid (with every SM: 0.4088 against
                 // 0.4066 ms per 262k decode step)
                 (rc == DSA_OK && !fuse) ? dsa::kpool_compress_ctas(a->B, a->kpool, a->max_pools)
                                         : (fuse ? a->B : 0));
  if (r != DSA_OK) return r;
  // the attention's inputs other than the token ids predate this call
  return dsa::launch_mla_selected_decode(a->q_lat, a->kv_latent, a->cu_seqlens, a->q_seq,
                                         a->token_ids, a->Q, a->B, a->Hm, a->L, a->out_width,
                                         a->sm_scale, a->dtype, a->out, a->lse, a->ws_mla,
                                         a->ws_mla_bytes, a->status_dev, st, true);
}

}  // extern "C"
