/*
 * dsa.h - C ABI of libdsa: DeepSeek-Sparse-Attention kpool token selection and
 * selected-row NoPE MLA decode for one GLM-5.3-Flash-style layer, on GB300
 * (sm_103a).
 *
 * The five stage entry points follow the stage list of the DSA module page
 * (module glm5next_dsa, "Shape of the pipeline"):
 *
 *   k, gate, valid, ape -> dsa_kpool_compress -> pool keys / starts / valid
 *                       -> dsa_index_scores   -> [Q, P_ld] fp32 scores (-inf = not a candidate)
 *                       -> dsa_topk_pools     -> [Q, select_k] pool ids
 *                       -> dsa_expand_selection -> [Q, out_width] token ids (-1 = none)
 *                       -> dsa_mla_selected_decode -> [Q, Hm, L] latent output + lse
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Ownership:  the caller allocates and owns every buffer, workspaces included
 *             (sizes from the *_workspace_size queries).  The library never
 *             allocates, frees or synchronizes; it keeps no state between calls.
 * Pointers:   every tensor pointer is a DEVICE pointer of the current CUDA
 *             device.  Tensors are dense, row-major, with the shapes given per
 *             argument.  bf16/fp32 activation rows must start on 16-byte
 *             boundaries (row sizes here are multiples of 16 bytes).
 * Streams:    `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *             stream).  Every call is asynchronous on that stream and may be
 *             captured into a CUDA graph.
 * Geometry:   every size is an explicit argument; nothing is defaulted (module
 *             glm5next_dsa, Structs, Glm5NextDsaConfig: geometry is read from
 *             the checkpoint config, never defaulted).
 * Validation: arguments are checked on the host before anything is launched.
 *             On any error the call returns a non-zero DSA_ERR_* code, launches
 *             nothing and writes no output.  Nothing is silently truncated: a
 *             kpool above 8 is refused (module glm5next_dsa, Constants,
 *             KERNEL_MAX_KPOOL).
 * Device faults: faults only the device can see (a token id outside its
 *             sequence, a pool count larger than its cache slice, ...) are
 *             OR-ed as DSA_DEV_* bits into *status_dev when status_dev is not
 *             NULL; the offending item is skipped, never trapped.  The caller
 *             zeroes *status_dev and reads it back when convenient.
 * Empty work: Q == 0 or B == 0 is a valid no-op returning DSA_OK.
 *
 * Layouts
 * -------
 * Token axis: the B sequences are concatenated; sequence b owns rows
 *   [cu_seqlens[b], cu_seqlens[b+1]) of k, gate, valid and kv_latent.  Its
 *   tokens are numbered 0..T_b-1 on its own axis, left padding included.
 * Pool cache: sequence b owns entries [cu_pool_cap[b], cu_pool_cap[b+1]) of
 *   pool_keys / pool_start / pool_valid (its capacity cap_b).  Pool ids and
 *   pool_start values are local to the sequence.
 * Queries: query q reads sequence q_seq[q] (q_seq == NULL: every query reads
 *   sequence 0; pass cache pointers offset to the wanted sequence).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------ */
#define DSA_OK 0
#define DSA_ERR_INVALID_ARG 1  /* bad size, null pointer, kpool not in [1,8], out_width too small */
#define DSA_ERR_MISALIGNED 2   /* a pointer is not aligned as documented                         */
#define DSA_ERR_UNSUPPORTED 3  /* geometry / dtype combination the library has no kernel for     */
#define DSA_ERR_WORKSPACE 4    /* workspace missing or smaller than the size query returns       */
#define DSA_ERR_CUDA 5         /* a CUDA launch failed (cudaGetLastError after the launch)       */

/* ---- activation dtypes ------------------------------------------------- */
#define DSA_BF16 0
#define DSA_F32 1
#define DSA_FP8_E4M3 2  /* paged latent rows only: 8-bit E4M3 codes, one fp32 scale per row */

/* ---- device status bits (OR-ed into *status_dev) ----------------------- */
#define DSA_DEV_BAD_TOKEN 1        /* MLA: token id >= T_b; the row is skipped          */
#define DSA_DEV_POOL_OVERFLOW 2    /* compress: more complete pools than cap_b           */
#define DSA_DEV_POOL_UNCOVERED 4   /* compress: complete pools past pool_begin+max_pools */
#define DSA_DEV_BAD_POOL_ID 8      /* expand: pool id >= cap_b; expands to -1            */
#define DSA_DEV_BAD_QSEQ 16        /* q_seq[q] outside [0, B); the query gets no output  */
#define DSA_DEV_POOL_RANGE 32      /* index: n_pools[b] > cap_b or > P_ld; clamped       */
#define DSA_DEV_TIMEOUT 64         /* a bounded wait inside a kernel gave up             */
#define DSA_DEV_BAD_PAGE 256      /* paged MLA: block past the table or page outside
                                      [0, n_pages); the row is skipped              */
#define DSA_DEV_HIST_MISMATCH 128  /* dsa_select: workspace histogram did not match the
                                      scores (workspace not zero-filled); exact fallback ran */

#define DSA_KPOOL_MAX 8            /* module glm5next_dsa, Constants, KERNEL_MAX_KPOOL   */
#define DSA_SELECT_K_MAX 4096

/*
 * dsa_kpool_compress - LayerNorm the indexer keys and pool them kpool at a time.
 *
 * Source: module glm5next_dsa, "Shape of the pipeline" (k, gate, valid, ape ->
 * kpool_compress -> pool keys / indices / valid) and "Traps carried from Slice
 * 8": k_norm is a LayerNorm with bias, not RMSNorm; the pool softmax runs over
 * the slot axis per channel; pooling starts at the first valid token; a pool
 * counts only if every slot is valid.  Constants, LAYERNORM_MODULE: the
 * LayerNorm output is stored in the activation dtype before pooling.
 *
 * For sequence b: t0 = first token with valid != 0 (T_b if none),
 * P_b = floor((T_b - t0) / kpool).  Pool p covers tokens t0 + p*kpool + s:
 *   kn[s]      = LayerNorm(k[token]) * ln_gamma + ln_beta   (population variance,
 *                ln_eps inside the square root), rounded to the activation dtype
 *   logit[s,d] = gate[token, d] + ape[s, d]
 *   key[p, d]  = sum_s softmax_s(logit[., d]) * kn[s][d], rounded to the dtype
 *   pool_start[p] = t0 + p*kpool;  pool_valid[p] = all slots valid.
 * Written pools: p in [pool_begin[b], min(pool_begin[b] + max_pools, cap_b)).
 * Of those, p < P_b are computed and p >= P_b get the sentinel (key 0, start
 * -1, valid 0).  Other entries are not touched (decode: pass the first pool
 * that may have completed since the previous call).  n_pools[b] = min(P_b, cap_b).
 *
 *   k, gate     [sum T_b, D]  activation dtype
 *   valid       [sum T_b]     uint8 (0 = padding / not a token)
 *   ape         [kpool, D]    fp32, added to the gate logits per slot
 *   ln_gamma, ln_beta [D]     activation dtype
 *   cu_seqlens  [B+1] int32, cu_pool_cap [B+1] int32
 *   pool_begin  [B] int32 or NULL (all zero)
 *   max_pools   >= 0: launch extent in pools per sequence
 *   pool_keys   [sum cap_b, D] activation dtype; pool_start [sum cap_b] int32;
 *   pool_valid  [sum cap_b] uint8; n_pools [B] int32
 * Supported: D in {32, 64, 128, 256}; kpool in [1, 8]; dtype DSA_BF16 or DSA_F32.
 * Device faults: DSA_DEV_POOL_OVERFLOW, DSA_DEV_POOL_UNCOVERED.
 */
int dsa_kpool_compress(const void* k, const void* gate, const uint8_t* valid, const float* ape,
                       const void* ln_gamma, const void* ln_beta, float ln_eps,
                       const int32_t* cu_seqlens, const int32_t* cu_pool_cap,
                       const int32_t* pool_begin, int B, int D, int kpool, int max_pools,
                       int dtype, void* pool_keys, int32_t* pool_start, uint8_t* pool_valid,
                       int32_t* n_pools, int32_t* status_dev, void* stream);

/*
 * dsa_index_scores - score every pool of the query's sequence.
 *
 * Source: module glm5next_dsa::tp, "Why the indexer is REPLICATED, not
 * sharded": the score is a plain sum over heads of weights[h] * relu(scale *
 * dot); module glm5next_dsa, "Shape of the pipeline": [Q, P] scores plus
 * candidate validity.
 *
 *   scores[q, p] = sum_h weights[q, h] * max(0, scale * <q[q, h, :], pool_keys[p, :]>)
 * for a candidate pool, -inf otherwise; -0 is written as +0; every one of the
 * P_ld entries of a row is written.  Pool p of sequence b is a candidate when
 * p < n_pools[b], pool_valid[p] != 0 and, if q_pos is not NULL,
 * pool_start[p] + kpool - 1 <= q_pos[q] (the pool is complete at the query's
 * position).  pool_start must be as dsa_kpool_compress wrote it.
 *
 *   q        [Q, H, D] activation dtype;  weights [Q, H] fp32;  scale > 0
 *   pool_keys the cache written by dsa_kpool_compress, pool_rows rows of D
 *            (pool_rows >= cu_pool_cap[B]; no row at or past it is read)
 *   pool_*   the rest of that cache (pool_start may be NULL when q_pos is
 *            NULL); n_pools [B]; cu_pool_cap [B+1]
 *   q_seq    [Q] int32 or NULL;  q_pos [Q] int32 or NULL (every complete pool)
 *   scores   [Q, P_ld] fp32
 * Supported: any H in [1, 64] and D in {32, 64, 128, 256} for both dtypes;
 * H = 32, D = 128, bf16 runs on the tcgen05 tensor cores (with q_seq == NULL
 * and Q >= 64, eight queries share each key tile: the dense prefill-chunk
 * form).  pool_keys and q must be 16-byte aligned.
 * Device faults: DSA_DEV_BAD_QSEQ, DSA_DEV_POOL_RANGE.
 */
int dsa_index_scores(const void* q, const float* weights, float scale, const void* pool_keys,
                     int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
                     const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                     const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                     int dtype, float* scores, int32_t* status_dev, void* stream);

/*
 * dsa_topk_pools - deterministic top-k over each score row.
 *
 * Source: module glm5next_dsa::tp, "Why the indexer is REPLICATED": the tie
 * order is pinned - higher score first, then the smaller pool index - because
 * the order torch.topk gives equal values is undefined.  module glm5next_dsa,
 * "Shape of the pipeline": [Q, select_k] pool ids.
 *
 * Candidates are the entries with score > -inf (NaN is not a candidate); -0
 * and +0 are equal.  pool_ids[q, :] lists the first min(select_k, #candidates)
 * candidates in (score descending, pool index ascending) order; the remaining
 * entries are -1.  The result is unique and bit-reproducible.
 *
 *   scores   [Q, P_ld] fp32;  pool_ids [Q, select_k] int32
 *   workspace: dsa_topk_pools_workspace_size(Q, P_ld, select_k) bytes (currently 0:
 *   the histogram and candidate lists live in shared memory); may be NULL when 0
 * Supported: 1 <= select_k <= DSA_SELECT_K_MAX.
 */
int dsa_topk_pools(const float* scores, int Q, int P_ld, int select_k, int32_t* pool_ids,
                   void* workspace, size_t ws_bytes, void* stream);
size_t dsa_topk_pools_workspace_size(int Q, int P_ld, int select_k);

/*
 * dsa_expand_selection - pool ids to token ids.
 *
 * Source: module glm5next_dsa, "Shape of the pipeline" ([Q, out_width] token
 * ids, -1 = invalid) and "Traps carried from Slice 8": the -1 destination is
 * written in full (an unwritten tail once turned uninitialised memory into
 * token indices).
 *
 *   token_ids[q, j*kpool + s] = pool_start[cap_base(b) + pool_ids[q, j]] + s
 * for a selected pool; -1 when pool_ids[q, j] < 0 or its pool_start is -1;
 * every column >= select_k*kpool is -1.  All Q*out_width entries are written.
 *
 *   pool_ids [Q, select_k]; pool_start, cu_pool_cap as for the cache; q_seq [Q] or NULL
 *   token_ids [Q, out_width] int32, out_width >= select_k * kpool
 * Device faults: DSA_DEV_BAD_POOL_ID (id >= cap_b -> -1), DSA_DEV_BAD_QSEQ.
 */
int dsa_expand_selection(const int32_t* pool_ids, const int32_t* pool_start,
                         const int32_t* cu_pool_cap, const int32_t* q_seq, int Q, int B,
                         int select_k, int kpool, int out_width, int32_t* token_ids,
                         int32_t* status_dev, void* stream);

/*
 * dsa_mla_selected_decode - NoPE MLA decode restricted to the selected rows.
 *
 * Source: module glm5next_dsa, "Shape of the pipeline" (NoPE MLA restricted to
 * the selected tokens), Modules, attend (the selected-index NoPE MLA decode
 * launcher) and "Traps carried from Slice 8" (NoPE: no rotary slice anywhere).
 *
 * For query q (sequence b) and head h, over the selected rows
 * c_j = kv_latent[cu_seqlens[b] + token_ids[q, j]] with token_ids[q, j] >= 0:
 *   z_j = sm_scale * <q_lat[q, h, :], c_j>
 *   out[q, h, :] = sum_j softmax(z)_j * c_j        (absorbed MLA: value = latent row)
 *   lse[q, h]    = log(sum_j exp(z_j))            (natural log)
 * An empty selection gives out = 0 and lse = -inf.
 *
 *   q_lat [Q, Hm, L] activation dtype; kv_latent [sum T_b, L] activation dtype
 *   token_ids [Q, out_width] int32 (from dsa_expand_selection)
 *   out [Q, Hm, L] activation dtype; lse [Q, Hm] fp32 (may be NULL)
 *   workspace: dsa_mla_selected_decode_workspace_size(...) bytes, 16-byte aligned
 * Supported: L multiple of 8 up to 1024 and Hm up to 128 in both dtypes; bf16
 * with L = 512 and Hm a multiple of 16 runs on the tensor cores.
 * Device faults: DSA_DEV_BAD_TOKEN (token id >= T_b: row skipped), DSA_DEV_BAD_QSEQ.
 */
int dsa_mla_selected_decode(const void* q_lat, const void* kv_latent, const int32_t* cu_seqlens,
                            const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int Hm,
                            int L, int out_width, float sm_scale, int dtype, void* out,
                            float* lse, void* workspace, size_t ws_bytes, int32_t* status_dev,
                            void* stream);
size_t dsa_mla_selected_decode_workspace_size(int Q, int Hm, int L, int out_width, int dtype);

/*
 * dsa_mla_paged_decode - the selected-row attention above, reading the latent
 * rows from a paged cache, in bf16 or as 8-bit E4M3 codes.
 *
 * Source: module glm5next_dsa, Modules, attend (the launcher of the
 * selected-index NoPE MLA *paged* decode) and Constants, KERNEL_KV_LORA_DIM
 * (its kernel mla_paged_decode and the _fp8 twin).  The pages give no layout;
 * this one is the plain reading:
 *
 *   pages [n_pages * page_size, L]: page g holds rows g*page_size ..
 *     g*page_size + page_size - 1; 16-byte aligned; kv_dtype DSA_BF16, DSA_F32
 *     or DSA_FP8_E4M3 (E4M3 of the OCP 8-bit floating-point format);
 *   row_scale [n_pages * page_size] fp32 (DSA_FP8_E4M3 only, else NULL): the
 *     value of a row is decode(code) * row_scale[row];
 *   block_table [B, max_pages] int32: token t of sequence b is row
 *     t % page_size of page block_table[b * max_pages + t / page_size];
 *   seq_lens [B] int32: token ids at or past seq_lens[b] are flagged.
 * Every other argument, output and fault is that of dsa_mla_selected_decode.
 * A token whose block is past the table or whose page is outside [0, n_pages)
 * is skipped and flagged DSA_DEV_BAD_PAGE.  The library reads the cache and
 * the table; it owns none of them.
 * Supported: dtype bf16 with kv_dtype bf16 or E4M3, 64 heads and L = 512 on the
 * tensor cores (any number of queries); any geometry of dsa_mla_selected_decode
 * on the generic kernel.
 */
typedef struct dsa_paged_kv {
  const void* pages;
  const float* row_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int n_pages, page_size, max_pages, kv_dtype;
} dsa_paged_kv;
int dsa_mla_paged_decode(const void* q_lat, const dsa_paged_kv* kv, const int32_t* q_seq,
                         const int32_t* token_ids, int Q, int B, int Hm, int L, int out_width,
                         float sm_scale, int dtype, void* out, float* lse, void* workspace,
                         size_t ws_bytes, int32_t* status_dev, void* stream);
size_t dsa_mla_paged_decode_workspace_size(int Q, int Hm, int L, int out_width, int dtype,
                                           int kv_dtype);

/*
 * dsa_select - index_scores -> topk_pools -> expand_selection in one call.
 *
 * Source: module glm5next_dsa, Modules, select (the production launcher of the
 * indexer pipeline) and "Shape of the pipeline".  Writes exactly what the three
 * stage calls above write, in the same buffers (scores [Q, P_ld], pool_ids
 * [Q, select_k], token_ids [Q, out_width]), with the same arguments and device
 * faults, but fuses the expansion into the top-k kernel and, for the decode
 * geometry (bf16, H = 32, D = 128, one query per key tile), the top-k
 * histogram into the scoring kernel.
 *
 *   workspace: dsa_select_workspace_size(Q, P_ld, select_k) bytes, 16-byte
 *   aligned, ZERO-FILLED BEFORE ITS FIRST USE; every call leaves it zeroed, so a
 *   workspace is zeroed once at allocation and then reused.  Two calls in
 *   flight at the same time must not share a workspace.
 */
int dsa_select(const void* q, const float* weights, float scale, const void* pool_keys,
               int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
               const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
               const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
               int select_k, int out_width, int dtype,
               float* scores, int32_t* pool_ids, int32_t* token_ids, void* workspace,
               size_t ws_bytes, int32_t* status_dev, void* stream);
size_t dsa_select_workspace_size(int Q, int P_ld, int select_k);

/*
 * dsa_select_noalloc - dsa_select for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a deployment variant of dsa_select.
 * Callers recording into a CUDA stream capture, plugins whose host framework
 * owns every device allocation, or serving loops that forbid allocation after
 * start-up cannot provide dsa_select's workspace.  This call takes the same
 * arguments minus the workspace and writes the same outputs; its scratch (a
 * 4096-bin histogram per query) lives in a static 1 MiB device array that every
 * GPU loading the library keeps until the process exits.
 *   Q must be <= 64 (else DSA_ERR_UNSUPPORTED).  All calls on a device share the
 *   array: each call clears the part it uses first, and calls that overlap on
 *   the GPU race on it.  The first call on a device (with Q > 0) looks up the
 *   array's device address; make it before any stream capture.  The address
 *   is kept for the life of the process: the device's primary context must not
 *   be reset in between (cudaDeviceReset).  It allocates nothing.
 */
int dsa_select_noalloc(const void* q, const float* weights, float scale, const void* pool_keys,
                       int pool_rows, const int32_t* pool_start, const uint8_t* pool_valid,
                       const int32_t* n_pools, const int32_t* cu_pool_cap, const int32_t* q_seq,
                       const int32_t* q_pos, int Q, int B, int H, int D, int kpool, int P_ld,
                       int select_k, int out_width, int dtype, float* scores, int32_t* pool_ids,
                       int32_t* token_ids, int32_t* status_dev, void* stream);

/*
 * dsa_decode_layer - one layer of the decode path in one call:
 *   dsa_kpool_compress (the pools [pool_begin[b], pool_begin[b] + max_pools))
 *   -> dsa_select -> dsa_mla_selected_decode.
 *
 * Source: module glm5next_dsa, "Shape of the pipeline" (the five stages in
 * order).  The pages have no fused call; this one writes exactly what the three
 * calls above write, with their arguments (gathered in the struct below), their
 * validation (all three stages are checked before anything is launched) and
 * their device faults.  Being one call, its later kernels may start on data
 * that its earlier kernels do not write: the scoring kernel streams the key
 * tiles below pool_begin[b] while the compress still runs (decode geometry,
 * q_pos == NULL), and the attention kernel loads its query block before the
 * token ids exist.  With max_pools == 1 in that geometry (a decode step: one
 * new pool per sequence, bf16, D = 128) the compress runs inside the scoring
 * kernel and the call launches one kernel fewer.  As with every call, inputs
 * are ordered by the stream: work enqueued before the call has finished
 * writing them when it starts.
 *   ws_select: dsa_select_workspace_size(Q, P_ld, select_k) bytes, zero-filled
 *              before first use, left zeroed (as for dsa_select).
 *   ws_mla:    dsa_mla_selected_decode_workspace_size(Q, Hm, L, out_width, dtype).
 *   pool_begin may be NULL (every pool from 0; no early streaming).
 */
typedef struct dsa_decode_layer_args {
  /* kpool_compress inputs */
  const void* k;
  const void* gate;
  const uint8_t* valid;
  const float* ape;
  const void* ln_gamma;
  const void* ln_beta;
  float ln_eps;
  const int32_t* cu_seqlens;
  const int32_t* pool_begin;
  int max_pools;
  /* pool cache (written by the compress, read by the selection) */
  void* pool_keys;
  int pool_rows;
  int32_t* pool_start;
  uint8_t* pool_valid;
  int32_t* n_pools;
  const int32_t* cu_pool_cap;
  /* queries */
  const void* q;
  const float* weights;
  float scale;
  const int32_t* q_seq;
  const int32_t* q_pos;
  const void* q_lat;
  const void* kv_latent;
  float sm_scale;
  /* geometry */
  int Q, B, H, D, kpool, P_ld, select_k, out_width, Hm, L, dtype;
  /* outputs and workspaces */
  float* scores;
  int32_t* pool_ids;
  int32_t* token_ids;
  void* out;
  float* lse;
  void* ws_select;
  size_t ws_select_bytes;
  void* ws_mla;
  size_t ws_mla_bytes;
  int32_t* status_dev;
} dsa_decode_layer_args;
int dsa_decode_layer(const dsa_decode_layer_args* args, void* stream);
/* Workspace sizes for the geometry in *args; returns their sum. */
size_t dsa_decode_layer_workspace_size(const dsa_decode_layer_args* args, size_t* ws_select,
                                       size_t* ws_mla);

/*
 * dsa_indexer_project - the per-token projections that feed the path: the
 * indexer key, its slot logits and head weights from the hidden state, the
 * indexer query and the MLA no-rope query from the query latent, and the
 * latent-space MLA query (module glm5next_dsa, Modules: build and layer, the
 * DSA block's tensors; Traps carried from Slice 8: NoPE, no rotary part).
 * The pages name these tensors but print no formula; the library takes them
 * as plain bias-free linear maps, every output feature f of token t being
 *   out[t, f] = alpha * sum_k W[f, k] * in[t, k]     (fp32 accumulation)
 *
 *   x      [T, hidden]  bf16   hidden states of the T tokens
 *   w_kgw  [2D + H, hidden] bf16  rows 0..D-1 -> k, D..2D-1 -> gate,
 *                              2D..2D+H-1 -> weights (alpha = weights_scale)
 *   cq     [T, q_rank]  bf16   query latent of the T tokens
 *   w_q    [H*D + Hm*nope, q_rank] bf16  rows 0..H*D-1 -> q (head h owns
 *                              rows h*D..h*D+D-1), the rest -> q_nope
 *   w_uk_t [Hm, L, nope] bf16  per MLA head, the key up-projection W_uk_h
 *                              ([nope, L]) stored transposed (a load-time
 *                              re-layout): q_lat[t, h, l] =
 *                              sum_n q_nope[t, h, n] * W_uk_h[n, l], so that
 *                              <q_lat_h, c> = <q_nope_h, W_uk_h c> for a latent
 *                              cache row c.
 * Outputs (bf16 unless stated; every element of every token is written):
 *   k_out, gate_out [rows, D]: token t to row kv_rows[t] (kv_rows NULL: row t;
 *                   a negative entry drops the token), e.g. straight into the
 *                   key and gate caches that dsa_kpool_compress reads
 *   weights_out     [T, H] fp32
 *   q_out           [T, H, D]
 *   q_nope_out      [T, Hm, nope] (also the input of the latent projection)
 *   q_lat_out       [T, Hm, L]
 * Sizes: hidden and q_rank multiples of 8, nope a multiple of 64.
 * Alignment: x, w_kgw, cq, w_q, w_uk_t, q_nope_out and the workspace on 16
 * bytes; bf16 outputs on 2, weights_out, kv_rows and status_dev on 4.
 * Workspace: dsa_indexer_project_workspace_size bytes (0: none needed).  Its
 * first bytes are counters that must be ZERO before the first call that uses
 * the workspace; every call leaves them zero.  Calls that share a workspace
 * must not overlap on the GPU.
 * Outputs are deterministic: a contraction split across CTAs is added in split
 * order whatever order the CTAs finish in.
 * Device faults: DSA_DEV_TIMEOUT (outputs unspecified).
 * Returns DSA_ERR_UNSUPPORTED for sizes outside the above, DSA_ERR_WORKSPACE
 * for a missing or short workspace; T == 0 is a no-op.
 */
int dsa_indexer_project(const void* x, const void* w_kgw, const void* cq, const void* w_q,
                        const void* w_uk_t, int T, int hidden, int q_rank, int H, int D, int Hm,
                        int nope, int L, float weights_scale, const int32_t* kv_rows,
                        void* k_out, void* gate_out, float* weights_out, void* q_out,
                        void* q_nope_out, void* q_lat_out, void* workspace, size_t ws_bytes,
                        int32_t* status_dev, void* stream);
size_t dsa_indexer_project_workspace_size(int T, int hidden, int q_rank, int H, int D, int Hm,
                                          int nope, int L);

/*
 * dsa_set_failure_drill - arm (DSA_DRILL_SKIP_ARM) or disarm (0) a drill of
 * the kernels' give-up path, for tests of failure detection.
 *
 * The pages have no counterpart: the library's waits on its own asynchronous
 * copies and tensor-core MMAs are bounded (1 s of the GPU's global timer), and
 * a wait that runs out sets DSA_DEV_TIMEOUT in *status_dev, issues nothing
 * more, waits (bounded) for what it already issued, frees its tensor memory
 * and returns, so the CUDA context stays usable.  Nothing in a correct run
 * makes such a wait run out.  While the drill is armed, every launch of the
 * tensor-core kernels (index scoring, attention) skips arming the barrier its
 * first wait needs: that wait runs out after 1 ms with no copy or MMA in
 * flight, the kernel takes the give-up path, and the call's outputs are
 * unspecified (status_dev carries DSA_DEV_TIMEOUT).  The setting is process
 * wide and read when a call launches its kernels (a graph captured meanwhile
 * keeps it).  Never arm it in production.  Returns DSA_OK, or
 * DSA_ERR_INVALID_ARG for an unknown drill.
 */
#define DSA_DRILL_SKIP_ARM 1
/* The streaming attention kernel (many queries, or any paged call) issues its
 * MMAs but arms none of the barriers of its PV chunks: those waits run out with
 * MMAs in flight; the kernel issues nothing more, drains them through one more
 * commit, frees its tensor memory and returns (DSA_DEV_TIMEOUT).  The other
 * tensor-core kernels take it as DSA_DRILL_SKIP_ARM. */
#define DSA_DRILL_SKIP_PV_COMMIT 2
int dsa_set_failure_drill(int drill);

/* Human-readable name of a DSA_* return code (static string). */
const char* dsa_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int dsa_version(void);

/* Number of kernels the library has launched, or recorded into a stream
   capture, since it was loaded (every thread and device).  Replays of a
   captured graph launch its kernels without passing through the library and
   are not counted: count the capture, then multiply by the replays. */
uint64_t dsa_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
