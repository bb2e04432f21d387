// NoPE MLA decode over the selected latent rows on the tcgen05 tensor cores.
//
// Module glm5next_dsa, "Shape of the pipeline" (NoPE MLA restricted to the
// selected tokens), Modules, attend, and "Traps carried from Slice 8" (NoPE: the
// score is the plain latent dot product).  In absorbed MLA the value of a latent
// row is the row itself, so one gathered tile feeds both products.
//
// Geometry: bf16, 64 heads, latent 512.  One CTA = one query, one split of 128
// selected rows and one half of the heads (32):
//   1. the query's q_lat half (32 x 512) and the split's 128 latent rows are
//      gathered with 16-byte cp.async into 128-byte-swizzled tiles (eight
//      64-column blocks each; bf16 rows in one cp.async group per block);
//   2. S^T = C q^T on the tensor cores: M = 128 rows, N = 32 heads, K = 512, one
//      thread issues 32 MMAs into TMEM, four per block as each block lands;
//   3. softmax per head over the 128 rows: each thread reads its row's scores
//      of 16 heads, a butterfly over the warp reduces the 16 columns across the
//      warp's 32 rows, four warps combine through shared memory; the
//      probabilities are written to shared memory row-major (P: 128 rows x 32
//      heads, bf16, one 64-byte swizzled line per row, two 16-byte stores per
//      thread, read MN-major by the tensor cores) and the per-head max (base
//      2) and sum are kept;
//   4. O^T = C^T P^T: M = 128 latent columns (four chunks), N = 32 heads, K = 128
//      rows.  A is the same gathered tile read MN-major, so the rows are never
//      transposed;
//   5. O^T is staged in shared memory (the row tile is no longer needed) and the
//      unnormalised partial rows leave with coalesced 16-byte stores, with the
//      per-head max and sum (or, with a single split, the normalised output and
//      lse go straight to the outputs); the merge kernel combines the splits.
// Waits on the MMA completions are bounded (DSA_DEV_TIMEOUT on expiry).
//
// The same kernel reads a paged cache (Modules, attend: the paged decode; a
// block table maps a token to its page) in bf16 or as E4M3 codes with one fp32
// scale per row (Constants, KERNEL_KV_LORA_DIM: the _fp8 twin).  E4M3 codes
// convert exactly to bf16 while they are gathered, so the tensor cores see the
// codes; the row's scale multiplies its logit and its probability in the P^T
// tile, and the softmax sum stays that of the unscaled probabilities:
//   z = s * <q, code row>,  O = sum_r p_r * s_r * code_r / sum_r p_r.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>

#include "dsa_internal.cuh"
#include "umma.cuh"

namespace dsa {
namespace {

constexpr int kL = 512, kHm = 64, kHh = 32, kRows = 128;
constexpr int kThreadsM = 256;
constexpr int kKvBlock = kRows * 128;   // 128 rows x 64 latent columns, 16 KB
constexpr int kQBlock = kHh * 128;      // 32 heads x 64 latent columns, 4 KB
constexpr int kPBytes = kRows * kHh * 2;  // P: 128 rows x 32 heads, bf16, 8 KB
constexpr int kTmemCols = 256;          // S^T (32 columns) + O^T (4 x 32 columns)
constexpr float kLog2e = 1.4426950408889634f;


// Row sources of the kernel.
constexpr int kKvContig = 0;   // bf16 rows at cu_seqlens[b] + tok
constexpr int kKvPaged = 1;    // bf16 rows through the block table
constexpr int kKvPagedE4M3 = 2;  // E4M3 rows through the block table, one fp32 scale per row

struct MCtl {
  float m_fin[kHh], l_fin[kHh];  // first: 16-byte aligned
  uint64_t s_ready, o_ready;
  uint32_t tmem_base;
  int pad;
  int tok[kRows];
  int prow[kRows];   // the row of the cache (-1: none)
  float rs[kRows];   // E4M3: the row's scale
  float red[2][4][16];  // [head quarter pair][row quarter][head]: per-warp partials
};
constexpr size_t kOffKv = 0;
constexpr size_t kOffQ = kOffKv + 8 * (size_t)kKvBlock;
constexpr size_t kOffPt = kOffQ + 8 * (size_t)kQBlock;
constexpr size_t kOffCtl = kOffPt + (size_t)kPBytes;
constexpr size_t kSmemBytes = 1024 + kOffCtl + sizeof(MCtl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert((size_t)kHh * kL * 4 <= 8 * (size_t)kKvBlock, "O staging fits the row tile");
static_assert(kOffCtl % 16 == 0, "m_fin is read as float4");

// Two E4M3 codes (low byte first) -> two bf16 (low half first), exactly: every
// E4M3 value is a half and a bfloat16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  const __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 values per lane (one row, 16 heads) reduced over the warp's 32 rows; lanes
// l and l + 16 end with the reduction of head l.  A plain exchange across the
// two half-warps, then halving steps that keep half of the values and swap the
// other half with the partner lane: 31 shuffles in all.
template <bool kMax>
__device__ __forceinline__ float transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float o = __shfl_xor_sync(0xffffffffu, v[i], 16);
    v[i] = kMax ? fmaxf(v[i], o) : v[i] + o;
  }
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

template <int kKv>
__global__ void __launch_bounds__(kThreadsM, 1)
    mla_umma_kernel(const __nv_bfloat16* __restrict__ q_lat, const __nv_bfloat16* __restrict__ kv,
                    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ q_seq,
                    const int32_t* __restrict__ token_ids, int B, int W, float sm_scale,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                    float* __restrict__ part_o, float* __restrict__ part_ml, int early,
                    PagedKv pk, int drill, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sb = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  MCtl& c = *reinterpret_cast<MCtl*>(sb + kOffCtl);
  const int split = blockIdx.x, n_split = gridDim.x, hf = blockIdx.y, qi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qw = warp & 3;   // TMEM lanes 32 qw .. 32 qw + 31
  const int hq = warp >> 2;  // softmax: heads 16 hq .. 16 hq + 15; epilogue: chunk pair

  if (threadIdx.x == 0) {
    mbar_init(&c.s_ready, 1);
    mbar_init(&c.o_ready, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<kTmemCols>(&c.tmem_base);
    tc_fence_before();
  }
  // Standalone, every input may come from the kernel just before: wait for it
  // first.  Inside a call whose earlier kernels write only the token ids
  // (early), the query block and the sequence lookup go ahead of the wait.
  if (!early) {
    pdl_wait();
    pdl_launch_dependents();
  }

  // ---- 1. gathers: the query block first (no dependency), then the rows
  const long long qh0 = (long long)qi * kHm + hf * kHh;   // first (query, head) row
  const __nv_bfloat16* qsrc = q_lat + qh0 * kL;
  for (int i = threadIdx.x; i < kHh * 64; i += kThreadsM) {
    const int h = i >> 6, ch = i & 63;
    cp_async16(smem_u32(sb + kOffQ + (ch >> 3) * kQBlock + h * 128 + (((ch & 7) ^ (h & 7)) << 4)),
               qsrc + (long long)h * kL + ch * 8, true);
  }
  cp_async_commit();
  const int b = q_seq ? q_seq[qi] : 0;
  const bool seq_ok = b >= 0 && b < B;
  if (!seq_ok && split == 0 && hf == 0 && threadIdx.x == 0) flag(status, DSA_DEV_BAD_QSEQ);
  long long row_base = 0;
  int Tb = 0;
  if (kKv == kKvContig) {
    row_base = seq_ok ? cu_seqlens[b] : 0;
    Tb = seq_ok ? cu_seqlens[b + 1] - cu_seqlens[b] : 0;
  } else {
    Tb = seq_ok ? pk.seq_lens[b] : 0;
  }
  if (early) {
    pdl_wait();  // the token ids of this call
    pdl_launch_dependents();
  }
  if (threadIdx.x < kRows) {
    const int j = split * kRows + threadIdx.x;
    int tok = (j < W && seq_ok) ? token_ids[(long long)qi * W + j] : -1;
    if (tok >= Tb) {
      if (hf == 0) flag(status, DSA_DEV_BAD_TOKEN);
      tok = -1;
    }
    tok = tok < 0 ? -1 : tok;
    long long prow = tok >= 0 ? row_base + tok : -1;
    if (kKv != kKvContig && tok >= 0) {
      const int blk = tok / pk.page_size;
      const int page = blk < pk.max_pages ? pk.block_table[(long long)b * pk.max_pages + blk] : -1;
      if (page < 0 || page >= pk.n_pages) {
        if (hf == 0) flag(status, DSA_DEV_BAD_PAGE);
        tok = -1;
        prow = -1;
      } else {
        prow = (long long)page * pk.page_size + tok % pk.page_size;
      }
    }
    c.tok[threadIdx.x] = tok;
    c.prow[threadIdx.x] = (int)prow;
  }
  __syncthreads();
  const uint32_t kvb = smem_u32(sb + kOffKv), qb = smem_u32(sb + kOffQ);
  const uint32_t ptb = smem_u32(sb + kOffPt);
  constexpr uint32_t idesc_s = umma_idesc_bf16(kRows, kHh, false);
  // a failure drill issues no MMA and arms no barrier: the first wait runs out
  const bool issue = drill == 0;
  const unsigned long long wait_ns = drill ? kDrillWaitNs : kWaitNs;

  // ---- 2. S^T = C q^T  (M = 128 rows, N = 32 heads, K = 512)
  if (kKv != kKvPagedE4M3) {
    // One cp.async group per 64-column block of the rows (after the query
    // block's group).  The four MMAs of a block go out as soon as it has
    // landed, while the later blocks are still in flight.
    const __nv_bfloat16* src =
        kKv == kKvContig ? kv : static_cast<const __nv_bfloat16*>(pk.pages);
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
#pragma unroll
      for (int u = 0; u < kRows * 8 / kThreadsM; ++u) {
        const int i = u * kThreadsM + threadIdx.x;
        const int r = i >> 3, c8 = i & 7;  // eight consecutive threads: one 128-byte row piece
        const int prow = c.prow[r];
        const bool ok = prow >= 0;
        cp_async16(smem_u32(sb + kOffKv + blk * kKvBlock + r * 128 + ((c8 ^ (r & 7)) << 4)),
                   ok ? src + (long long)prow * kL + blk * 64 + c8 * 8 : src, ok);
      }
      cp_async_commit();
    }
#pragma unroll
    for (int blk = 0; blk < 8; ++blk) {
      cp_async_wait_pending(7 - blk);  // the query block and row blocks 0..blk
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (threadIdx.x == 0 && issue) {
        tc_fence_after();
        const uint32_t tm = c.tmem_base;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_bf16(tm, sw128_desc(kvb + blk * kKvBlock + k * 32),
                    sw128_desc(qb + blk * kQBlock + k * 32), idesc_s, (blk | k) ? 1u : 0u);
      }
    }
  } else {
    // 16 codes per 16-byte load, every load of the tile in flight at once; each
    // load becomes two 16-byte bf16 chunks of the swizzled tile
    const uint4* src = static_cast<const uint4*>(pk.pages);
    constexpr int kPer = kRows * (kL / 16) / kThreadsM;  // 16 loads per thread
    uint4 raw[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = u * kThreadsM + threadIdx.x;
      const int prow = c.prow[i >> 5];
      raw[u] = prow >= 0 ? __ldg(src + (long long)prow * (kL / 16) + (i & 31))
                         : make_uint4(0u, 0u, 0u, 0u);
    }
    if (threadIdx.x < kRows) {
      const int prow = c.prow[threadIdx.x];
      c.rs[threadIdx.x] = prow >= 0 ? pk.row_scale[prow] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int i = u * kThreadsM + threadIdx.x;
      const int r = i >> 5, c16 = i & 31;
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int ch = 2 * c16 + half;
        const uint4 v = make_uint4(e4m3x2_to_bf16x2(w[2 * half] & 0xffffu),
                                   e4m3x2_to_bf16x2(w[2 * half] >> 16),
                                   e4m3x2_to_bf16x2(w[2 * half + 1] & 0xffffu),
                                   e4m3x2_to_bf16x2(w[2 * half + 1] >> 16));
        *reinterpret_cast<uint4*>(sb + kOffKv + (ch >> 3) * kKvBlock + r * 128 +
                                  (((ch & 7) ^ (r & 7)) << 4)) = v;
      }
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && issue) {
      tc_fence_after();
      const uint32_t tm = c.tmem_base;
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const uint32_t blk = kk >> 2, off = (kk & 3) * 32;
        umma_bf16(tm, sw128_desc(kvb + blk * kKvBlock + off),
                  sw128_desc(qb + blk * kQBlock + off), idesc_s, kk > 0 ? 1u : 0u);
      }
    }
  }
  if (threadIdx.x == 0 && issue) umma_commit(&c.s_ready);
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const bool s_done = mbar_wait_bounded(&c.s_ready, 0, wait_ns);
  tc_fence_after();

  // ---- 3. softmax over the rows, per head (thread = row r, heads 16 hq .. 16 hq + 15)
  const int r = qw * 32 + lane;
  float z[16];
  tmem_ld16(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(hq * 16), z);
  const bool row_ok = c.tok[r] >= 0;
  const float rs = kKv == kKvPagedE4M3 ? c.rs[r] : 1.f;  // the row's E4M3 scale
  const float zs = kKv == kKvPagedE4M3 ? sm_scale * kLog2e * rs : sm_scale * kLog2e;
#pragma unroll
  for (int i = 0; i < 16; ++i) z[i] = row_ok ? z[i] * zs : -INFINITY;
  {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = z[i];
    const float m = transpose_reduce16<true>(t, lane);
    if (lane < 16) c.red[hq][qw][lane] = m;
  }
  // Every thread takes the same branch from here: the scores exist only if
  // every thread saw them complete.  After a timeout nothing more is issued.
  bool ok = __syncthreads_and(s_done) != 0;
  uint64_t* pending = (!ok && issue) ? &c.s_ready : nullptr;  // issued, completion unseen
  if (ok) {
    if (threadIdx.x < kHh) {
      const int h2 = threadIdx.x >> 4, l2 = threadIdx.x & 15;
      c.m_fin[threadIdx.x] = fmaxf(fmaxf(c.red[h2][0][l2], c.red[h2][1][l2]),
                                   fmaxf(c.red[h2][2][l2], c.red[h2][3][l2]));
    }
    __syncthreads();
    // p = 2^(z - m); a head with no row (m = -inf) has only z = -inf, 2^-inf = 0
    float p[16];
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const float4 m4 = reinterpret_cast<const float4*>(c.m_fin + hq * 16)[q4];
      const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        p[4 * q4 + e] = ex2_fast(z[4 * q4 + e] - (mv[e] == -INFINITY ? 0.f : mv[e]));
    }
    // P row-major: row r's 32 heads in one 64-byte line (64-byte swizzle), read
    // MN-major by the tensor cores; this thread's 16 heads are the 16-byte
    // chunks 2 hq and 2 hq + 1
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float sc = kKv == kKvPagedE4M3 ? rs : 1.f;
      const uint4 w = make_uint4(pack_bf16(p[8 * q] * sc, p[8 * q + 1] * sc),
                                 pack_bf16(p[8 * q + 2] * sc, p[8 * q + 3] * sc),
                                 pack_bf16(p[8 * q + 4] * sc, p[8 * q + 5] * sc),
                                 pack_bf16(p[8 * q + 6] * sc, p[8 * q + 7] * sc));
      *reinterpret_cast<uint4*>(sb + kOffPt + r * 64 + (((2 * hq + q) ^ ((r >> 1) & 3)) << 4)) = w;
    }
    {
      const float l = transpose_reduce16<false>(p, lane);
      if (lane < 16) c.red[hq][qw][lane] = l;
    }
    fence_proxy_async_smem();  // P^T is read by the tensor cores next
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < kHh) {
      const int h2 = threadIdx.x >> 4, l2 = threadIdx.x & 15;
      c.l_fin[threadIdx.x] =
          (c.red[h2][0][l2] + c.red[h2][1][l2]) + (c.red[h2][2][l2] + c.red[h2][3][l2]);
    }

    // ---- 4. O^T = C^T P^T  (M = 128 latent columns x 4 chunks, N = 32 heads, K = 128 rows)
    if (threadIdx.x == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = umma_idesc_bf16(128, kHh, true, true);
#pragma unroll
      for (int mc = 0; mc < 4; ++mc) {
#pragma unroll
        for (int kr = 0; kr < 8; ++kr) {
          const uint64_t a = umma_desc_sw128(kvb + 2 * mc * kKvBlock + kr * 2048, kKvBlock, 1024);
          // 16 rows of P per step; 8-row groups 512 bytes apart; N = 32 is one atom
          const uint64_t bd = umma_desc_sw64(ptb + kr * 1024, kPBytes, 512);
          umma_bf16(tmem + kHh + mc * kHh, a, bd, idesc, kr > 0 ? 1u : 0u);
        }
      }
      umma_commit(&c.o_ready);
    }
    const bool o_done = mbar_wait_bounded(&c.o_ready, 0, wait_ns);
    ok = __syncthreads_and(o_done) != 0;  // (this barrier also publishes l_fin)
    if (!ok) pending = &c.o_ready;
    tc_fence_after();
  }

  if (ok) {
    // ---- 5. epilogue.  Split partials: straight from TMEM (a warp's 32 lanes are
    // 32 consecutive latent columns of one head, so each store is a 128-byte row
    // piece).  A single split: staged through shared memory [head][latent] (the
    // row tile is free now) and normalised into bf16 with 8-byte stores.
    if (n_split > 1) {
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int mc = hq + 2 * cc;
        const int col = mc * 128 + qw * 32 + lane;
        float o[32];
        tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(kHh + mc * kHh), o);
        float* dst = part_o + (qh0 * n_split + split) * kL + col;
#pragma unroll
        for (int i = 0; i < 32; ++i) dst[(long long)i * n_split * kL] = o[i];
      }
      tc_fence_before();
    }
    float* stage = reinterpret_cast<float*>(sb + kOffKv);
    if (n_split == 1) {
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        const int mc = hq + 2 * cc;
        const int col = mc * 128 + qw * 32 + lane;
        float o[32];
        tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(kHh + mc * kHh), o);
#pragma unroll
        for (int i = 0; i < 32; ++i) stage[i * kL + col] = o[i];
      }
      tc_fence_before();
    }
    __syncthreads();
    for (int f = threadIdx.x; n_split == 1 && f < kHh * kL / 4; f += kThreadsM) {
      const int h = f / (kL / 4), c4 = f % (kL / 4);
      const float4 v = *reinterpret_cast<const float4*>(stage + h * kL + c4 * 4);
      const float l = c.l_fin[h];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      *reinterpret_cast<uint2*>(out + (qh0 + h) * kL + c4 * 4) =
          make_uint2(pack_bf16(v.x * inv, v.y * inv), pack_bf16(v.z * inv, v.w * inv));
    }
    if (threadIdx.x < kHh) {
      const int h = threadIdx.x;
      const float m = c.m_fin[h], l = c.l_fin[h];
      if (n_split == 1) {
        if (lse) lse[qh0 + h] = l > 0.f ? (m + log2f(l)) / kLog2e : -INFINITY;
      } else {
        part_ml[((qh0 + h) * n_split + split) * 2] = m;
        part_ml[((qh0 + h) * n_split + split) * 2 + 1] = l;
      }
    }
  } else {
    // Gave up: this CTA's share reads as "nothing selected" (a split with a
    // zero sum is skipped by the merge).
    if (threadIdx.x == 0) flag(status, DSA_DEV_TIMEOUT);
    if (n_split == 1) {
      for (int f = threadIdx.x; f < kHh * kL / 4; f += kThreadsM)
        *reinterpret_cast<uint2*>(out + qh0 * kL + (long long)f * 4) = make_uint2(0u, 0u);
      if (lse && threadIdx.x < kHh) lse[qh0 + threadIdx.x] = -INFINITY;
    } else if (threadIdx.x < kHh) {
      part_ml[((qh0 + threadIdx.x) * n_split + split) * 2] = -INFINITY;
      part_ml[((qh0 + threadIdx.x) * n_split + split) * 2 + 1] = 0.f;
    }
  }
  // TMEM is freed only after every MMA this CTA issued has retired (bounded).
  if (threadIdx.x == 0 && pending != nullptr) mbar_wait_bounded(pending, 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem);
  }
}

// ---- streaming form: many queries ------------------------------------------
// One CTA = one query, all 64 heads, and a range of 128-row tiles taken in
// turn; the output accumulator O^T stays in TMEM across the tiles and the
// softmax is the online one (running max and sum per head).  Each tile:
// gather the rows (the next tile's rows are prefetched into L2 meanwhile),
// S^T = C q^T (M 128 rows, N 64 heads), softmax against the running max,
// O^T += C^T P^T (M 128 latent x 4 chunks, N 64 heads).  The running max is
// raised only when a tile's max exceeds it by more than 8 (base 2): then O^T
// and the sum are rescaled first; otherwise probabilities up to 2^8 are kept,
// which is exact up to rounding since O and the sum share the reference.
//
// The row tile is loaded two column blocks (128 latent columns) at a time, one
// cp.async group each.  O^T += C^T P^T reads exactly those two blocks per latent
// chunk, so each chunk's MMAs commit on their own barrier and, once they have
// completed, the chunk's blocks take the next tile's rows; the next tile's
// S^T MMAs then start on each block pair as it lands.  P is stored row-major
// (64 heads of a row in one 128-byte swizzled line) and read MN-major by the
// tensor cores, so each thread writes its 32 probabilities as four 16-byte
// pieces.
constexpr int kHs = 64;                  // heads per CTA
constexpr int kQBlockS = kHs * 128;      // 64 heads x 64 latent columns, 8 KB
constexpr int kPBytesS = kRows * 128;    // P: 128 rows x 64 heads, bf16, 16 KB
constexpr int kTmemColsS = 512;          // S^T (64) + O^T (4 x 64)
constexpr float kRescaleAt = 8.f;        // base-2 growth of the max that forces a rescale

struct SCtl {
  float m_run[kHs], l_run[kHs], alpha[kHs];  // first: 16-byte aligned
  float red[4][kHs];  // [row quarter][head]: per-warp partials
  float rs[2][kRows];  // row scales (E4M3) of the current and the next tile
  int tok[2][kRows];
  int prow[2][kRows];
  uint64_t s_ready, o_ready[4];
  uint64_t drain;  // give-up path: one commit that tracks every MMA issued
  uint32_t tmem_base;
  int rescale;
  int exceed[2];  // [tile parity]: a score passed its head's reference by the margin
};
constexpr size_t kOffKvS = 0;
constexpr size_t kOffQS = kOffKvS + 8 * (size_t)kKvBlock;
constexpr size_t kOffPtS = kOffQS + 8 * (size_t)kQBlockS;
constexpr size_t kOffCtlS = kOffPtS + (size_t)kPBytesS;
constexpr size_t kSmemBytesS = 1024 + kOffCtlS + sizeof(SCtl);
static_assert(kSmemBytesS <= 227 * 1024, "shared memory budget");
static_assert((size_t)kHs * kL * 4 <= 8 * (size_t)kKvBlock, "O staging fits the row tile");
static_assert(kOffCtlS % 16 == 0, "the control block's float arrays are read as float4");

// 32 values per lane (one row, 32 heads) reduced over the warp's 32 rows; lane l
// ends with the reduction of head l (31 shuffles).
template <bool kMax>
__device__ __forceinline__ float transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? v[i] : v[i + s];
      const float keep = upper ? v[i + s] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// Two fp32 multiplies / adds in one packed instruction (each element rounded as
// the scalar instruction rounds it).
__device__ __forceinline__ void mul2(float& a0, float& a1, float b0, float b1) {
  unsigned long long a, b;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  unsigned long long a, b;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(b));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(a));
}


template <int kKv>
__global__ void __launch_bounds__(kThreadsM, 1)
    mla_stream_kernel(const __nv_bfloat16* __restrict__ q_lat,
                      const __nv_bfloat16* __restrict__ kv, const int32_t* __restrict__ cu_seqlens,
                      const int32_t* __restrict__ q_seq, const int32_t* __restrict__ token_ids,
                      int B, int W, int tiles_per_split, float sm_scale,
                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                      float* __restrict__ part_o, float* __restrict__ part_ml, PagedKv pk,
                      int prefetch, int drill, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sb = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  SCtl& c = *reinterpret_cast<SCtl*>(sb + kOffCtlS);
  const int split = blockIdx.x, n_split = gridDim.x, qi = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qw = warp & 3;   // TMEM lanes 32 qw .. 32 qw + 31
  const int hg = warp >> 2;  // heads 32 hg .. 32 hg + 31
  const int n_tiles = (W + kRows - 1) / kRows;
  const int t_lo = split * tiles_per_split;
  const int t_hi = min(n_tiles, t_lo + tiles_per_split);

  if (threadIdx.x == 0) {
    mbar_init(&c.s_ready, 1);
#pragma unroll
    for (int mc = 0; mc < 4; ++mc) mbar_init(&c.o_ready[mc], 1);
    mbar_init(&c.drain, 1);
    fence_mbar_init();
    c.exceed[0] = c.exceed[1] = 0;
  }
  if (warp == 1) {
    tmem_alloc<kTmemColsS>(&c.tmem_base);
    tc_fence_before();
  }
  if (threadIdx.x < kHs) {
    c.m_run[threadIdx.x] = -INFINITY;
    c.l_run[threadIdx.x] = 0.f;
  }
  pdl_wait();  // every input may come from the kernel just before
  pdl_launch_dependents();

  const long long qh0 = (long long)qi * kHm;  // the query's first (query, head) row
  {
    const __nv_bfloat16* qsrc = q_lat + qh0 * kL;
    for (int i = threadIdx.x; i < kHs * 64; i += kThreadsM) {
      const int h = i >> 6, ch = i & 63;
      cp_async16(
          smem_u32(sb + kOffQS + (ch >> 3) * kQBlockS + h * 128 + (((ch & 7) ^ (h & 7)) << 4)),
          qsrc + (long long)h * kL + ch * 8, true);
    }
    cp_async_commit();
  }
  const int b = q_seq ? q_seq[qi] : 0;
  const bool seq_ok = b >= 0 && b < B;
  if (!seq_ok && split == 0 && threadIdx.x == 0) flag(status, DSA_DEV_BAD_QSEQ);
  long long row_base = 0;
  int Tb = 0;
  if (kKv == kKvContig) {
    row_base = seq_ok ? cu_seqlens[b] : 0;
    Tb = seq_ok ? cu_seqlens[b + 1] - cu_seqlens[b] : 0;
  } else {
    Tb = seq_ok ? pk.seq_lens[b] : 0;
  }
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  const uint32_t kvb = smem_u32(sb + kOffKvS), qb = smem_u32(sb + kOffQS);
  const uint32_t ptb = smem_u32(sb + kOffPtS);
  const int32_t* toks = token_ids + (long long)qi * W;
  const size_t row_bytes = kKv == kKvPagedE4M3 ? (size_t)kL : (size_t)kL * 2;
  const unsigned char* rows_base = static_cast<const unsigned char*>(
      kKv == kKvContig ? static_cast<const void*>(kv) : pk.pages);
  bool ok = true;
  int r = qw * 32 + lane;  // this thread's row of the tile in the softmax
  // Failure drills: DSA_DRILL_SKIP_ARM issues no MMA and arms no barrier (the
  // first wait runs out); DSA_DRILL_SKIP_PV_COMMIT issues every MMA but arms
  // no PV chunk barrier (those waits run out with MMAs in flight).
  const bool issue = drill != DSA_DRILL_SKIP_ARM;
  const bool arm_pv = drill != DSA_DRILL_SKIP_PV_COMMIT;
  const unsigned long long wait_ns = drill ? kDrillWaitNs : kWaitNs;
  bool pv_failed = false;  // this thread's wait on a PV chunk ran out
  float l_part[32];  // row r's softmax sums of heads 32 hg .. (same reference as O^T)
#pragma unroll
  for (int i = 0; i < 32; ++i) l_part[i] = 0.f;

  // token id of row (threadIdx.x mod 128) of tile t, as stored (-1: none)
  auto load_tok = [&](int t) -> int {
    const int j = t * kRows + (threadIdx.x & (kRows - 1));
    return (j < W && seq_ok) ? toks[j] : -1;
  };
  // the cache row of a stored token id (-1: none); flags bad ids and pages
  auto row_of = [&](int tok, int* tok_out) -> int {
    if (tok >= Tb) {
      flag(status, DSA_DEV_BAD_TOKEN);
      tok = -1;
    }
    tok = tok < 0 ? -1 : tok;
    long long prow = tok >= 0 ? row_base + tok : -1;
    if (kKv != kKvContig && tok >= 0) {
      const int blk = tok / pk.page_size;
      const int page = blk < pk.max_pages ? pk.block_table[(long long)b * pk.max_pages + blk] : -1;
      if (page < 0 || page >= pk.n_pages) {
        flag(status, DSA_DEV_BAD_PAGE);
        tok = -1;
        prow = -1;
      } else {
        prow = (long long)page * pk.page_size + tok % pk.page_size;
      }
    }
    *tok_out = tok;
    return (int)prow;
  };
  // a tile's token ids (from load_tok) -> its cache rows in slot `buf` (threads
  // 0..127); with `prefetch`, threads 128..255 bring the same rows into L2
  // (rows that few queries share are cold: measured 58 against 65 us on a
  // 64-sequence decode batch; a prefill chunk's rows, shared by its thousands of
  // queries, mostly sit in L2 already: 1.78 against 1.89 ms without)
  auto tile_ids = [&](int tok_raw, int buf) {
    if (threadIdx.x < kRows) {
      int tok;
      const int prow = row_of(tok_raw, &tok);
      c.tok[buf][threadIdx.x] = tok;
      c.prow[buf][threadIdx.x] = prow;
    } else if (prefetch && tok_raw >= 0 && tok_raw < Tb) {
      long long prow = row_base + tok_raw;
      if (kKv != kKvContig) {
        const int blk = tok_raw / pk.page_size;
        const int page =
            blk < pk.max_pages ? pk.block_table[(long long)b * pk.max_pages + blk] : -1;
        prow = (page >= 0 && page < pk.n_pages)
                   ? (long long)page * pk.page_size + tok_raw % pk.page_size
                   : -1;
      }
      if (prow >= 0) {
        const unsigned char* p = rows_base + (size_t)prow * row_bytes;
        for (size_t o = 0; o < row_bytes; o += 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
      }
    }
  };
  // bf16 rows: this thread copies sixteen bytes of rows (tid / 16) + 16 k,
  // k = 0..7, in every block pair; their cache rows are read once per tile
  int my_rows[8];
  auto load_my_rows = [&](int buf) {
#pragma unroll
    for (int k = 0; k < 8; ++k) my_rows[k] = c.prow[buf][(threadIdx.x >> 4) + 16 * k];
  };
  // E4M3 rows: a tile's codes, all sixteen 16-byte loads per thread, go to
  // registers ahead of the blocks being free (rows (i / 8), i = u * 256 + tid,
  // codes 16 (8 j + i mod 8) .. of block pair j), with the rows' scales
  constexpr int kE4Per = kRows * 8 / kThreadsM;
  uint4 e_raw[kKv == kKvPagedE4M3 ? 4 : 1][kE4Per];
  auto e4m3_load = [&](int buf) {
    if (kKv == kKvPagedE4M3) {
      const uint4* src = reinterpret_cast<const uint4*>(rows_base);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int u = 0; u < kE4Per; ++u) {
          const int i = u * kThreadsM + threadIdx.x;
          const int prow = c.prow[buf][i >> 3];
          e_raw[j][u] = prow >= 0 ? __ldg(src + (long long)prow * (kL / 16) + 8 * j + (i & 7))
                                  : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // the scales by threads 128..255: thread 0 issues the MMAs and must not
      // wait for a load here
      if (threadIdx.x >= kRows) {
        const int rr = threadIdx.x - kRows;
        const int prow = c.prow[buf][rr];
        c.rs[buf][rr] = prow >= 0 ? pk.row_scale[prow] : 0.f;
      }
    }
  };
  // column blocks 2j and 2j + 1 (latent 128 j .. 128 j + 127) of the tile whose
  // cache rows are in slot `buf` (bf16: in my_rows; E4M3: codes in e_raw), as
  // one cp.async group
  auto gather_pair = [&](int buf, int j) {
    if (kKv != kKvPagedE4M3) {
      const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(rows_base);
      const int ch = 16 * j + (threadIdx.x & 15);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int rr = (threadIdx.x >> 4) + 16 * k;
        const int prow = my_rows[k];
        const bool okr = prow >= 0;
        cp_async16(smem_u32(sb + kOffKvS + (ch >> 3) * kKvBlock + rr * 128 +
                            (((ch & 7) ^ (rr & 7)) << 4)),
                   okr ? src + (long long)prow * kL + ch * 8 : src, okr);
      }
    } else {
      // the codes were loaded into e_raw by e4m3_load; convert and store
#pragma unroll
      for (int u = 0; u < kE4Per; ++u) {
        const int i = u * kThreadsM + threadIdx.x;
        const int rr = i >> 3, c16 = 8 * j + (i & 7);
        const uint32_t w[4] = {e_raw[j][u].x, e_raw[j][u].y, e_raw[j][u].z, e_raw[j][u].w};
#pragma unroll
        for (int hf2 = 0; hf2 < 2; ++hf2) {
          const int ch = 2 * c16 + hf2;
          const uint4 v = make_uint4(e4m3x2_to_bf16x2(w[2 * hf2] & 0xffffu),
                                     e4m3x2_to_bf16x2(w[2 * hf2] >> 16),
                                     e4m3x2_to_bf16x2(w[2 * hf2 + 1] & 0xffffu),
                                     e4m3x2_to_bf16x2(w[2 * hf2 + 1] >> 16));
          *reinterpret_cast<uint4*>(sb + kOffKvS + (ch >> 3) * kKvBlock + rr * 128 +
                                    (((ch & 7) ^ (rr & 7)) << 4)) = v;
        }
      }
    }
    cp_async_commit();
  };

  if (t_lo < t_hi) {
    tile_ids(load_tok(t_lo), 0);
    __syncthreads();
    if (kKv != kKvPagedE4M3) load_my_rows(0);
    e4m3_load(0);
#pragma unroll
    for (int j = 0; j < 4; ++j) gather_pair(0, j);
  }
  for (int t = t_lo; t < t_hi; ++t) {
    const int cur = (t - t_lo) & 1;
    const uint32_t ph = (uint32_t)cur;
    const int tok_next = t + 1 < t_hi ? load_tok(t + 1) : -1;  // in flight during step 1
    // ---- 1. S^T = C q^T  (M = 128 rows, N = 64 heads, K = 512), two column
    // blocks at a time as their rows land
    bool go = true;  // no thread gave up on a PV chunk (the tile's first barrier says)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      cp_async_wait_pending(3 - j);  // the query's group is older than every row group
      fence_proxy_async_smem();
      tc_fence_before();
      if (j == 0)
        go = __syncthreads_or(pv_failed) == 0;
      else
        __syncthreads();
      tc_fence_after();
      if (threadIdx.x == 0 && issue) {
        // after a thread gave up on a PV chunk no MMA is issued; the commit
        // still comes, and completes once the MMAs already issued have drained
        if (go) {
          constexpr uint32_t idesc = umma_idesc_bf16(kRows, kHs, false);
#pragma unroll
          for (int kk = 8 * j; kk < 8 * j + 8; ++kk) {
            const uint32_t blk = kk >> 2, off = (kk & 3) * 32;
            umma_bf16(tmem, sw128_desc(kvb + blk * kKvBlock + off),
                      sw128_desc(qb + blk * kQBlockS + off), idesc, kk > 0 ? 1u : 0u);
          }
        }
        if (j == 3) umma_commit(&c.s_ready);
      }
    }
    // the next tile's ids meanwhile (slot cur ^ 1 is free: its tile is done)
    if (t + 1 < t_hi) tile_ids(tok_next, cur ^ 1);
    const bool s_done = mbar_wait_bounded(&c.s_ready, ph, wait_ns);
    tc_fence_after();

    // ---- 2. softmax against the running reference (thread = row r, heads 32 hg ..)
    float z[32];
    tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(hg * 32), z);
    const bool row_ok = c.tok[cur][r] >= 0;
    const float rsr = kKv == kKvPagedE4M3 ? c.rs[cur][r] : 1.f;
    const float zs = kKv == kKvPagedE4M3 ? sm_scale * kLog2e * rsr : sm_scale * kLog2e;
#pragma unroll
    for (int i = 0; i < 32; i += 2) mul2(z[i], z[i + 1], zs, zs);
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = row_ok ? z[i] : -INFINITY;
    // The tile's max per head is needed only where a score passes the head's
    // reference by more than the margin (always on a head's first valid row:
    // the reference starts at -inf); a flag per tile says whether any did.
    float mv[32];
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      const float4 m4 = reinterpret_cast<const float4*>(c.m_run + hg * 32)[q4];
      mv[4 * q4] = m4.x;
      mv[4 * q4 + 1] = m4.y;
      mv[4 * q4 + 2] = m4.z;
      mv[4 * q4 + 3] = m4.w;
    }
    bool exceed = false;
#pragma unroll
    for (int i = 0; i < 32; ++i) exceed |= z[i] > mv[i] + kRescaleAt;
    if (exceed) c.exceed[cur] = 1;
    if (threadIdx.x == 0) c.exceed[cur ^ 1] = 0;  // read last in the previous tile
    // Every thread takes the same branch: the scores exist only if every thread
    // saw them complete.  After a timeout nothing more is issued.
    ok = __syncthreads_and(s_done) != 0 && go;
    if (!ok) break;
    const bool full = c.exceed[cur] != 0;
    bool rescale = false;
    if (full) {
      {
        float tt[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) tt[i] = z[i];
        c.red[qw][hg * 32 + lane] = transpose_reduce32<true>(tt, lane);
      }
      if (threadIdx.x == 0) c.rescale = 0;
      __syncthreads();
      if (threadIdx.x < kHs) {
        const int h = threadIdx.x;
        const float tmax =
            fmaxf(fmaxf(c.red[0][h], c.red[1][h]), fmaxf(c.red[2][h], c.red[3][h]));
        const float m_old = c.m_run[h];
        float m_new = m_old, alpha = 1.f;
        if (m_old == -INFINITY) {
          m_new = tmax;  // first rows of this head: nothing accumulated yet
        } else if (tmax > m_old + kRescaleAt) {
          m_new = tmax;
          alpha = exp2f(m_old - m_new);
          c.rescale = 1;
        }
        c.m_run[h] = m_new;
        c.alpha[h] = alpha;
      }
      __syncthreads();
      rescale = c.rescale != 0;
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const float4 m4 = reinterpret_cast<const float4*>(c.m_run + hg * 32)[q4];
        mv[4 * q4] = m4.x;
        mv[4 * q4 + 1] = m4.y;
        mv[4 * q4 + 2] = m4.z;
        mv[4 * q4 + 3] = m4.w;
      }
    }
    // p = 2^(z - m); a head with no row so far (m = -inf) has only z = -inf
    // here, and 2^-inf = 0
    float p[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) p[i] = ex2_fast(z[i] - (mv[i] == -INFINITY ? 0.f : mv[i]));
    // row r of P: heads 32 hg .. 32 hg + 31 are the 16-byte chunks 4 hg .. 4 hg + 3
    // of its 128-byte line, at the swizzled position chunk ^ (r & 7)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float sc = kKv == kKvPagedE4M3 ? rsr : 1.f;
      const uint4 w = make_uint4(pack_bf16(p[8 * q] * sc, p[8 * q + 1] * sc),
                                 pack_bf16(p[8 * q + 2] * sc, p[8 * q + 3] * sc),
                                 pack_bf16(p[8 * q + 4] * sc, p[8 * q + 5] * sc),
                                 pack_bf16(p[8 * q + 6] * sc, p[8 * q + 7] * sc));
      *reinterpret_cast<uint4*>(sb + kOffPtS + r * 128 + (((hg * 4 + q) ^ (r & 7)) << 4)) = w;
    }
    // this row's running sums per head (reduced over the rows at the end), and
    // on a raised reference what O^T holds so far, rescaled first
    if (rescale) {
#pragma unroll
      for (int i = 0; i < 32; ++i) l_part[i] = l_part[i] * c.alpha[hg * 32 + i] + p[i];
      if (t > t_lo) {
#pragma unroll 1
        for (int mc = 0; mc < 4; ++mc) {
          float o[32];
          const uint32_t ta =
              tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(kHs + mc * kHs + hg * 32);
          tmem_ld32(ta, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= c.alpha[hg * 32 + i];
          tmem_st32(ta, o);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; i += 2) add2(l_part[i], l_part[i + 1], p[i], p[i + 1]);
    }
    fence_proxy_async_smem();  // P is read by the tensor cores next
    tc_fence_before();
    __syncthreads();

    // ---- 3. O^T += C^T P^T  (M = 128 latent x 4 chunks, N = 64 heads, K = 128
    // rows); chunk mc reads column blocks 2 mc and 2 mc + 1 and commits alone.
    // The issuing thread stays one chunk ahead: it would otherwise wait for
    // room in the tensor pipe's queue while every thread waits for it.
    auto issue_pv = [&](int mc) {
      if (threadIdx.x == 0) {
        constexpr uint32_t idesc = umma_idesc_bf16(128, kHs, true, true);
#pragma unroll
        for (int kr = 0; kr < 8; ++kr) {
          const uint64_t a = umma_desc_sw128(kvb + 2 * mc * kKvBlock + kr * 2048, kKvBlock, 1024);
          const uint64_t bd = umma_desc_sw128(ptb + kr * 2048, kPBytesS, 1024);
          umma_bf16(tmem + kHs + mc * kHs, a, bd, idesc, (t > t_lo || kr > 0) ? 1u : 0u);
        }
        if (arm_pv) umma_commit(&c.o_ready[mc]);
      }
    };
    if (threadIdx.x == 0) tc_fence_after();
    issue_pv(0);
    if (t + 1 < t_hi) {
      if (kKv != kKvPagedE4M3)
        load_my_rows(cur ^ 1);
      else
        e4m3_load(cur ^ 1);  // the loads fly while the PV chunks run
    }
    // As each chunk completes, its two column blocks take the next tile's rows.
    // Every thread waits for the chunk itself (no block barrier: the issuing
    // thread may still be queueing the next chunk).  A thread that gives up
    // skips its copies and says so at the next block barrier (the next tile's
    // first one, or the end of the loop).
#pragma unroll
    for (int mc = 0; mc < 4; ++mc) {
      if (mc + 1 < 4) issue_pv(mc + 1);
      const bool o_done = mbar_wait_bounded(&c.o_ready[mc], ph, wait_ns);
      tc_fence_after();
      if (!o_done) pv_failed = true;
      if (o_done && t + 1 < t_hi) gather_pair(cur ^ 1, mc);
    }
  }
  // the last tile's chunks: each thread waited for them; all must have landed
  ok = __syncthreads_and(ok && !pv_failed) != 0;
  cp_async_wait<0>();  // no copy into shared memory is left in flight

  // ---- 5. epilogue: the sums over the rows, O^T -> shared [head][latent] fp32,
  // then whole rows out
  if (ok) {
    c.red[qw][hg * 32 + lane] = transpose_reduce32<false>(l_part, lane);
    __syncthreads();
    if (threadIdx.x < kHs) {
      const int h = threadIdx.x;
      c.l_run[h] = (c.red[0][h] + c.red[1][h]) + (c.red[2][h] + c.red[3][h]);
    }
    float* stage = reinterpret_cast<float*>(sb + kOffKvS);
    const bool any = t_hi > t_lo;
#pragma unroll 1
    for (int mc = 0; mc < 4; ++mc) {
      float o[32];
      tmem_ld32(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)(kHs + mc * kHs + hg * 32), o);
      const int col = mc * 128 + qw * 32 + lane;
#pragma unroll
      for (int i = 0; i < 32; ++i) stage[(hg * 32 + i) * kL + col] = any ? o[i] : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    for (int f = threadIdx.x; f < kHs * kL / 4; f += kThreadsM) {
      const int h = f / (kL / 4), c4 = f % (kL / 4);
      const float4 v = *reinterpret_cast<const float4*>(stage + h * kL + c4 * 4);
      if (n_split == 1) {
        const float l = c.l_run[h];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        *reinterpret_cast<uint2*>(out + (qh0 + h) * kL + c4 * 4) =
            make_uint2(pack_bf16(v.x * inv, v.y * inv), pack_bf16(v.z * inv, v.w * inv));
      } else {
        *reinterpret_cast<float4*>(part_o + ((qh0 + h) * n_split + split) * kL + c4 * 4) = v;
      }
    }
    if (threadIdx.x < kHs) {
      const int h = threadIdx.x;
      const float m = c.m_run[h], l = any ? c.l_run[h] : 0.f;
      if (n_split == 1) {
        if (lse) lse[qh0 + h] = l > 0.f ? (m + log2f(l)) / kLog2e : -INFINITY;
      } else {
        part_ml[((qh0 + h) * n_split + split) * 2] = m;
        part_ml[((qh0 + h) * n_split + split) * 2 + 1] = l;
      }
    }
  } else {
    // Gave up: this CTA's share reads as "nothing selected" (a split with a
    // zero sum is skipped by the merge).
    if (threadIdx.x == 0) flag(status, DSA_DEV_TIMEOUT);
    if (n_split == 1) {
      for (int f = threadIdx.x; f < kHs * kL / 4; f += kThreadsM)
        *reinterpret_cast<uint2*>(out + qh0 * kL + (long long)f * 4) = make_uint2(0u, 0u);
      if (lse && threadIdx.x < kHs) lse[qh0 + threadIdx.x] = -INFINITY;
    } else if (threadIdx.x < kHs) {
      part_ml[((qh0 + threadIdx.x) * n_split + split) * 2] = -INFINITY;
      part_ml[((qh0 + threadIdx.x) * n_split + split) * 2 + 1] = 0.f;
    }
  }
  // TMEM is freed only after every MMA this CTA issued has retired: after a
  // give-up, one more commit tracks all of them (bounded wait).
  if (!ok && issue && threadIdx.x == 0) {
    umma_commit(&c.drain);
    mbar_wait_bounded(&c.drain, 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kTmemColsS>(tmem);
  }
}

}  // namespace

int mla_umma_splits(int out_width) { return (out_width + kRows - 1) / kRows; }
// Few queries (decode): one CTA per 128 selected rows and 32 heads, at most
// four waves of CTAs; many queries keep the 16-head-group kernel, whose splits
// adapt to Q.
bool mla_umma_ok(int Q, int Hm, int L, int out_width, int dtype) {
  return mla_umma_shape_ok(Hm, L, dtype) &&
         (long long)Q * mla_umma_splits(out_width) * (kHm / kHh) <= 4LL * num_sms();
}
bool mla_umma_shape_ok(int Hm, int L, int dtype) {
  return dtype == DSA_BF16 && Hm == kHm && L == kL;
}

namespace {
template <int kKv>
int launch_kind(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int out_width,
                float sm_scale, void* out, float* lse, float* part_o, float* part_ml, bool early,
                const PagedKv& pk, int32_t* status_dev, cudaStream_t stream) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(mla_umma_kernel<kKv>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kSmemBytes);
  });
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(mla_umma_splits(out_width), kHm / kHh, Q);
  cfg.blockDim = dim3(kThreadsM, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return launch_kernel(&cfg, mla_umma_kernel<kKv>, (const __nv_bfloat16*)q_lat,
                       (const __nv_bfloat16*)kv, cu_seqlens, q_seq, token_ids, B, out_width,
                       sm_scale, (__nv_bfloat16*)out, lse, part_o, part_ml, early ? 1 : 0,
                       pk, failure_drill(), status_dev) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}
}  // namespace

int mla_stream_splits(int Q, int out_width) {
  const int n_tiles = (out_width + kRows - 1) / kRows;
  const int sms = num_sms();
  int s = Q >= sms ? 1 : sms / Q;  // CTAs within one wave
  s = s < 1 ? 1 : (s > n_tiles ? n_tiles : s);
  const int per = (n_tiles + s - 1) / s;
  return (n_tiles + per - 1) / per;
}

namespace {
template <int kKv>
int launch_stream_kind(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                       const int32_t* q_seq, const int32_t* token_ids, int Q, int B,
                       int out_width, float sm_scale, void* out, float* lse, float* part_o,
                       float* part_ml, const PagedKv& pk, int32_t* status_dev,
                       cudaStream_t stream) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(mla_stream_kernel<kKv>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)kSmemBytesS);
  });
  const int n_tiles = (out_width + kRows - 1) / kRows;
  const int n_split = mla_stream_splits(Q, out_width);
  const int per = (n_tiles + n_split - 1) / n_split;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_split, 1, Q);
  cfg.blockDim = dim3(kThreadsM, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytesS;
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  // prefetch the rows into L2 unless many queries share each sequence's rows
  const int prefetch = (long long)Q < 4LL * B ? 1 : 0;
  return launch_kernel(&cfg, mla_stream_kernel<kKv>, (const __nv_bfloat16*)q_lat,
                       (const __nv_bfloat16*)kv, cu_seqlens, q_seq, token_ids, B, out_width,
                       per, sm_scale, (__nv_bfloat16*)out, lse, part_o, part_ml, pk, prefetch,
                       failure_drill(), status_dev) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}
}  // namespace

int launch_mla_stream(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                      const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int out_width,
                      float sm_scale, void* out, float* lse, float* part_o, float* part_ml,
                      int32_t* status_dev, cudaStream_t stream, const PagedKv* paged) {
  if (!paged)
    return launch_stream_kind<kKvContig>(q_lat, kv, cu_seqlens, q_seq, token_ids, Q, B,
                                         out_width, sm_scale, out, lse, part_o, part_ml,
                                         PagedKv{}, status_dev, stream);
  if (paged->kv_dtype == DSA_FP8_E4M3)
    return launch_stream_kind<kKvPagedE4M3>(q_lat, nullptr, nullptr, q_seq, token_ids, Q, B,
                                            out_width, sm_scale, out, lse, part_o, part_ml,
                                            *paged, status_dev, stream);
  return launch_stream_kind<kKvPaged>(q_lat, nullptr, nullptr, q_seq, token_ids, Q, B,
                                      out_width, sm_scale, out, lse, part_o, part_ml, *paged,
                                      status_dev, stream);
}

int launch_mla_umma(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                    const int32_t* q_seq, const int32_t* token_ids, int Q, int B, int out_width,
                    float sm_scale, void* out, float* lse, float* part_o, float* part_ml,
                    bool early, int32_t* status_dev, cudaStream_t stream, const PagedKv* paged) {
  if (!paged)
    return launch_kind<kKvContig>(q_lat, kv, cu_seqlens, q_seq, token_ids, Q, B, out_width,
                                  sm_scale, out, lse, part_o, part_ml, early, PagedKv{},
                                  status_dev, stream);
  if (paged->kv_dtype == DSA_FP8_E4M3)
    return launch_kind<kKvPagedE4M3>(q_lat, nullptr, nullptr, q_seq, token_ids, Q, B, out_width,
                                     sm_scale, out, lse, part_o, part_ml, early, *paged,
                                     status_dev, stream);
  return launch_kind<kKvPaged>(q_lat, nullptr, nullptr, q_seq, token_ids, Q, B, out_width,
                               sm_scale, out, lse, part_o, part_ml, early, *paged, status_dev,
                               stream);
}

}  // namespace dsa
