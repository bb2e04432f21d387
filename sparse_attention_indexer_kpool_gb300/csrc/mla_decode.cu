// NoPE MLA decode restricted to the selected latent-KV rows.
//
// Module glm5next_dsa, "Shape of the pipeline" (NoPE MLA restricted to the
// selected tokens), Modules, attend (selected-index NoPE MLA decode) and "Traps
// carried from Slice 8" (NoPE: the rotary slice is empty, so a score is the
// plain latent dot product).  The value of an absorbed-MLA latent row is the
// row itself, so one gathered row feeds both the score and the output.
//
// Tensor-core kernel (bf16, L = 512, Hm % 16 == 0): one CTA = one query, one
// group of 16 heads and one split of the selected rows; splits are sized so the
// CTAs cover the SMs once.  Eight warps: warp w owns latent quarter w % 4 and
// row half w / 4 of each 64-row tile.  Scores: each warp contracts its latent
// quarter for its 32 rows (partial 16 x 32 tiles summed through shared
// memory).  Output: each warp accumulates its latent quarter over its 32 rows
// (64 fp32 accumulators per thread); the two row halves are added at the end.
// Selected rows are gathered 64 at a time with 16-byte cp.async into a
// double-buffered, XOR-swizzled shared ring (conflict-free ldmatrix), and the
// softmax is the usual online (running max / running sum) form in base 2.
// With more than one split, each CTA writes its unnormalised partial and its
// (max, sum) to the workspace and a small merge kernel combines them.
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "dsa_internal.cuh"

namespace dsa {
namespace {

constexpr int kL = 512;
constexpr int kHG = 16;            // heads per CTA
constexpr int kNT = 64;            // rows per tile
constexpr int kRing = 2;           // gather stages
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunks = kL / 8;    // 16-byte chunks per latent row
constexpr int kPStride = kNT + 8;  // bf16 per sP row (padded)
constexpr int kMaxRows = 8192;     // rows per split held in shared memory
constexpr float kLog2e = 1.4426950408889634f;

struct MlaSmem {
  union {
    __nv_bfloat16 kv[kRing][kNT * kL];   // swizzled gather ring
    float ohalf[4][kHG][128];            // row-half-1 partial outputs (after the loop)
  };
  __nv_bfloat16 q[kHG * kL];             // swizzled
  float s_part[4][kHG][kNT];
  __nv_bfloat16 p[kHG * kPStride];
  float m[kHG], l[kHG], alpha[kHG];
  // followed by int s_tok[rows_per_split rounded up to a tile]
};

__device__ __forceinline__ int swz(int row, int chunk) {  // element offset of a 16B chunk
  return row * kL + ((chunk ^ (row & 7)) << 3);
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_mma_kernel(const __nv_bfloat16* __restrict__ q_lat, const __nv_bfloat16* __restrict__ kv,
                   const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ q_seq,
                   const int32_t* __restrict__ token_ids, int B, int Hm, int W, int rows_per_split,
                   float sm_scale, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                   float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* status) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  MlaSmem& sm = *reinterpret_cast<MlaSmem*>(smem_raw);
  int* s_tok = reinterpret_cast<int*>(smem_raw + sizeof(MlaSmem));
  const int qi = blockIdx.z, hg = blockIdx.y, split = blockIdx.x, n_split = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int g = lane >> 2, t = lane & 3;

  if (threadIdx.x < kHG) {
    sm.m[threadIdx.x] = -INFINITY;
    sm.l[threadIdx.x] = 0.f;
  }
  // every input may come from the kernel just before: wait for it first
  pdl_wait();
  pdl_launch_dependents();  // the merge kernel may start its prologue
  const __nv_bfloat16* qsrc = q_lat + ((long long)qi * Hm + hg * kHG) * kL;
  for (int c = threadIdx.x; c < kHG * kChunks; c += kThreads) {
    const int r = c / kChunks, ch = c % kChunks;
    cp_async16(smem_u32(&sm.q[swz(r, ch)]), qsrc + (long long)r * kL + ch * 8, true);
  }
  const int j_lo = min(W, split * rows_per_split);
  const int j_hi = min(W, j_lo + rows_per_split);
  const int n_tiles = (j_hi - j_lo + kNT - 1) / kNT;
  const int32_t* toks = token_ids + (long long)qi * W;
  // token ids first: their loads do not wait for the sequence lookup
  constexpr int kTokPer = 8;  // covers rows_per_split <= kThreads * kTokPer in one pass
  int tk[kTokPer];
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) {
    const int j = j_lo + u * kThreads + threadIdx.x;
    tk[u] = j < j_hi ? toks[j] : -1;
  }
  const int b = q_seq ? q_seq[qi] : 0;
  const bool seq_ok = b >= 0 && b < B;
  if (!seq_ok && split == 0 && hg == 0 && threadIdx.x == 0) flag(status, DSA_DEV_BAD_QSEQ);
  const long long row_base = seq_ok ? cu_seqlens[b] : 0;
  const int Tb = seq_ok ? cu_seqlens[b + 1] - cu_seqlens[b] : 0;
  // validated token ids of this split (-1 = not a row), padded to whole tiles
  for (int j0 = 0; j0 < n_tiles * kNT; j0 += kThreads * kTokPer) {
#pragma unroll
    for (int u = 0; u < kTokPer; ++u) {
      const int jj = j0 + u * kThreads + threadIdx.x;
      if (jj >= n_tiles * kNT) continue;
      int tok = (j0 == 0) ? tk[u] : (j_lo + jj < j_hi ? toks[j_lo + jj] : -1);
      if (!seq_ok) tok = -1;
      if (tok >= Tb) {
        if (hg == 0) flag(status, DSA_DEV_BAD_TOKEN);
        tok = -1;
      }
      if (tok < 0) tok = -1;
      s_tok[jj] = tok;
    }
  }
  __syncthreads();

  auto load_tile = [&](int tile) {
    const int buf = tile % kRing;
    const int* tt = s_tok + tile * kNT;
    for (int c = threadIdx.x; c < kNT * kChunks; c += kThreads) {
      const int r = c / kChunks, ch = c % kChunks;
      const int tok = tt[r];
      const bool ok = tok >= 0;
      const __nv_bfloat16* src = kv + (row_base + (ok ? tok : 0)) * kL + ch * 8;
      cp_async16(smem_u32(&sm.kv[buf][swz(r, ch)]), ok ? src : kv, ok);
    }
  };
  if (n_tiles > 0) load_tile(0);
  cp_async_commit();

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  uint32_t qf[8][4];
  const float zscale = sm_scale * kLog2e;

  for (int tile = 0; tile < n_tiles; ++tile) {
    const int buf = tile % kRing;
    if (tile + 1 < n_tiles) load_tile(tile + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (tile == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int ch = quarter * 16 + kk * 2 + (lane >> 4);
        ldmatrix_x4(qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3],
                    smem_u32(&sm.q[swz(lane & 15, ch)]));
      }
    }
    // ---- partial scores: this warp's latent quarter x its 32 rows
    const __nv_bfloat16* kvb = sm.kv[buf];
    float sacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t b0, b1, b2, b3;
        const int ch = quarter * 16 + kk * 2 + (lane >> 3);
        ldmatrix_x4(b0, b1, b2, b3, smem_u32(&kvb[swz(half * 32 + nt * 8 + (lane & 7), ch)]));
        mma_bf16_16816(sacc[nt], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16_16816(sacc[nt], qf[kk + 1][0], qf[kk + 1][1], qf[kk + 1][2], qf[kk + 1][3], b2,
                       b3);
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = half * 32 + nt * 8 + 2 * t;
      *reinterpret_cast<float2*>(&sm.s_part[quarter][g][c]) = make_float2(sacc[nt][0], sacc[nt][1]);
      *reinterpret_cast<float2*>(&sm.s_part[quarter][g + 8][c]) =
          make_float2(sacc[nt][2], sacc[nt][3]);
    }
    __syncthreads();
    // ---- online softmax: thread -> head h = tid/16, columns 4*(tid%16) .. +3
    {
      const int h = threadIdx.x >> 4, c0 = (threadIdx.x & 15) * 4;
      float sv[4];
      float mx = -INFINITY;
      const float4 p0 = *reinterpret_cast<const float4*>(&sm.s_part[0][h][c0]);
      const float4 p1 = *reinterpret_cast<const float4*>(&sm.s_part[1][h][c0]);
      const float4 p2 = *reinterpret_cast<const float4*>(&sm.s_part[2][h][c0]);
      const float4 p3 = *reinterpret_cast<const float4*>(&sm.s_part[3][h][c0]);
      const float ssum[4] = {p0.x + p1.x + p2.x + p3.x, p0.y + p1.y + p2.y + p3.y,
                             p0.z + p1.z + p2.z + p3.z, p0.w + p1.w + p2.w + p3.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v = s_tok[tile * kNT + c0 + i] >= 0 ? ssum[i] * zscale : -INFINITY;
        sv[i] = v;
        mx = fmaxf(mx, v);
      }
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      const float m_old = sm.m[h];
      const float m_new = fmaxf(m_old, mx);
      const bool none = m_new == -INFINITY;
      const float alpha = none ? 1.f : exp2f(m_old - m_new);
      float ps = 0.f;
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pv[i] = none ? 0.f : exp2f(sv[i] - m_new);
        ps += pv[i];
      }
#pragma unroll
      for (int o2 = 1; o2 < 16; o2 <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
      *reinterpret_cast<uint2*>(&sm.p[h * kPStride + c0]) =
          make_uint2(pack_bf16(pv[0], pv[1]), pack_bf16(pv[2], pv[3]));
      __syncwarp();
      if ((threadIdx.x & 15) == 0) {
        sm.m[h] = m_new;
        sm.l[h] = sm.l[h] * alpha + ps;
        sm.alpha[h] = alpha;
      }
    }
    __syncthreads();
    // ---- O = O * alpha + P V: latent quarter, this warp's 32 rows
    const float a_lo = sm.alpha[g], a_hi = sm.alpha[g + 8];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      o[nt][0] *= a_lo; o[nt][1] *= a_lo; o[nt][2] *= a_hi; o[nt][3] *= a_hi;
    }
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const int rbase = half * 32 + kk * 16;
      uint32_t a0, a1, a2, a3;
      ldmatrix_x4(a0, a1, a2, a3,
                  smem_u32(&sm.p[(lane & 15) * kPStride + rbase + (lane >> 4) * 8]));
#pragma unroll
      for (int nt = 0; nt < 16; nt += 2) {
        uint32_t b0, b1, b2, b3;
        const int r = rbase + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ch = quarter * 16 + nt + (lane >> 4);
        ldmatrix_x4_trans(b0, b1, b2, b3, smem_u32(&kvb[swz(r, ch)]));
        mma_bf16_16816(o[nt], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(o[nt + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();  // this ring slot, p and s_part are rewritten next tile
  }
  cp_async_wait<0>();
  __syncthreads();
  // ---- add the two row halves
  if (half == 1) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      *reinterpret_cast<float2*>(&sm.ohalf[quarter][g][nt * 8 + 2 * t]) =
          make_float2(o[nt][0], o[nt][1]);
      *reinterpret_cast<float2*>(&sm.ohalf[quarter][g + 8][nt * 8 + 2 * t]) =
          make_float2(o[nt][2], o[nt][3]);
    }
  }
  __syncthreads();
  if (half == 1) return;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const float2 x = *reinterpret_cast<const float2*>(&sm.ohalf[quarter][g][nt * 8 + 2 * t]);
    const float2 y = *reinterpret_cast<const float2*>(&sm.ohalf[quarter][g + 8][nt * 8 + 2 * t]);
    o[nt][0] += x.x; o[nt][1] += x.y; o[nt][2] += y.x; o[nt][3] += y.y;
  }
  const int h_lo = hg * kHG + g, h_hi = h_lo + 8;
  const float m_lo = sm.m[g], m_hi = sm.m[g + 8];
  const float l_lo = sm.l[g], l_hi = sm.l[g + 8];
  if (n_split == 1) {
    const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
    const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
    __nv_bfloat16* o_lo = out + ((long long)qi * Hm + h_lo) * kL + quarter * 128;
    __nv_bfloat16* o_hi = out + ((long long)qi * Hm + h_hi) * kL + quarter * 128;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      *reinterpret_cast<uint32_t*>(o_lo + nt * 8 + 2 * t) =
          pack_bf16(o[nt][0] * inv_lo, o[nt][1] * inv_lo);
      *reinterpret_cast<uint32_t*>(o_hi + nt * 8 + 2 * t) =
          pack_bf16(o[nt][2] * inv_hi, o[nt][3] * inv_hi);
    }
    if (lse && quarter == 0 && t == 0) {
      lse[(long long)qi * Hm + h_lo] = l_lo > 0.f ? (m_lo + log2f(l_lo)) / kLog2e : -INFINITY;
      lse[(long long)qi * Hm + h_hi] = l_hi > 0.f ? (m_hi + log2f(l_hi)) / kLog2e : -INFINITY;
    }
    return;
  }
  // partial: unnormalised O, running max (base 2) and sum
  const long long slot_lo = ((long long)qi * Hm + h_lo) * n_split + split;
  const long long slot_hi = ((long long)qi * Hm + h_hi) * n_split + split;
  float* p_lo = part_o + slot_lo * kL + quarter * 128;
  float* p_hi = part_o + slot_hi * kL + quarter * 128;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    *reinterpret_cast<float2*>(p_lo + nt * 8 + 2 * t) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(p_hi + nt * 8 + 2 * t) = make_float2(o[nt][2], o[nt][3]);
  }
  if (quarter == 0 && t == 0) {
    part_ml[slot_lo * 2] = m_lo;
    part_ml[slot_lo * 2 + 1] = l_lo;
    part_ml[slot_hi * 2] = m_hi;
    part_ml[slot_hi * 2 + 1] = l_hi;
  }
}

// Merge split partials: one CTA per (query, head); 128 threads x 4 latent columns.
// Every split's partial row and (max, sum) pair of a batch is requested before
// any of them is used, and the batch maximum rescales the running sums, so up to
// kMergeMax splits cost a single round trip to memory.
constexpr int kMergeMax = 16;   // splits held in registers per batch
__global__ void __launch_bounds__(128)
    mla_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml, int Hm,
                     int n_split, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  pdl_wait();
  // the kernel after this one (the first of the next call) may start its
  // prologue: it waits for this one before it reads anything
  pdl_launch_dependents();
  const long long qh = (long long)blockIdx.y * Hm + blockIdx.x;
  const float* ml = part_ml + qh * n_split * 2;
  const int d = threadIdx.x * 4;
  float mx = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n_split; s0 += kMergeMax) {
    float4 v[kMergeMax];
    float mm[kMergeMax], ll[kMergeMax];
#pragma unroll
    for (int u = 0; u < kMergeMax; ++u) {
      const int sp = s0 + u;
      ll[u] = 0.f;
      mm[u] = -INFINITY;
      if (sp < n_split) {
        v[u] = __ldg(reinterpret_cast<const float4*>(part_o + (qh * n_split + sp) * kL + d));
        mm[u] = __ldg(ml + 2 * sp);
        ll[u] = __ldg(ml + 2 * sp + 1);
      }
    }
    float bm = mx;
#pragma unroll
    for (int u = 0; u < kMergeMax; ++u)
      if (ll[u] > 0.f) bm = fmaxf(bm, mm[u]);
    if (bm == -INFINITY) continue;  // nothing selected so far
    const float r = mx == -INFINITY ? 0.f : ex2_fast(mx - bm);
    den *= r;
    acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
    mx = bm;
#pragma unroll
    for (int u = 0; u < kMergeMax; ++u) {
      if (ll[u] > 0.f) {
        const float w = ex2_fast(mm[u] - mx);
        den += ll[u] * w;
        acc.x += w * v[u].x; acc.y += w * v[u].y; acc.z += w * v[u].z; acc.w += w * v[u].w;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  *reinterpret_cast<uint2*>(out + qh * kL + d) =
      make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
  if (lse && threadIdx.x == 0) lse[qh] = den > 0.f ? (mx + log2f(den)) / kLog2e : -INFINITY;
}

// Generic SIMT kernel: one CTA per (head, query); two passes over the rows.
template <typename T>
__global__ void __launch_bounds__(256)
    mla_simt_kernel(const T* __restrict__ q_lat, const T* __restrict__ kv,
                    const int32_t* __restrict__ cu_seqlens, const int32_t* __restrict__ q_seq,
                    const int32_t* __restrict__ token_ids, int B, int Hm, int L, int W,
                    float sm_scale, T* __restrict__ out, float* __restrict__ lse,
                    int32_t* status) {
  extern __shared__ float sh[];  // q [L] | z [W] | red [32]
  float* sq = sh;
  float* sz = sh + L;
  float* red = sz + W;
  pdl_wait();
  const int h = blockIdx.x, qi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int b = q_seq ? q_seq[qi] : 0;
  const bool seq_ok = b >= 0 && b < B;
  if (!seq_ok && h == 0 && threadIdx.x == 0) flag(status, DSA_DEV_BAD_QSEQ);
  const long long row_base = seq_ok ? cu_seqlens[b] : 0;
  const int Tb = seq_ok ? cu_seqlens[b + 1] - cu_seqlens[b] : 0;
  for (int d = threadIdx.x; d < L; d += blockDim.x)
    sq[d] = Act<T>::to_f(q_lat[((long long)qi * Hm + h) * L + d]);
  __syncthreads();
  const int32_t* toks = token_ids + (long long)qi * W;
  for (int j = warp; j < W; j += nw) {
    const int tok = seq_ok ? toks[j] : -1;
    float z = -INFINITY;
    if (tok >= Tb && lane == 0 && h == 0) flag(status, DSA_DEV_BAD_TOKEN);
    if (tok >= 0 && tok < Tb) {
      const T* row = kv + (row_base + tok) * L;
      float acc = 0.f;
      for (int d = lane; d < L; d += 32) acc = fmaf(Act<T>::to_f(row[d]), sq[d], acc);
      z = warp_sum(acc) * sm_scale;
    }
    if (lane == 0) sz[j] = z;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < W; j += blockDim.x) mx = fmaxf(mx, sz[j]);
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
    red[0] = m;
  }
  __syncthreads();
  const float m = red[0];
  __syncthreads();
  float den = 0.f;
  for (int j = threadIdx.x; j < W; j += blockDim.x) {
    const float e = (m == -INFINITY || sz[j] == -INFINITY) ? 0.f : expf(sz[j] - m);
    sz[j] = e;
    den += e;
  }
  den = warp_sum(den);
  if (lane == 0) red[warp] = den;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[w];
    red[0] = s;
  }
  __syncthreads();
  den = red[0];
  const float inv = den > 0.f ? 1.f / den : 0.f;
  for (int d = threadIdx.x; d < L; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < W; ++j) {
      const float e = sz[j];
      if (e != 0.f) acc = fmaf(e, Act<T>::to_f(kv[(row_base + toks[j]) * L + d]), acc);
    }
    out[((long long)qi * Hm + h) * L + d] = Act<T>::from_f(acc * inv);
  }
  if (lse && threadIdx.x == 0) lse[(long long)qi * Hm + h] = den > 0.f ? m + logf(den) : -INFINITY;
}

// Generic kernel on a paged cache: the kernel above with each token's row found
// through the block table and read as bf16, fp32 or E4M3 code * row scale.
__device__ __forceinline__ float paged_value(const PagedKv& pk, long long prow, int d, int L) {
  const long long o = prow * L + d;
  if (pk.kv_dtype == DSA_BF16)
    return __bfloat162float(static_cast<const __nv_bfloat16*>(pk.pages)[o]);
  if (pk.kv_dtype == DSA_F32) return static_cast<const float*>(pk.pages)[o];
  const __half_raw h =
      __nv_cvt_fp8_to_halfraw(static_cast<const __nv_fp8_storage_t*>(pk.pages)[o], __NV_E4M3);
  return __half2float(*reinterpret_cast<const __half*>(&h)) * pk.row_scale[prow];
}

template <typename T>
__global__ void __launch_bounds__(256)
    mla_simt_paged_kernel(const T* __restrict__ q_lat, PagedKv pk,
                          const int32_t* __restrict__ q_seq, const int32_t* __restrict__ token_ids,
                          int B, int Hm, int L, int W, float sm_scale, T* __restrict__ out,
                          float* __restrict__ lse, int32_t* status) {
  extern __shared__ float sh[];  // q [L] | z [W] | row [W] (int) | red [32]
  float* sq = sh;
  float* sz = sh + L;
  int* srow = reinterpret_cast<int*>(sz + W);
  float* red = reinterpret_cast<float*>(srow + W);
  pdl_wait();
  const int h = blockIdx.x, qi = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int b = q_seq ? q_seq[qi] : 0;
  const bool seq_ok = b >= 0 && b < B;
  if (!seq_ok && h == 0 && threadIdx.x == 0) flag(status, DSA_DEV_BAD_QSEQ);
  const int Tb = seq_ok ? pk.seq_lens[b] : 0;
  for (int d = threadIdx.x; d < L; d += blockDim.x)
    sq[d] = Act<T>::to_f(q_lat[((long long)qi * Hm + h) * L + d]);
  const int32_t* toks = token_ids + (long long)qi * W;
  for (int j = threadIdx.x; j < W; j += blockDim.x) {
    const int tok = seq_ok ? toks[j] : -1;
    int prow = -1;
    if (tok >= Tb) {
      if (h == 0) flag(status, DSA_DEV_BAD_TOKEN);
    } else if (tok >= 0) {
      const int blk = tok / pk.page_size;
      const int page = blk < pk.max_pages ? pk.block_table[(long long)b * pk.max_pages + blk] : -1;
      if (page < 0 || page >= pk.n_pages) {
        if (h == 0) flag(status, DSA_DEV_BAD_PAGE);
      } else {
        prow = page * pk.page_size + tok % pk.page_size;
      }
    }
    srow[j] = prow;
  }
  __syncthreads();
  for (int j = warp; j < W; j += nw) {
    const int prow = srow[j];
    float z = -INFINITY;
    if (prow >= 0) {
      float acc = 0.f;
      for (int d = lane; d < L; d += 32) acc = fmaf(paged_value(pk, prow, d, L), sq[d], acc);
      z = warp_sum(acc) * sm_scale;
    }
    if (lane == 0) sz[j] = z;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < W; j += blockDim.x) mx = fmaxf(mx, sz[j]);
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
    red[0] = m;
  }
  __syncthreads();
  const float m = red[0];
  __syncthreads();
  float den = 0.f;
  for (int j = threadIdx.x; j < W; j += blockDim.x) {
    const float e = (m == -INFINITY || sz[j] == -INFINITY) ? 0.f : expf(sz[j] - m);
    sz[j] = e;
    den += e;
  }
  den = warp_sum(den);
  if (lane == 0) red[warp] = den;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[w];
    red[0] = s;
  }
  __syncthreads();
  den = red[0];
  const float inv = den > 0.f ? 1.f / den : 0.f;
  for (int d = threadIdx.x; d < L; d += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < W; ++j) {
      const float e = sz[j];
      if (e != 0.f) acc = fmaf(e, paged_value(pk, srow[j], d, L), acc);
    }
    out[((long long)qi * Hm + h) * L + d] = Act<T>::from_f(acc * inv);
  }
  if (lse && threadIdx.x == 0) lse[(long long)qi * Hm + h] = den > 0.f ? m + logf(den) : -INFINITY;
}

bool fast_path(int Hm, int L, int dtype) { return dtype == DSA_BF16 && L == kL && Hm % kHG == 0; }

// Split count: (query, head group, split) CTAs covering the SMs once at most;
// at most 64 splits (the merge keeps one weight per split on chip).
void split_plan(int Q, int Hm, int W, int* n_split, int* rows_per_split) {
  const int n_hg = Hm / kHG;
  int s = num_sms() / (Q * n_hg);
  const int max_s = (W + kNT - 1) / kNT;
  if (s > max_s) s = max_s;
  if (s > 64) s = 64;
  if (s < 1) s = 1;
  int rows = (W + s - 1) / s;
  *rows_per_split = rows;
  *n_split = (W + rows - 1) / rows;
}

}  // namespace

size_t mla_workspace_size(int Q, int Hm, int L, int out_width, int dtype) {
  int n_split = 1;
  if (mla_umma_ok(Q, Hm, L, out_width, dtype)) {
    n_split = mla_umma_splits(out_width);
  } else if (mla_umma_shape_ok(Hm, L, dtype)) {
    n_split = mla_stream_splits(Q, out_width);
  } else if (fast_path(Hm, L, dtype)) {
    int rows;
    split_plan(Q, Hm, out_width, &n_split, &rows);
  }
  if (n_split == 1) return 0;
  const size_t slots = (size_t)Q * Hm * n_split;
  return slots * L * 4 + slots * 2 * 4;
}

int launch_mla_selected_decode(const void* q_lat, const void* kv, const int32_t* cu_seqlens,
                               const int32_t* q_seq, const int32_t* token_ids, int Q, int B,
                               int Hm, int L, int out_width, float sm_scale, int dtype, void* out,
                               float* lse, void* workspace, size_t ws_bytes, int32_t* status_dev,
                               cudaStream_t stream, bool early) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (mla_umma_ok(Q, Hm, L, out_width, dtype)) {
    const int n_split = mla_umma_splits(out_width);
    if (n_split > 1 && ws_bytes < mla_workspace_size(Q, Hm, L, out_width, dtype))
      return DSA_ERR_WORKSPACE;
    float* part_o = n_split > 1 ? static_cast<float*>(workspace) : nullptr;
    float* part_ml = part_o ? part_o + (size_t)Q * Hm * n_split * L : nullptr;
    const int r = launch_mla_umma(q_lat, kv, cu_seqlens, q_seq, token_ids, Q, B, out_width,
                                  sm_scale, out, lse, part_o, part_ml, early, status_dev,
                                  stream);
    if (r != DSA_OK || n_split == 1) return r;
    cfg.gridDim = dim3(Hm, Q, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    return launch_kernel(&cfg, mla_merge_kernel, (const float*)part_o,
                         (const float*)part_ml, Hm, n_split, (__nv_bfloat16*)out,
                         lse) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  if (mla_umma_shape_ok(Hm, L, dtype)) {  // many queries: the streaming tcgen05 kernel
    const int n_split = mla_stream_splits(Q, out_width);
    if (n_split > 1 && ws_bytes < mla_workspace_size(Q, Hm, L, out_width, dtype))
      return DSA_ERR_WORKSPACE;
    float* part_o = n_split > 1 ? static_cast<float*>(workspace) : nullptr;
    float* part_ml = part_o ? part_o + (size_t)Q * Hm * n_split * L : nullptr;
    const int r = launch_mla_stream(q_lat, kv, cu_seqlens, q_seq, token_ids, Q, B, out_width,
                                    sm_scale, out, lse, part_o, part_ml, status_dev, stream);
    if (r != DSA_OK || n_split == 1) return r;
    cfg.gridDim = dim3(Hm, Q, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    return launch_kernel(&cfg, mla_merge_kernel, (const float*)part_o,
                         (const float*)part_ml, Hm, n_split, (__nv_bfloat16*)out,
                         lse) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  if (fast_path(Hm, L, dtype)) {
    int n_split, rows;
    split_plan(Q, Hm, out_width, &n_split, &rows);
    if (rows > kMaxRows) return DSA_ERR_UNSUPPORTED;
    if (n_split > 1 && ws_bytes < mla_workspace_size(Q, Hm, L, out_width, dtype))
      return DSA_ERR_WORKSPACE;
    float* part_o = static_cast<float*>(workspace);
    float* part_ml = part_o ? part_o + (size_t)Q * Hm * n_split * L : nullptr;
    const size_t smem = sizeof(MlaSmem) + (size_t)((rows + kNT - 1) / kNT * kNT) * 4;
    cudaFuncSetAttribute(mla_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cfg.gridDim = dim3(n_split, Hm / kHG, Q);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    if (launch_kernel(&cfg, mla_mma_kernel, (const __nv_bfloat16*)q_lat,
                      (const __nv_bfloat16*)kv, cu_seqlens, q_seq, token_ids, B, Hm,
                      out_width, rows, sm_scale, (__nv_bfloat16*)out, lse, part_o, part_ml,
                      status_dev) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (n_split > 1) {
      cfg.gridDim = dim3(Hm, Q, 1);
      cfg.blockDim = dim3(128, 1, 1);
      cfg.dynamicSmemBytes = 0;
      if (launch_kernel(&cfg, mla_merge_kernel, (const float*)part_o,
                        (const float*)part_ml, Hm, n_split, (__nv_bfloat16*)out,
                        lse) != cudaSuccess)
        return DSA_ERR_CUDA;
    }
    return DSA_OK;
  }
  if (L % 8 != 0 || L > 1024 || Hm > 128 || out_width > 16384) return DSA_ERR_UNSUPPORTED;
  const size_t smem = ((size_t)L + out_width + 32) * 4;
  cfg.gridDim = dim3(Hm, Q, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaError_t e;
  if (dtype == DSA_BF16) {
    cudaFuncSetAttribute(mla_simt_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    e = launch_kernel(&cfg, mla_simt_kernel<__nv_bfloat16>, (const __nv_bfloat16*)q_lat,
                      (const __nv_bfloat16*)kv, cu_seqlens, q_seq, token_ids, B, Hm, L,
                      out_width, sm_scale, (__nv_bfloat16*)out, lse, status_dev);
  } else {
    cudaFuncSetAttribute(mla_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    e = launch_kernel(&cfg, mla_simt_kernel<float>, (const float*)q_lat, (const float*)kv,
                      cu_seqlens, q_seq, token_ids, B, Hm, L, out_width, sm_scale,
                      (float*)out, lse, status_dev);
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

namespace {
// The paged calls run the tcgen05 kernels at every query count: the one-tile
// kernel for few queries, the streaming one beyond four waves of its CTAs.
bool paged_umma(int Q, int Hm, int L, int out_width, int dtype, int kv_dtype) {
  (void)Q;
  (void)out_width;
  return mla_umma_shape_ok(Hm, L, dtype) && (kv_dtype == DSA_BF16 || kv_dtype == DSA_FP8_E4M3);
}
}  // namespace

size_t mla_paged_workspace_size(int Q, int Hm, int L, int out_width, int dtype, int kv_dtype) {
  if (!paged_umma(Q, Hm, L, out_width, dtype, kv_dtype)) return 0;
  const int n_split = mla_umma_ok(Q, Hm, L, out_width, dtype) ? mla_umma_splits(out_width)
                                                              : mla_stream_splits(Q, out_width);
  if (n_split == 1) return 0;
  const size_t slots = (size_t)Q * Hm * n_split;
  return slots * L * 4 + slots * 2 * 4;
}

int launch_mla_paged_decode(const void* q_lat, const PagedKv& kv, const int32_t* q_seq,
                            const int32_t* token_ids, int Q, int B, int Hm, int L, int out_width,
                            float sm_scale, int dtype, void* out, float* lse, void* workspace,
                            size_t ws_bytes, int32_t* status_dev, cudaStream_t stream) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (paged_umma(Q, Hm, L, out_width, dtype, kv.kv_dtype)) {
    // few queries: one CTA per 128 rows and 32 heads; many: the streaming kernel
    const bool few = mla_umma_ok(Q, Hm, L, out_width, dtype);
    const int n_split = few ? mla_umma_splits(out_width) : mla_stream_splits(Q, out_width);
    if (ws_bytes < mla_paged_workspace_size(Q, Hm, L, out_width, dtype, kv.kv_dtype))
      return DSA_ERR_WORKSPACE;
    float* part_o = n_split > 1 ? static_cast<float*>(workspace) : nullptr;
    float* part_ml = part_o ? part_o + (size_t)Q * Hm * n_split * L : nullptr;
    const int r = few ? launch_mla_umma(q_lat, nullptr, nullptr, q_seq, token_ids, Q, B,
                                        out_width, sm_scale, out, lse, part_o, part_ml, false,
                                        status_dev, stream, &kv)
                      : launch_mla_stream(q_lat, nullptr, nullptr, q_seq, token_ids, Q, B,
                                          out_width, sm_scale, out, lse, part_o, part_ml,
                                          status_dev, stream, &kv);
    if (r != DSA_OK || n_split == 1) return r;
    cfg.gridDim = dim3(Hm, Q, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    return launch_kernel(&cfg, mla_merge_kernel, (const float*)part_o,
                         (const float*)part_ml, Hm, n_split, (__nv_bfloat16*)out,
                         lse) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  if (L % 8 != 0 || L > 1024 || Hm > 128 || out_width > 16384) return DSA_ERR_UNSUPPORTED;
  const size_t smem = ((size_t)L + 2 * (size_t)out_width + 32) * 4;
  cfg.gridDim = dim3(Hm, Q, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaError_t e;
  if (dtype == DSA_BF16) {
    cudaFuncSetAttribute(mla_simt_paged_kernel<__nv_bfloat16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    e = launch_kernel(&cfg, mla_simt_paged_kernel<__nv_bfloat16>,
                      (const __nv_bfloat16*)q_lat, kv, q_seq, token_ids, B, Hm, L, out_width,
                      sm_scale, (__nv_bfloat16*)out, lse, status_dev);
  } else {
    cudaFuncSetAttribute(mla_simt_paged_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    e = launch_kernel(&cfg, mla_simt_paged_kernel<float>, (const float*)q_lat, kv, q_seq,
                      token_ids, B, Hm, L, out_width, sm_scale, (float*)out, lse,
                      status_dev);
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
