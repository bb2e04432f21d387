// Combining split-KV partials of the selected-row attention.
//
// A split covers a subset of a query's selected rows and leaves, per (query,
// head), its unnormalised output O_s = sum_j 2^(z_j - m_s) c_j over its rows,
// the reference m_s (base 2) and the sum l_s = sum_j 2^(z_j - m_s).  The
// attention over all rows is (sum_s 2^(m_s - M) O_s) / (sum_s 2^(m_s - M) l_s)
// for any M; M = max over the splits with l_s > 0 keeps every factor <= 1, and
// lse = (M + log2 sum) / log2(e).  A split with l_s = 0 selected nothing.
#pragma once

#include "dsa_internal.cuh"

namespace dsa {

constexpr float kMergeLog2e = 1.4426950408889634f;
constexpr int kMergeBatch = 16;  // splits whose partials are requested at once

// Merge the n_split partials of (query, head) row `qh` at latent columns
// d .. d+3 and write them (normalised, bf16) to out; lse is written when
// `write_lse`.  Every partial of a batch is requested before any is used, and
// the batch maximum rescales the running sums, so up to kMergeBatch splits cost
// one round trip to memory.  Loads bypass L1: the partials may come from other
// CTAs of the same grid.
template <int kL>
__device__ __forceinline__ void merge_partials(const float* __restrict__ part_o,
                                               const float* __restrict__ part_ml, long long qh,
                                               int n_split, int d, __nv_bfloat16* __restrict__ out,
                                               float* __restrict__ lse, bool write_lse) {
  const float* ml = part_ml + qh * n_split * 2;
  float mx = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < n_split; s0 += kMergeBatch) {
    float4 v[kMergeBatch];
    float mm[kMergeBatch], ll[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int sp = s0 + u;
      ll[u] = 0.f;
      mm[u] = -INFINITY;
      if (sp < n_split) {
        v[u] = __ldcg(reinterpret_cast<const float4*>(part_o + (qh * n_split + sp) * kL + d));
        mm[u] = __ldcg(ml + 2 * sp);
        ll[u] = __ldcg(ml + 2 * sp + 1);
      }
    }
    float bm = mx;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u)
      if (ll[u] > 0.f) bm = fmaxf(bm, mm[u]);
    if (bm == -INFINITY) continue;  // nothing selected so far
    const float r = mx == -INFINITY ? 0.f : exp2f(mx - bm);
    den *= r;
    acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
    mx = bm;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      if (ll[u] > 0.f) {
        const float w = exp2f(mm[u] - mx);
        den += ll[u] * w;
        acc.x += w * v[u].x; acc.y += w * v[u].y; acc.z += w * v[u].z; acc.w += w * v[u].w;
      }
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  *reinterpret_cast<uint2*>(out + qh * kL + d) =
      make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
  if (write_lse && lse) lse[qh] = den > 0.f ? (mx + log2f(den)) / kMergeLog2e : -INFINITY;
}

}  // namespace dsa
