// The arithmetic of one pool of kpool_compress, shared by the compress
// kernels (kpool_compress.cu) and by the scoring kernel that compresses a
// decode step's new pools itself (index_scores_umma.cu), so that every path
// writes bit-identical keys.
//
// Module glm5next_dsa, "Traps carried from Slice 8": LayerNorm with bias per
// token, rounded to the activation dtype; softmax over the slot axis per
// channel of gate + ape; the pooled key is the softmax-weighed sum of the
// normalised rows.  A pool is valid when all its slots are.
#pragma once

#include "dsa_internal.cuh"

namespace dsa {

// softmax weights as 2^((l - max) log2 e): e^x in the form the special-function
// unit evaluates (the same expression in every compress kernel, so they agree)
constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32, a few ulp); the
// arguments here are <= 0, and a result below 2^-126 flushes to zero: a slot
// weight that small is lost against the largest slot's weight of 1
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// sum of N channel values, left to right
template <int N>
__device__ __forceinline__ float lane_sum(const float* x) {
  float v = x[0];
#pragma unroll
  for (int i = 1; i < N; ++i) v = v + x[i];
  return v;
}
// sum of squares of N channel values, left to right
template <int N>
__device__ __forceinline__ float lane_sq(const float* x) {
  float v = x[0] * x[0];
#pragma unroll
  for (int i = 1; i < N; ++i) v = fmaf(x[i], x[i], v);
  return v;
}
// warp sum: lanes 2j and 2j + 1 first, then across the pairs
__device__ __forceinline__ float pair_first_warp_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
#pragma unroll
  for (int o = 16; o > 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T, int V>
struct Vec;  // V consecutive activation values
template <>
struct Vec<float, 1> {
  static __device__ __forceinline__ void load(const float* p, float* o) { o[0] = __ldg(p); }
  static __device__ __forceinline__ void store(float* p, const float* v) { *p = v[0]; }
};
template <>
struct Vec<float, 2> {
  static __device__ __forceinline__ void load(const float* p, float* o) {
    float2 t = __ldg(reinterpret_cast<const float2*>(p));
    o[0] = t.x; o[1] = t.y;
  }
  static __device__ __forceinline__ void store(float* p, const float* v) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
  }
};
template <>
struct Vec<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float* o) {
    float4 t = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = t.x; o[1] = t.y; o[2] = t.z; o[3] = t.w;
  }
  static __device__ __forceinline__ void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<float, 8> {
  static __device__ __forceinline__ void load(const float* p, float* o) {
    Vec<float, 4>::load(p, o);
    Vec<float, 4>::load(p + 4, o + 4);
  }
  static __device__ __forceinline__ void store(float* p, const float* v) {
    Vec<float, 4>::store(p, v);
    Vec<float, 4>::store(p + 4, v + 4);
  }
};
template <>
struct Vec<__nv_bfloat16, 1> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* o) {
    o[0] = __bfloat162float(p[0]);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
    p[0] = __float2bfloat16_rn(v[0]);
  }
};
template <>
struct Vec<__nv_bfloat16, 2> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* o) {
    uint32_t t = __ldg(reinterpret_cast<const unsigned int*>(p));
    o[0] = bf16lo(t); o[1] = bf16hi(t);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
    *reinterpret_cast<uint32_t*>(p) = pack_bf16(v[0], v[1]);
  }
};
template <>
struct Vec<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* o) {
    uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
    o[0] = bf16lo(t.x); o[1] = bf16hi(t.x); o[2] = bf16lo(t.y); o[3] = bf16hi(t.y);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
  }
};
template <>
struct Vec<__nv_bfloat16, 8> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* o) {
    uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
    o[0] = bf16lo(t.x); o[1] = bf16hi(t.x); o[2] = bf16lo(t.y); o[3] = bf16hi(t.y);
    o[4] = bf16lo(t.z); o[5] = bf16hi(t.z); o[6] = bf16lo(t.w); o[7] = bf16hi(t.w);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
    *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]),
                                              pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  }
};


// One complete pool by one warp: lane l owns channels [l*V, l*V + V) of the
// D = 32*V channels; s0 is the pool's first token row.  Writes the key (out:
// the lane's channels of the key row), the pool's first token (`start`) and
// its valid byte.
template <typename T, int V>
__device__ __forceinline__ void compress_pool_warp(
    const T* __restrict__ k, const T* __restrict__ gate, const uint8_t* __restrict__ valid,
    const float* __restrict__ ape, const T* __restrict__ ln_gamma, const T* __restrict__ ln_beta,
    float ln_eps, long long s0, int kpool, int lane, T* out, int start, int32_t* start_out,
    uint8_t* valid_out) {
  constexpr int D = 32 * V;
  float g[V], be[V];
  Vec<T, V>::load(ln_gamma + lane * V, g);
  Vec<T, V>::load(ln_beta + lane * V, be);

  float kn[kKpoolMax][V], lg[kKpoolMax][V], ap[kKpoolMax][V];
  bool all_valid = true;
  // every slot's rows and slot biases are requested before any reduction runs,
  // so the loads of the pool overlap instead of waiting one slot at a time
#pragma unroll
  for (int s = 0; s < kKpoolMax; ++s) {
    if (s < kpool) {
      Vec<T, V>::load(k + (s0 + s) * D + lane * V, kn[s]);
      Vec<T, V>::load(gate + (s0 + s) * D + lane * V, lg[s]);
#pragma unroll
      for (int i = 0; i < V; ++i) ap[s][i] = __ldg(ape + s * D + lane * V + i);  // 4-byte aligned
      all_valid &= valid[s0 + s] != 0;
    }
  }
  // logits, their per-channel maximum over the slots
#pragma unroll
  for (int s = 0; s < kKpoolMax; ++s)
    if (s < kpool)
#pragma unroll
      for (int i = 0; i < V; ++i) lg[s][i] = lg[s][i] + ap[s][i];
  float m[V], den[V], acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    m[i] = lg[0][i];
#pragma unroll
    for (int s = 1; s < kKpoolMax; ++s)
      if (s < kpool) m[i] = fmaxf(m[i], lg[s][i]);
    den[i] = acc[i] = 0.f;
  }
  // per slot: LayerNorm (statistics summed over the lane's channels, then the
  // lane pair, then the warp: the order of the bulk kernel below), the
  // normalised row rounded to the activation dtype, and its softmax weight
#pragma unroll
  for (int s = 0; s < kKpoolMax; ++s) {
    if (s < kpool) {
      const float mean = pair_first_warp_sum(lane_sum<V>(kn[s])) * (1.0f / D);
      float dx[V];
#pragma unroll
      for (int i = 0; i < V; ++i) dx[i] = kn[s][i] - mean;
      const float var = pair_first_warp_sum(lane_sq<V>(dx)) * (1.0f / D);
      const float rstd = rsqrtf(var + ln_eps);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const float y = Act<T>::round(fmaf(dx[i] * rstd, g[i], be[i]));
        const float e = exp2_approx((lg[s][i] - m[i]) * kLog2e);
        den[i] += e;
        acc[i] = fmaf(e, y, acc[i]);
      }
    }
  }
  float res[V];
#pragma unroll
  for (int i = 0; i < V; ++i) res[i] = __fdividef(acc[i], den[i]);  // den in [1, kpool]
  Vec<T, V>::store(out, res);
  if (lane == 0) {
    *start_out = start;
    *valid_out = all_valid ? 1 : 0;
  }
}

// A sentinel entry (past the sequence's complete pools): zero key, start -1,
// not valid.
template <typename T, int V>
__device__ __forceinline__ void compress_sentinel_warp(int lane, T* out, int32_t* start_out,
                                                       uint8_t* valid_out) {
  float z[V];
#pragma unroll
  for (int i = 0; i < V; ++i) z[i] = 0.f;
  Vec<T, V>::store(out, z);
  if (lane == 0) {
    *start_out = -1;
    *valid_out = 0;
  }
}

// First valid token of the sequence at rows [lo, lo + T) by one warp (T when
// there is none): 256 valid bytes per round, every lane gets the value.
__device__ __forceinline__ int first_valid_warp(const uint8_t* __restrict__ valid, long long lo,
                                                int T, int lane) {
  for (int base = 0; base < T; base += 256) {
    uint32_t nz[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // every load first, then the votes
      const int t = base + j * 32 + lane;
      nz[j] = t < T ? valid[lo + t] : 0u;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t m = __ballot_sync(0xffffffffu, nz[j] != 0u);
      if (m != 0u) return base + j * 32 + __ffs((int)m) - 1;
    }
  }
  return T;
}

}  // namespace dsa
