// Indexer projections: the dense contractions that turn one layer's per-token
// activations into the indexer's and the attention's inputs (module
// glm5next_dsa, Modules: build and layer - the DSA block's tensors; Traps
// carried from Slice 8 - NoPE, so the query carries no rotary part):
//
//   hidden x      -> k, gate (the indexer key and its slot logits, D each)
//                    and the per-head indexer weights (H)
//   query latent  -> the indexer query (H x D) and the MLA no-rope query
//                    (Hm x nope)
//   MLA no-rope query, per head -> the query in latent space (L): the key
//                    up-projection is absorbed, so the attention scores a
//                    latent cache row c directly (<q_lat_h, c> equals
//                    <q_nope_h, W_uk_h c>)
//
// One tcgen05 kernel does all three.  A tile is 128 output features (the MMA's
// M, one TMEM lane each) by BN tokens (the MMA's N): in decode the token count
// is a handful and the kernel is a stream over the weight rows; in a prefill
// chunk it is a compute-bound grid of 128 x 128 tiles.  Operands come in by TMA
// with the 128-byte swizzle (64 contraction elements per stage), one thread
// issues the MMAs, the accumulator lives in TMEM, and four epilogue warps read
// it back (tcgen05.ld), scale it and store each feature to its output tensor.
// When a grid of whole tiles would leave SMs idle, the contraction is split:
// every split writes an fp32 partial tile to the workspace, and the split that
// arrives last (a counter per tile, no waiting) adds the partials in split
// order - the result does not depend on arrival order - writes the output and
// re-arms the counter.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "umma.cuh"

namespace dsa {
namespace {

constexpr int kPM = 128;            // output features per tile (MMA M = TMEM lanes)
constexpr int kPK = 64;             // contraction elements per stage (one 128-byte row)
constexpr int kPSegs = 3;           // output tensors per launch

// Features [f0, f1) of every batch go to one output tensor:
//   dst[row(t) * ld + b * bstride + (f - f0)] = alpha * acc[f, t]
// with row(t) = row_map[t] when the segment uses the map (a negative entry
// drops the token), else t.
struct ProjSeg {
  void* dst;
  long long ld;
  long long bstride;
  int f0, f1;
  int f32;       // 1: fp32 output, 0: bf16
  int use_map;
  float alpha;
};
struct ProjArgs {
  ProjSeg seg[kPSegs];
  int n_segs;
  int M;             // output features per batch
  int T;             // tokens
  int k_steps;       // contraction stages per batch (ceil(K / 64))
  int x_col_batch;   // column offset of batch b's inputs in x: b * x_col_batch
  const int32_t* row_map;
  float* part;       // split partials: [tile][split][BN][128] fp32
  uint32_t* counter; // per tile
  int wait_start;    // 1: wait for the previous kernel before reading anything;
                     // 2: before reading x (the weights may be read earlier)
  int wait_end;      // wait for the previous kernel before finishing
};

template <int BN>
struct PCfg {
  static constexpr int kABytes = kPM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN <= 16 ? 4 : BN <= 64 ? 6 : BN <= 128 ? 5 : 4;
  // a handful of tokens: up to three CTAs per SM, each streaming its own
  // weight rows; otherwise one persistent CTA per SM
  static constexpr int kCtasPerSm = BN <= 16 ? 3 : 1;
  // warp 0 TMA, warp 1 MMA, then the epilogue: four warps (one per TMEM lane
  // quarter) for a handful of tokens, eight (two per quarter, each taking half
  // of the tile's tokens) otherwise
  static constexpr int kEpiWarps = BN <= 16 ? 4 : 8;
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int kAccCols = BN;                    // one accumulator
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;  // two, double-buffered
  // per epilogue warp, 16 tokens x 32 features of fp32 on their way to
  // 16-byte stores (rows padded to 36 floats: 16-byte aligned, and the
  // 128-bit reads of eight lanes fall on distinct banks)
  static constexpr int kOutPitch = 36;
  static constexpr int kOutBytes = BN <= 16 ? 0 : kEpiWarps * 16 * kOutPitch * 4;
  static constexpr size_t kSmem = 1024 + (size_t)kStages * kStageBytes + kOutBytes;
};

template <int kWarps>
__device__ __forceinline__ void proj_epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory");
}

// One output feature: where its values go, fixed for the whole tile.
struct ProjOut {
  unsigned char* base;  // the feature's element of token row 0 (batch offset included)
  long long ld_bytes;   // bytes between token rows
  const int32_t* map;   // token -> row, or null
  float alpha;
  bool f32, on;
};
__device__ __forceinline__ ProjOut proj_out(const ProjArgs& pa, int b, int f) {
  ProjOut o{};
  o.on = false;
  if (f >= pa.M) return o;
  for (int s = 0; s < pa.n_segs; ++s) {
    const ProjSeg& g = pa.seg[s];
    if (f >= g.f0 && f < g.f1) {
      const int es = g.f32 ? 4 : 2;
      o.base = static_cast<unsigned char*>(g.dst) + ((long long)b * g.bstride + (f - g.f0)) * es;
      o.ld_bytes = g.ld * es;
      o.map = g.use_map ? pa.row_map : nullptr;
      o.alpha = g.alpha;
      o.f32 = g.f32 != 0;
      o.on = true;
    }
  }
  return o;
}
__device__ __forceinline__ long long proj_row(const int32_t* map, int t) {
  return map ? (long long)map[t] : (long long)t;  // negative: a dropped token
}
__device__ __forceinline__ void proj_put(const ProjOut& o, int t, float v) {
  const long long row = proj_row(o.map, t);
  if (row < 0) return;
  unsigned char* p = o.base + row * o.ld_bytes;
  if (o.f32)
    *reinterpret_cast<float*>(p) = o.alpha * v;
  else
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(o.alpha * v);
}
// Eight consecutive features [f, f + 8) of one segment, 16-byte aligned in
// every token row: stored with one (bf16) or two (fp32) 16-byte stores.
__device__ __forceinline__ bool proj_vec_ok(const ProjArgs& pa, int b, int f, ProjOut* o) {
  *o = proj_out(pa, b, f);
  if (!o->on || f + 8 > pa.M) return false;
  const ProjOut e = proj_out(pa, b, f + 7);
  if (!e.on || e.base != o->base + 7 * (o->f32 ? 4 : 2)) return false;  // one segment
  return ((reinterpret_cast<uintptr_t>(o->base) | (uintptr_t)o->ld_bytes) & 15) == 0;
}

// Work item w (persistent CTAs take w = blockIdx.x, + gridDim.x, ...): the
// output tile (token tiles fastest, then feature tiles, then batches) and the
// split of its contraction.
struct ProjItem {
  int nt, mt, b, split, ks_lo, n_k, tile;
};
__device__ __forceinline__ ProjItem proj_item(const ProjArgs& pa, int w, int S, int n_tiles,
                                              int m_tiles) {
  ProjItem it;
  it.tile = w / S;
  it.split = w % S;
  it.nt = it.tile % n_tiles;
  it.mt = (it.tile / n_tiles) % m_tiles;
  it.b = it.tile / (n_tiles * m_tiles);
  it.ks_lo = (int)((long long)pa.k_steps * it.split / S);
  it.n_k = (int)((long long)pa.k_steps * (it.split + 1) / S) - it.ks_lo;  // >= 1
  return it;
}

template <int BN>
__global__ void __launch_bounds__(PCfg<BN>::kThreads, PCfg<BN>::kCtasPerSm)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_x, const ProjArgs pa, int n_items,
                     int S, int32_t* status) {
  using C = PCfg<BN>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* sbase = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* s_out = reinterpret_cast<float*>(sbase + (size_t)C::kStages * C::kStageBytes);
  __shared__ uint64_t full[C::kStages], empty[C::kStages], tfull[2], tempty[2], done;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort, s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = (pa.T + BN - 1) / BN, m_tiles = (pa.M + kPM - 1) / kPM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&tfull[j], 1);
      mbar_init(&tempty[j], C::kEpiWarps);  // every epilogue warp
    }
    mbar_init(&done, 1);
    fence_mbar_init();
    s_abort = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_w))
                 : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_x))
                 : "memory");
  }
  if (warp == 1) {
    tmem_alloc<C::kTmemCols>(&s_tmem);
    tc_fence_before();
  }
  // wait_start 1: every input may come from the kernel just before; 2: only
  // x may - the weights are model parameters, so the producer streams the
  // first stages of weight rows of its first tile before it waits
  const ProjItem first = proj_item(pa, blockIdx.x, S, n_tiles, m_tiles);
  const int pre = pa.wait_start == 2 ? min(first.n_k, C::kStages) : 0;
  if (pa.wait_start == 1) pdl_wait();
  __syncthreads();  // the barriers are initialised
  if (pre > 0) {
    if (threadIdx.x == 0) {
      const int a_row = first.b * pa.M + first.mt * kPM;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], C::kStageBytes);
        tma_load_2d(sbase + (size_t)i * C::kStageBytes, &tmap_w, (first.ks_lo + i) * kPK, a_row,
                    &full[i]);
      }
    }
    pdl_wait();
  }
  pdl_launch_dependents();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  volatile int* abort = &s_abort;
  auto give_up = [&]() {
    flag(status, DSA_DEV_TIMEOUT);
    *abort = 1;
  };

  if (warp == 0) {
    // ================= TMA producer: one ring across all of this CTA's tiles
    if (lane == 0) {
      int it = 0;  // k-steps issued
      bool stop = false;
      for (int w = blockIdx.x; w < n_items && !stop; w += gridDim.x) {
        const ProjItem pi = proj_item(pa, w, S, n_tiles, m_tiles);
        const int a_row = pi.b * pa.M + pi.mt * kPM;
        for (int i = 0; i < pi.n_k; ++i, ++it) {
          const int st = it % C::kStages;
          if (it >= pre) {  // (the first `pre` weight tiles are already on their way)
            if (*abort) { stop = true; break; }
            if (it >= C::kStages &&
                !mbar_wait_bounded(&empty[st], (uint32_t)((it / C::kStages) - 1) & 1)) {
              give_up();
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(&full[st], C::kStageBytes);
            tma_load_2d(sbase + (size_t)st * C::kStageBytes, &tmap_w, (pi.ks_lo + i) * kPK,
                        a_row, &full[st]);
          }
          tma_load_2d(sbase + (size_t)st * C::kStageBytes + C::kABytes, &tmap_x,
                      pi.b * pa.x_col_batch + (pi.ks_lo + i) * kPK, pi.nt * BN, &full[st]);
        }
      }
      // never leave a copy in flight: wait for the last fill of every stage used
      for (int f = max(0, it - C::kStages); f < it; ++f)
        mbar_wait_bounded(&full[f % C::kStages], (uint32_t)(f / C::kStages) & 1);
    }
  } else if (warp == 1) {
    // ================= MMA issuer: accumulators alternate between two TMEM buffers
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kPM, BN, false);
      int it = 0, j = 0;
      bool stop = false;
      for (int w = blockIdx.x; w < n_items && !stop; w += gridDim.x, ++j) {
        const ProjItem pi = proj_item(pa, w, S, n_tiles, m_tiles);
        const int acc = j & 1;
        if (*abort) break;
        if (j >= 2 && !mbar_wait_bounded(&tempty[acc], (uint32_t)((j >> 1) - 1) & 1)) {
          give_up();
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * C::kAccCols);
        for (int i = 0; i < pi.n_k; ++i, ++it) {
          const int st = it % C::kStages;
          if (*abort || !mbar_wait_bounded(&full[st], (uint32_t)(it / C::kStages) & 1)) {
            give_up();
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(sbase + (size_t)st * C::kStageBytes);
          const uint32_t bb = a + C::kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // 16 elements = 32 bytes per MMA
            umma_bf16(d, sw128_desc(a + kk * 32), sw128_desc(bb + kk * 32), idesc,
                      (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&empty[st]);  // the stage may be refilled once these MMAs are done
        }
        if (!stop) umma_commit(&tfull[acc]);  // the tile's accumulator is complete
      }
      umma_commit(&done);               // every MMA issued above has completed
      mbar_wait_bounded(&done, 0);      // retire them before TMEM is freed
    }
  } else {
    // ================= epilogue (warps 2..)
    const int quarter = warp & 3;  // the TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;  // which half of the tile's tokens (8 warps)
    const int r = quarter * 32 + lane;
    float* so = s_out + (size_t)(warp - 2) * 16 * C::kOutPitch;
    int j = 0;
    for (int w = blockIdx.x; w < n_items; w += gridDim.x, ++j) {
      const ProjItem pi = proj_item(pa, w, S, n_tiles, m_tiles);
      const int acc = j & 1;
      // after a failed wait the loop still runs to the end with nothing read
      // or stored, so that the four warps pass the same named barriers
      const bool ok = !*abort && mbar_wait_bounded(&tfull[acc], (uint32_t)(j >> 1) & 1);
      if (!ok) give_up();
      tc_fence_after();
      const int t0 = pi.nt * BN;
      const int fw = pi.mt * kPM + quarter * 32;  // this warp's first feature
      const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      if (S > 1) {
        // split contraction: fp32 partial to the workspace; the split of this
        // tile that arrives last adds the partials in split order
        float* part = pa.part + ((size_t)pi.tile * S + pi.split) * BN * kPM;
#pragma unroll 1
        for (int c0 = 0; ok && half == 0 && c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(tb + c0, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) part[(c0 + c) * kPM + r] = v[c];
        }
        __threadfence();
        proj_epi_bar<C::kEpiWarps>();
        if (warp == 2 && lane == 0)
          s_last = atomicAdd(&pa.counter[pi.tile], 1u) == (uint32_t)(S - 1);
        proj_epi_bar<C::kEpiWarps>();
        if (s_last && ok && half == 0) {
          __threadfence();
          const ProjOut out = proj_out(pa, pi.b, fw + lane);
          const float* p0 = pa.part + (size_t)pi.tile * S * BN * kPM;
          // 4 token columns x 8 splits of loads in flight per round; each
          // column is still summed in split order
          for (int c0 = 0; c0 < BN && t0 + c0 < pa.T; c0 += 4) {
            float sum[4];
            for (int s0 = 0; s0 < S; s0 += 8) {
              float v[8][4];
#pragma unroll
              for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  v[u][c] = s0 + u < S ? __ldcg(p0 + ((size_t)(s0 + u) * BN + c0 + c) * kPM + r)
                                       : 0.f;
#pragma unroll
              for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                  if (s0 + u == 0)
                    sum[c] = v[u][c];
                  else if (s0 + u < S)
                    sum[c] += v[u][c];
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (out.on && t0 + c0 + c < pa.T) proj_put(out, t0 + c0 + c, sum[c]);
          }
        }
        if (s_last && warp == 2 && lane == 0) pa.counter[pi.tile] = 0u;  // re-armed
      } else if (!ok) {
        // nothing to read
      } else if (BN <= 16) {  // (four epilogue warps: half is 0)
        const ProjOut out = proj_out(pa, pi.b, fw + lane);
        float v[16];
        tmem_ld16(tb, v);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (out.on && t0 + c < pa.T) proj_put(out, t0 + c, v[c]);
      } else {
        // this warp's half of the tokens, 16 at a time through shared memory:
        // lane l then writes the 8 features [8 (l % 4), +8) of tokens l / 4
        // and l / 4 + 8 of the 16, as 16 bytes each
        const int chunk = lane & 3;
        ProjOut vo;
        const bool vec = proj_vec_ok(pa, pi.b, fw + 8 * chunk, &vo);
        const int c_lo = half * (BN / 2), c_hi = c_lo + BN / 2;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi && t0 + c0 < pa.T; c0 += 16) {
          float v[16];
          tmem_ld16(tb + c0, v);
#pragma unroll
          for (int c = 0; c < 16; ++c) so[c * C::kOutPitch + lane] = v[c];
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = (lane >> 2) + 8 * i, t = t0 + c0 + c;
            if (t >= pa.T) continue;
            const float4 lo = *reinterpret_cast<const float4*>(so + c * C::kOutPitch + 8 * chunk);
            const float4 hi =
                *reinterpret_cast<const float4*>(so + c * C::kOutPitch + 8 * chunk + 4);
            const float src[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
            if (vec) {
              const long long row = proj_row(vo.map, t);
              if (row < 0) continue;
              unsigned char* p = vo.base + row * vo.ld_bytes;
              float y[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) y[e] = vo.alpha * src[e];
              if (vo.f32) {
                reinterpret_cast<float4*>(p)[0] = make_float4(y[0], y[1], y[2], y[3]);
                reinterpret_cast<float4*>(p)[1] = make_float4(y[4], y[5], y[6], y[7]);
              } else {
                *reinterpret_cast<uint4*>(p) =
                    make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]),
                               pack_bf16(y[4], y[5]), pack_bf16(y[6], y[7]));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const ProjOut o = proj_out(pa, pi.b, fw + 8 * chunk + e);
                if (o.on) proj_put(o, t, src[e]);
              }
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive1(&tempty[acc]);  // the accumulator may be reused
    }
  }
  if (pa.wait_end) pdl_wait();  // finish after the kernel before this one
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<C::kTmemCols>(tmem);
  }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 proj_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A [rows, cols] bf16 matrix with `ld` elements between rows, read in boxes of
// 64 columns x box_rows rows with the 128-byte swizzle; reads past the matrix
// return zeros.
bool proj_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
              uint32_t box_rows) {
  auto fn = proj_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kPK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int proj_bn(int T) { return T <= 16 ? 16 : T <= 64 ? 64 : T <= 128 ? 128 : 256; }
int proj_ctas_per_sm(int bn) { return bn <= 16 ? PCfg<16>::kCtasPerSm : PCfg<256>::kCtasPerSm; }

// One projection GEMM: out features [0, M) per batch, nb batches, T tokens,
// contraction K.  Returns the split count and the workspace bytes it needs
// (tile counters, then the fp32 partials).
struct ProjPlan {
  int bn, tiles, splits, k_steps;
  size_t counter_bytes, part_bytes;
  size_t bytes() const { return counter_bytes + part_bytes; }
};
ProjPlan proj_plan(int M, int T, int K, int nb) {
  ProjPlan p{};
  p.bn = proj_bn(T);
  p.k_steps = (K + kPK - 1) / kPK;
  p.tiles = nb * ((M + kPM - 1) / kPM) * ((T + p.bn - 1) / p.bn);
  // A handful of tokens (one token tile) makes the call a stream over the
  // weight rows: split the contraction until the grid fills the resident CTA
  // slots once.  With more tokens the tiles themselves fill the GPU (and the
  // query projection runs beside the hidden-state one).
  const int want = proj_ctas_per_sm(p.bn) * num_sms();
  p.splits = 1;
  if (T <= p.bn && p.tiles < want) {
    const int by_grid = want / p.tiles;
    const int by_depth = max(1, p.k_steps / 4);  // at least four stages per split
    p.splits = max(1, min(by_grid, by_depth));
  }
  p.counter_bytes = p.splits > 1 ? ((size_t)p.tiles * 4 + 255) / 256 * 256 : 0;
  p.part_bytes = p.splits > 1 ? (size_t)p.tiles * p.splits * p.bn * kPM * 4 : 0;
  return p;
}

template <int BN>
int launch_proj_bn(const CUtensorMap& mw, const CUtensorMap& mx, const ProjArgs& pa,
                   const ProjPlan& plan, int32_t* status, cudaStream_t stream) {
  using C = PCfg<BN>;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(proj_gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)C::kSmem);
  });
  cudaLaunchConfig_t cfg = {};
  const int n_items = plan.tiles * plan.splits;
  cfg.gridDim = dim3(min(n_items, C::kCtasPerSm * num_sms()), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launch_kernel(&cfg, proj_gemm_kernel<BN>, mw, mx, pa, n_items, plan.splits, status) ==
                 cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

// w: [nb * M, K] rows (batch b's rows from b * M), x: token rows of ldx
// elements whose batch-b inputs start at column b * x_col_batch.
int launch_proj(const void* w, int M, int K, int nb, const void* x, long long ldx,
                long long x_cols, int x_col_batch, int T, const ProjSeg* segs, int n_segs,
                const int32_t* row_map, void* ws, int wait_start, int wait_end, int32_t* status,
                cudaStream_t stream) {
  const ProjPlan plan = proj_plan(M, T, K, nb);
  CUtensorMap mw, mx;
  if (!proj_map(&mw, w, (uint64_t)K, (uint64_t)nb * M, (uint64_t)K, kPM)) return DSA_ERR_CUDA;
  if (!proj_map(&mx, x, (uint64_t)x_cols, (uint64_t)T, (uint64_t)ldx, plan.bn))
    return DSA_ERR_CUDA;
  ProjArgs pa{};
  for (int s = 0; s < n_segs; ++s) pa.seg[s] = segs[s];
  pa.n_segs = n_segs;
  pa.M = M;
  pa.T = T;
  pa.k_steps = plan.k_steps;
  pa.x_col_batch = x_col_batch;
  pa.row_map = row_map;
  pa.counter = plan.splits > 1 ? static_cast<uint32_t*>(ws) : nullptr;
  pa.part = plan.splits > 1
                ? reinterpret_cast<float*>(static_cast<unsigned char*>(ws) + plan.counter_bytes)
                : nullptr;
  pa.wait_start = wait_start;
  pa.wait_end = wait_end;
  switch (plan.bn) {
    case 16: return launch_proj_bn<16>(mw, mx, pa, plan, status, stream);
    case 64: return launch_proj_bn<64>(mw, mx, pa, plan, status, stream);
    case 128: return launch_proj_bn<128>(mw, mx, pa, plan, status, stream);
    default: return launch_proj_bn<256>(mw, mx, pa, plan, status, stream);
  }
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct ProjGeom {
  ProjPlan hid, qry, abs;
  size_t off_hid, off_qry, off_abs, total;
};
ProjGeom proj_geom(int T, int hidden, int q_rank, int H, int D, int Hm, int nope, int L) {
  ProjGeom g{};
  g.hid = proj_plan(2 * D + H, T, hidden, 1);
  g.qry = proj_plan(H * D + Hm * nope, T, q_rank, 1);
  g.abs = proj_plan(L, T, nope, Hm);
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  g.off_hid = 0;
  g.off_qry = up(g.hid.bytes());
  g.off_abs = g.off_qry + up(g.qry.bytes());
  g.total = g.off_abs + up(g.abs.bytes());
  return g;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_indexer_project_workspace_size(int T, int hidden, int q_rank, int H, int D,
                                                     int Hm, int nope, int L) {
  if (T <= 0 || hidden <= 0 || q_rank <= 0 || H <= 0 || D <= 0 || Hm <= 0 || nope <= 0 || L <= 0)
    return 0;
  return proj_geom(T, hidden, q_rank, H, D, Hm, nope, L).total;
}

extern "C" int dsa_indexer_project(const void* x, const void* w_kgw, const void* cq,
                                   const void* w_q, const void* w_uk_t, int T, int hidden,
                                   int q_rank, int H, int D, int Hm, int nope, int L,
                                   float weights_scale, const int32_t* kv_rows, void* k_out,
                                   void* gate_out, float* weights_out, void* q_out,
                                   void* q_nope_out, void* q_lat_out, void* workspace,
                                   size_t ws_bytes, int32_t* status_dev, void* stream) {
  if (T < 0 || hidden < 1 || q_rank < 1 || H < 1 || D < 1 || Hm < 1 || nope < 1 || L < 1)
    return DSA_ERR_INVALID_ARG;
  if (!std::isfinite(weights_scale)) return DSA_ERR_INVALID_ARG;
  // TMA row strides are multiples of 16 bytes; a head's no-rope slice is a
  // whole number of 64-element stages (the stages of one head never reach
  // into the next head's columns)
  if (hidden % 8 || q_rank % 8 || nope % kPK) return DSA_ERR_UNSUPPORTED;
  if ((long long)2 * D + H > (1 << 30) || (long long)H * D + (long long)Hm * nope > (1 << 30) ||
      (long long)Hm * L > (1 << 30))
    return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!x || !w_kgw || !cq || !w_q || !w_uk_t || !k_out || !gate_out || !weights_out || !q_out ||
      !q_nope_out || !q_lat_out)
    return DSA_ERR_INVALID_ARG;
  if (!al16(x) || !al16(w_kgw) || !al16(cq) || !al16(w_q) || !al16(w_uk_t) || !al16(q_nope_out) ||
      (reinterpret_cast<uintptr_t>(k_out) & 1) || (reinterpret_cast<uintptr_t>(gate_out) & 1) ||
      (reinterpret_cast<uintptr_t>(q_out) & 1) || (reinterpret_cast<uintptr_t>(q_lat_out) & 1) ||
      (reinterpret_cast<uintptr_t>(weights_out) & 3) ||
      (kv_rows && (reinterpret_cast<uintptr_t>(kv_rows) & 3)) ||
      (status_dev && (reinterpret_cast<uintptr_t>(status_dev) & 3)))
    return DSA_ERR_MISALIGNED;
  const ProjGeom g = proj_geom(T, hidden, q_rank, H, D, Hm, nope, L);
  if (g.total > 0 && (!workspace || ws_bytes < g.total)) return DSA_ERR_WORKSPACE;
  if (workspace && !al16(workspace)) return DSA_ERR_MISALIGNED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);

  // 1. hidden -> k | gate | weights (k and gate to the cache rows kv_rows)
  const int use_map = kv_rows ? 1 : 0;
  ProjSeg sh[3] = {
      {k_out, D, 0, 0, D, 0, use_map, 1.f},
      {gate_out, D, 0, D, 2 * D, 0, use_map, 1.f},
      {weights_out, H, 0, 2 * D, 2 * D + H, 1, 0, weights_scale},
  };
  int r = launch_proj(w_kgw, 2 * D + H, hidden, 1, x, hidden, hidden, 0, T, sh, 3, kv_rows,
                      ws ? ws + g.off_hid : nullptr, 2, 0, status_dev, st);
  if (r != DSA_OK) return r;
  // 2. query latent -> indexer query | MLA no-rope query; it reads only the
  // call's inputs, so it runs beside the first and finishes after it
  ProjSeg sq[2] = {
      {q_out, (long long)H * D, 0, 0, H * D, 0, 0, 1.f},
      {q_nope_out, (long long)Hm * nope, 0, H * D, H * D + Hm * nope, 0, 0, 1.f},
  };
  r = launch_proj(w_q, H * D + Hm * nope, q_rank, 1, cq, q_rank, q_rank, 0, T, sq, 2, nullptr,
                  ws ? ws + g.off_qry : nullptr, 0, 1, status_dev, st);
  if (r != DSA_OK) return r;
  // 3. per MLA head: the no-rope query through the transposed key
  // up-projection, into latent space
  ProjSeg sa[1] = {{q_lat_out, (long long)Hm * L, L, 0, L, 0, 0, 1.f}};
  return launch_proj(w_uk_t, L, nope, Hm, q_nope_out, (long long)Hm * nope, (long long)Hm * nope,
                     nope, T, sa, 1, nullptr, ws ? ws + g.off_abs : nullptr, 2, 0, status_dev, st);
}
