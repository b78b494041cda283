// Router of the MoE layer: fp32 logits h = W_r x (+ b), softmax over the E
// experts, top-k with gates, and the per-expert balance statistics.
//
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散": eq. (1) (softmax router), eq. (2) (gates = p of the selected experts),
// eq. (4) and its numpy sketch (f = selected fraction, P = mean probability,
// aux = alpha N sum f P), section 学習を安定させる3つの工夫 (the router runs in
// float32 even when the rest is bf16).
//
// bf16 layers compute the logits on the tensor cores without giving up fp32:
// W_r (fp32) is split exactly into three bf16 parts, hi + mid + lo, which
// carry its 24-bit significand; x is already bf16, so every product
// x_i * part_e,i is exact in the fp32 accumulator, and h = x W_hi^T +
// x W_mid^T + x W_lo^T is the fp32 dot product up to the order of the fp32
// additions. One fused tcgen05 kernel per 128-token tile computes the logits
// of all experts into TMEM; when there are few token tiles, d is split over a
// cluster of up to eight CTAs, which add their partial logits in distributed
// shared memory (each CTA finishes its share of the tile's rows). Softmax,
// top-k and the statistics then run one warp per token on the summed logits,
// which never leave the chip. fp32 layers use a register-tiled CUDA-core
// kernel, one warp per token for the selection.
//
// Ties in the top-k go to the lower expert index (descending logit order
// keys, then ascending index). Importance and load are summed per CTA in a
// fixed order, then added into per-expert accumulators in the workspace: the
// loads as 32-bit integers, the importance as 64-bit fixed point (units of
// 2^-32). Integer addition is associative, so the totals do not depend on
// the order in which CTAs arrive and the statistics are bitwise
// reproducible. The last CTA to finish converts the totals, forms the aux
// loss with a fixed-shape tree and clears the accumulators.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {

namespace {

constexpr int RT = ROUTER_TOKENS;  // 64 tokens per selection block
constexpr int RBK = 16;            // d-slice per smem stage of the CUDA-core GEMM

struct RouterArgs {
  const void *x;
  const float *w_r;
  const float *bias;
  float *probs;
  int32_t *idx;
  float *gate;
  unsigned long long *acc_imp;  // [E] importance in units of 2^-32
  int32_t *acc_load;             // [E]
  int T, d, E, k, renorm;
  int k_route;                   // columns the load and f count (k; 1 with rerouting)
};

template <typename XT> __device__ __forceinline__ void load4(const XT *p, float *o);
template <> __device__ __forceinline__ void load4<float>(const float *p, float *o) {
  float4 v = *reinterpret_cast<const float4 *>(p);
  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}

// Order key of a logit: a larger float gives a larger key (-0.0 counts as
// +0.0, so equal logits have equal keys); every key is above 0.
__device__ __forceinline__ uint32_t logit_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The lane's best logit among its experts lane + 32 j (j < EPT) that are
// below E and not taken: its key (0 if none) and position j. Strict
// comparison: equal keys keep the lower j, i.e. the lower expert.
template <int EPT>
__device__ __forceinline__ void lane_head(const float (&hh)[EPT], uint32_t taken, bool live, int lane, int E,
                                          uint32_t &hk, int &hj) {
  hk = 0u;
  hj = 0;
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const uint32_t key = (live && lane + 32 * j < E && !((taken >> j) & 1u)) ? logit_key(hh[j]) : 0u;
    if (key > hk) { hk = key; hj = j; }
  }
}

template <int EPT, int TOKENS> constexpr size_t select_smem_bytes() {
  constexpr int EP = 32 * EPT;
  return sizeof(float) * ((size_t)TOKENS * (EP + 1) + 8 * EP) + sizeof(int) * EP;
}
template <int EPT> constexpr size_t simt_router_smem_bytes() {
  constexpr int EP = 32 * EPT;
  return sizeof(float) * ((size_t)RBK * RT + (size_t)RBK * EP) + select_smem_bytes<EPT, RT>();
}

// Softmax, top-k and per-block statistics for the block's 8 * TPW tokens,
// whose logits (bias included) are in lg[8 * TPW][EP + 1]. Needs cnt[] zeroed
// and a __syncthreads() before the call.
template <int EPT, int TPW>
__device__ __forceinline__ void select_block(const float *lg, float *impw, int *cnt, const RouterArgs &a, int t0) {
  constexpr int EP = 32 * EPT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E;
  float imp[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) imp[j] = 0.0f;

  // G tokens of the warp at a time: their reductions are independent, so the
  // shuffles of one hide the latency of the others. Token order (and so the
  // order of the importance sums) is unchanged.
  constexpr int G = EPT >= 4 ? (TPW < 2 ? TPW : 2) : (TPW < 4 ? TPW : 4);
  static_assert(TPW % G == 0, "tokens per warp");
  for (int i0 = 0; i0 < TPW; i0 += G) {
    float h[G][EPT], p[G][EPT], m[G], z[G];
    int tt[G];
    bool live[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int tl = warp * TPW + i0 + g;
      tt[g] = t0 + tl;
      live[g] = tt[g] < a.T;
      m[g] = -FLT_MAX;
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int e = lane + 32 * j;
        h[g][j] = (live[g] && e < E) ? lg[tl * (EP + 1) + e] : -FLT_MAX;
        m[g] = fmaxf(m[g], h[g][j]);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) m[g] = fmaxf(m[g], __shfl_xor_sync(0xffffffffu, m[g], o));
#pragma unroll
    for (int g = 0; g < G; ++g) {
      z[g] = 0.0f;
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int e = lane + 32 * j;
        p[g][j] = (e < E) ? expf(h[g][j] - m[g]) : 0.0f;
        z[g] += p[g][j];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) z[g] += __shfl_xor_sync(0xffffffffu, z[g], o);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float inv = 1.0f / z[g];
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int e = lane + 32 * j;
        p[g][j] = p[g][j] * inv;
        if (live[g] && e < E) {
          if (a.probs) a.probs[(int64_t)tt[g] * E + e] = p[g][j];
          imp[j] += p[g][j];
        }
      }
    }
    // top-k: k rounds of a warp arg-max over the not yet selected experts.
    // Each lane keeps the order key of its best remaining logit (its head);
    // a round takes the largest head (one max reduction) and, among the lanes
    // holding it, the lowest expert index (one min reduction); the winning
    // lane then drops that expert and recomputes its head.
    uint32_t hk[G];   // head key (0: nothing left in this lane)
    int hj[G];        // head position j (expert lane + 32 j)
    uint32_t taken[G];
    int my_e[G];
    float my_p[G], psum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      taken[g] = 0; my_e[g] = 0; my_p[g] = 0.0f; psum[g] = 0.0f;
      lane_head<EPT>(h[g], taken[g], live[g], lane, E, hk[g], hj[g]);
    }
    for (int r = 0; r < a.k; ++r) {
      uint32_t m[G];
#pragma unroll
      for (int g = 0; g < G; ++g) m[g] = __reduce_max_sync(0xffffffffu, hk[g]);
      int be[G];
#pragma unroll
      for (int g = 0; g < G; ++g)
        be[g] = (int)__reduce_min_sync(0xffffffffu, (m[g] != 0u && hk[g] == m[g]) ? (uint32_t)(lane + 32 * hj[g])
                                                                                 : 0x7fffffffu);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float pv = 0.0f;
        if (be[g] < E && lane == (be[g] & 31)) {
#pragma unroll
          for (int j = 0; j < EPT; ++j)
            if (lane + 32 * j == be[g]) { pv = p[g][j]; taken[g] |= 1u << j; }
          lane_head<EPT>(h[g], taken[g], live[g], lane, E, hk[g], hj[g]);
        }
        const float pe = __shfl_sync(0xffffffffu, pv, be[g] & 31);
        psum[g] += pe;
        if (lane == r) { my_e[g] = be[g]; my_p[g] = pe; }
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (live[g] && lane < a.k) {
        a.idx[(int64_t)tt[g] * a.k + lane] = my_e[g];
        a.gate[(int64_t)tt[g] * a.k + lane] = a.renorm ? my_p[g] / psum[g] : my_p[g];
        if (lane < a.k_route) atomicAdd(&cnt[my_e[g]], 1);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < EPT; ++j) impw[warp * EP + lane + 32 * j] = imp[j];
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += impw[w * EP + e];
    // s <= 8 * TPW tokens, so s * 2^32 < 2^41: exact to 2^-33 in a 64-bit integer
    const unsigned long long q = (unsigned long long)llrint((double)s * 4294967296.0);
    if (q) atomicAdd(a.acc_imp + e, q);
    if (cnt[e]) atomicAdd(a.acc_load + e, cnt[e]);
  }
}

// Run by every block after it added its statistics: the last block to arrive
// converts the accumulated importance and load, sums the aux terms as a
// fixed-shape tree, and clears the accumulators and the counter for the next
// call.
__device__ __forceinline__ void finish_if_last(const RouterArgs &a, float alpha, float *importance, int32_t *load,
                                               float *aux, unsigned int *counter) {
  __shared__ bool last;
  __shared__ float term[256];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int e = threadIdx.x;
  float v = 0.0f;
  if (e < a.E) {
    const unsigned long long q = __ldcg(a.acc_imp + e);
    const int c = __ldcg(a.acc_load + e);
    const float s = (float)((double)q * (1.0 / 4294967296.0));
    a.acc_imp[e] = 0ull;
    a.acc_load[e] = 0;
    importance[e] = s;
    load[e] = c;
    v = ((float)c / ((float)a.T * (float)a.k_route)) * (s / (float)a.T);
  }
  term[e] = v;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (e < w) term[e] += term[e + w];
    __syncthreads();
  }
  if (e == 0) {
    if (aux) *aux = alpha * (float)a.E * term[0];
    *counter = 0u;
  }
}

struct StatsOut {
  float alpha;
  float *importance;
  int32_t *load;
  float *aux;
  unsigned int *counter;
};

// ---------------------------------------------------------------- CUDA-core path (fp32 layers)
template <typename XT, int EPT>
__global__ void __launch_bounds__(256) router_simt_kernel(const RouterArgs a, const StatsOut so) {
  constexpr int EP = 32 * EPT;
  extern __shared__ float sm[];
  float *xs = sm;                      // [RBK][RT]
  float *wsm = xs + RBK * RT;          // [RBK][EP]
  float *lg = wsm + RBK * EP;          // [RT][EP + 1]
  float *impw = lg + RT * (EP + 1);    // [8][EP]
  int *cnt = reinterpret_cast<int *>(impw + 8 * EP);  // [EP]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * RT;
  const XT *x = reinterpret_cast<const XT *>(a.x);
  const int d = a.d, E = a.E;

  float acc[8][EPT];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < EPT; ++j) acc[i][j] = 0.0f;

  for (int k0 = 0; k0 < d; k0 += RBK) {
    {  // x slice: 64 tokens x 16, four consecutive elements per thread
      const int tk = tid >> 2, kq = (tid & 3) * 4;
      const int t = t0 + tk;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < a.T && k0 + kq < d) load4<XT>(x + (int64_t)t * d + k0 + kq, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) xs[(kq + q) * RT + tk] = v[q];
    }
    for (int i = tid; i < EP * 4; i += 256) {  // W_r slice, transposed to [kk][e]
      const int e = i >> 2, kq = (i & 3) * 4;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (e < E && k0 + kq < d) load4<float>(a.w_r + (int64_t)e * d + k0 + kq, v);
#pragma unroll
      for (int q = 0; q < 4; ++q) wsm[(kq + q) * EP + e] = v[q];
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < RBK; ++kk) {
      float xv[8], wv[EPT];
      const float4 x0 = *reinterpret_cast<const float4 *>(xs + kk * RT + warp * 8);
      const float4 x1 = *reinterpret_cast<const float4 *>(xs + kk * RT + warp * 8 + 4);
      xv[0] = x0.x; xv[1] = x0.y; xv[2] = x0.z; xv[3] = x0.w;
      xv[4] = x1.x; xv[5] = x1.y; xv[6] = x1.z; xv[7] = x1.w;
#pragma unroll
      for (int j = 0; j < EPT; ++j) wv[j] = wsm[kk * EP + lane * EPT + j];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane * EPT + j;
      const float b = (a.bias != nullptr && e < E) ? a.bias[e] : 0.0f;
      lg[(warp * 8 + i) * (EP + 1) + e] = acc[i][j] + b;
    }
  for (int e = tid; e < EP; e += 256) cnt[e] = 0;
  __syncthreads();
  select_block<EPT, 8>(lg, impw, cnt, a, t0);
  finish_if_last(a, so.alpha, so.importance, so.load, so.aux, so.counter);
}

// ---------------------------------------------------------------- tensor-core path (bf16 layers)
// W_r [E, d] fp32 -> parts [3][EP][d] bf16 with W = hi + mid + lo (rows >= E are zero).
__global__ void __launch_bounds__(256) router_split_kernel(const float *w_r, int E, int EP, int d, bf16 *parts) {
  // four consecutive weights per step (d is a multiple of 4: the row never changes inside one)
  const uint32_t n4 = (uint32_t)EP * (uint32_t)d / 4u;
  const size_t n = (size_t)EP * d;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += gridDim.x * blockDim.x) {
    const uint32_t e = (4u * i) / (uint32_t)d;
    float4 w = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if ((int)e < E) w = __ldg(reinterpret_cast<const float4 *>(w_r) + i);
    const float wv[4] = {w.x, w.y, w.z, w.w};
    bf16 hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      hi[j] = __float2bfloat16_rn(wv[j]);
      const float r1 = wv[j] - __bfloat162float(hi[j]);   // exact
      mid[j] = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid[j]);     // exact
      lo[j] = __float2bfloat16_rn(r2);
    }
    *reinterpret_cast<uint2 *>(parts + 4 * (size_t)i) = *reinterpret_cast<const uint2 *>(hi);
    *reinterpret_cast<uint2 *>(parts + n + 4 * (size_t)i) = *reinterpret_cast<const uint2 *>(mid);
    *reinterpret_cast<uint2 *>(parts + 2 * n + 4 * (size_t)i) = *reinterpret_cast<const uint2 *>(lo);
  }
}

namespace rf {
constexpr int BM = 128;        // tokens per CTA tile (TMEM lanes)
constexpr int BK = 64;         // K per stage (one 128-byte swizzled row of bf16)
constexpr int EPI_WARPS = 16;  // 4 per TMEM lane quarter, each on a quarter of the columns
constexpr int THREADS = 64 + 32 * EPI_WARPS;   // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-17 epilogue
constexpr int SMAX = 8;        // CTAs per cluster (K split)
constexpr int MAX_STAGES = 8;
constexpr int SMEM_LIMIT = 232448;

template <int EP> struct Geo {
  static constexpr int A_BYTES = BM * BK * 2;      // x tile
  static constexpr int B_BYTES = EP * BK * 2;      // one bf16 part of W_r
  static constexpr int STAGE_BYTES = A_BYTES + 3 * B_BYTES;
  static constexpr int TMEM_COLS = EP;             // EP >= 32, a power of two
  static constexpr int EPT = EP / 32;              // columns per lane in the row pass
  // after the mainloop, inside the idle ring: the partial logits of this CTA's
  // rows from every CTA of the cluster [S][BM / S][EP] (fp32, 16-byte units of
  // each row permuted by the row's low three bits), then the outgoing partials
  // of the other CTAs' rows [S - 1][BM / S][EP]; once the rows are done, the
  // warps' per-expert sums [16][EP] and the aux tree [256] reuse the first part
  static constexpr size_t SLAB_BYTES = (size_t)BM * EP * 4;
  static size_t epi_bytes(int S) {
    const size_t slabs = SLAB_BYTES + SLAB_BYTES / S * (S - 1);
    const size_t sums = (size_t)EPI_WARPS * EP * 4 + 256 * 4;
    return slabs > sums ? slabs : sums;
  }
};

struct __align__(8) Bars {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t acc_full;
  uint64_t drain;
  uint64_t recv;     // the other CTAs' partials of this CTA's rows have landed
  uint32_t tmem_base;
  int abort_flag;
  int last;          // this CTA finished last
  uint32_t cnt2[128];  // this CTA's loads, two 16-bit counts per word (at most 128 rows x 8 each)
};

struct Args {
  int T, E, k, renorm, S, nk, stages, score;
  int k_route;                    // columns the load and f count (k; 1 with rerouting)
  const float *bias;              // [E] added to h (or null)
  const float *sel_bias;          // [E] added to the scores for the choice only (or null)
  float *probs;                   // [T, E] scores, or null
  int32_t *idx;                   // [T, k]
  float *gate;                    // [T, k]
  unsigned long long *acc_imp;    // [E] importance in units of 2^-32
  int32_t *acc_load;              // [E]
  float alpha;
  float *importance;
  int32_t *load;
  float *aux;
  unsigned int *counter;
  DeviceStatus *st;
};

template <int EP> size_t smem_bytes(int stages) {
  return 1024 + (size_t)stages * Geo<EP>::STAGE_BYTES + sizeof(Bars);
}

// Inverse of logit_key on the high word (a -0.0 key comes back as +0.0).
__device__ __forceinline__ float cand_key_value(unsigned long long c) {
  const uint32_t key = (uint32_t)(c >> 32);
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
// The elementwise scores: sigmoid, and sqrt(softplus) with
// softplus(h) = max(h, 0) + log1p(exp(-|h|)) (no overflow for large h).
__device__ __forceinline__ float elem_score(float h, int score) {
  if (score == MOE_SCORE_SIGMOID) return 1.0f / (1.0f + expf(-h));
  return sqrtf(fmaxf(h, 0.0f) + log1pf(expf(-fabsf(h))));
}

// Bulk copy of `bytes` from this CTA's shared memory to another CTA's of the
// cluster, completing on that CTA's barrier (both addresses from mapa_shared).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "r"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity))
    if (global_timer_ns() - t0 > 200000000ull) break;
}
// One compare-exchange of a descending sort: position a before b when its key
// is larger, or equal with the lower expert.
__device__ __forceinline__ void cas_desc(uint32_t &ka, float &sa, uint32_t &ea, uint32_t &kb, float &sb,
                                         uint32_t &eb) {
  const bool sw = kb > ka || (kb == ka && eb < ea);
  const uint32_t k0 = sw ? kb : ka, k1 = sw ? ka : kb;
  const float s0 = sw ? sb : sa, s1 = sw ? sa : sb;
  const uint32_t e0 = sw ? eb : ea, e1 = sw ? ea : eb;
  ka = k0; kb = k1; sa = s0; sb = s1; ea = e0; eb = e1;
}
// Sorting networks for 1, 2, 4 and 8 candidates (1, 5 and 19 exchanges).
template <int N> __device__ __forceinline__ void sort_desc(uint32_t (&k)[N], float (&s)[N], uint32_t (&e)[N]) {
#define CX(i, j) cas_desc(k[i], s[i], e[i], k[j], s[j], e[j])
  if constexpr (N == 2) {
    CX(0, 1);
  } else if constexpr (N == 4) {
    CX(0, 1); CX(2, 3); CX(0, 2); CX(1, 3); CX(1, 2);
  } else if constexpr (N == 8) {
    CX(0, 1); CX(2, 3); CX(4, 5); CX(6, 7);
    CX(0, 2); CX(1, 3); CX(4, 6); CX(5, 7);
    CX(1, 2); CX(5, 6);
    CX(0, 4); CX(1, 5); CX(2, 6); CX(3, 7);
    CX(2, 4); CX(3, 5);
    CX(1, 2); CX(3, 4); CX(5, 6);
  }
#undef CX
}
// Drops the head of a sorted list (the last position becomes empty: key 0).
template <int N> __device__ __forceinline__ void pop_front(uint32_t (&k)[N], float (&s)[N], uint32_t (&e)[N]) {
#pragma unroll
  for (int j = 0; j + 1 < N; ++j) { k[j] = k[j + 1]; s[j] = s[j + 1]; e[j] = e[j + 1]; }
  k[N - 1] = 0u;
}
// Named barrier of the sixteen epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory"); }

// Float offset of column c of slab row `row` (rows EP floats apart; the 16-byte
// units of a row permuted by the row's low three bits, so that 32 lanes
// writing 32 rows, or reading 32 columns of one row, touch every bank once
// per 128 bytes).
template <int EP> __device__ __forceinline__ int slab_at(int row, int c) {
  return row * EP + ((((c >> 2) ^ (row & 7))) << 2) + (c & 3);
}

// Logits, scores, top-k and statistics of 128 tokens. The S CTAs of a cluster
// split d (each its share of the 64-deep K steps) and every CTA's MMAs cover
// all EP expert columns, so each holds partial logits of all 128 rows; row r
// belongs to CTA r / (128 / S), which receives the other CTAs' partials of
// its rows through distributed shared memory and adds them in CTA order.
//   warp 0: TMA of the x tile and of the hi/mid/lo parts of W_r, one K step
//           per stage;
//   warp 1: 3 x 4 tcgen05 MMAs (M 128, N EP, K 16) per stage into one fp32
//           TMEM accumulator;
//   warps 2-17: drain TMEM (thread per row, a quarter of the columns per
//           warp) into the owners' shared memory; then one warp per row of
//           this CTA's rows: the row's EP values spread over the lanes, warp
//           reductions for the softmax maximum and sum, k rounds of a warp
//           maximum over selection keys for the top-k, coalesced stores of
//           the scores, per-expert sums of the scores and the loads.
template <int EP>
__global__ void __launch_bounds__(THREADS, 1)
    router_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const Args a) {
  using G = Geo<EP>;
  constexpr int EPT = G::EPT;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *tiles = smem_raw + ((1024 - (raw & 1023)) & 1023);
  Bars &b = *reinterpret_cast<Bars *>(tiles + (size_t)a.stages * G::STAGE_BYTES);
  volatile int *abort_flag = &b.abort_flag;
  // Used only after the mainloops of the cluster have completed, in the then idle ring:
  float *slab = reinterpret_cast<float *>(tiles);                               // [S][rows][EP]
  float *outgoing = reinterpret_cast<float *>(tiles + G::SLAB_BYTES);            // [S - 1][rows][EP]
  float *imp_w = slab;                                                           // [16 warps][EP], after the rows
  float *term = imp_w + EPI_WARPS * EP;                                          // [256]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int rank = S > 1 ? (int)cluster_ctarank() : 0;
  const int rows = BM / S;                       // rows of the tile this CTA finishes
  const int m0 = blockIdx.y * BM;
  const int ks0 = (rank * a.nk) / S, ks1 = ((rank + 1) * a.nk) / S;
  const int E = a.E, k = a.k;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    for (int i = 0; i < a.stages; ++i) { mbar_init(&b.full[i], 1); mbar_init(&b.empty[i], 1); }
    mbar_init(&b.acc_full, 1);
    mbar_init(&b.drain, 1);
    mbar_init(&b.recv, 1);
    // the S - 1 incoming blocks of this CTA's rows (their bytes may land before or after this)
    if (S > 1) mbar_arrive_expect_tx(&b.recv, (uint32_t)((S - 1) * (BM / S) * EP * 4));
    b.abort_flag = 0;
    fence_barrier_init();
  } else if (warp == 1) {
    tmem_alloc(&b.tmem_base, G::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  for (int i = threadIdx.x; i < 128; i += THREADS) b.cnt2[i] = 0u;
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_parity = 0;
      for (int ks = ks0; ks < ks1; ++ks) {
        if (!mbar_wait_bounded(&b.empty[stage], phase ^ 1, abort_flag, a.st)) break;
        uint8_t *a_s = tiles + (size_t)stage * G::STAGE_BYTES;
        mbar_arrive_expect_tx(&b.full[stage], G::STAGE_BYTES);
        const int k0 = ks * BK;
        tma_load_2d(a_s, &tmX, &b.full[stage], k0, m0, pol_x);
#pragma unroll
        for (int part = 0; part < 3; ++part)
          tma_load_2d(a_s + G::A_BYTES + part * G::B_BYTES, &tmW, &b.full[stage], k0, part * EP, pol_w);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == a.stages) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag)
        for (int i = 0; i < a.stages; ++i)
          if (issued & (1u << i)) drain_wait(&b.full[i], (issued_parity >> i) & 1);
    }
    __syncwarp();
    if (S > 1) cluster_sync_all();
  } else if (warp == 1) {
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, EP, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ks = ks0; ks < ks1; ++ks) {
      if (!mbar_wait_bounded(&b.full[stage], phase, abort_flag, a.st)) { ok = false; break; }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t a0 = smem_u32(tiles + (size_t)stage * G::STAGE_BYTES);
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint32_t b0 = a0 + G::A_BYTES + part * G::B_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), smem_desc_sw128(b0 + kk * 32, 16, 1024),
                        IDESC, (ks > ks0 || part > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&b.empty[stage]);
      }
      __syncwarp();
      if (++stage == a.stages) { stage = 0; phase ^= 1; }
    }
    if (ok && lane == 0) tc_commit(&b.acc_full);
    __syncwarp();
    if (*abort_flag) {
      if (lane == 0) tc_commit(&b.drain);
      __syncwarp();
      drain_wait(&b.drain, 0);
    }
    if (S > 1) cluster_sync_all();
  } else {
    const int ew = warp - 2;               // epilogue warp 0..15
    const int q = warp & 3;                // TMEM lane quarter: rows 32 q .. 32 q + 31
    const int pp = ew >> 2;                // column quarter
    constexpr int CPW = EP / 4;            // columns a warp drains
    // warp-uniform: the TMEM loads below are warp-collective
    const bool acc_ok =
        __all_sync(0xffffffffu, mbar_wait_bounded(&b.acc_full, 0, abort_flag, a.st) ? 1 : 0) != 0;
    tc_fence_after();
    if (S > 1) cluster_sync_all();         // every CTA's ring is idle: the partials may land
    // drain: row r's partials go to slot `rank` of its owner's slab, directly for this CTA's own rows, through
    // the outgoing block of the owner (sent whole below) for the other CTAs' rows
    {
      const int r = q * 32 + lane;
      const int owner = r / rows, lr = r - owner * rows;
      const int srow = owner == rank ? rank * rows + lr : (owner < rank ? owner : owner - 1) * rows + lr;
      float *dst = owner == rank ? slab : outgoing;
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(pp * CPW);
      const uint32_t base = smem_u32(dst);
      auto put4 = [&](int c, float v0, float v1, float v2, float v3) {
        const uint32_t addr = base + 4u * (uint32_t)slab_at<EP>(srow, c);
        asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v0), "f"(v1), "f"(v2), "f"(v3)
                     : "memory");
      };
      if constexpr (CPW >= 32) {
        uint32_t v[CPW / 32][32];
        if (acc_ok) {
#pragma unroll
          for (int c = 0; c < CPW / 32; ++c) tmem_ld32_issue(t_row + c * 32, v[c]);
#pragma unroll
          for (int c = 0; c < CPW / 32; ++c) tmem_wait32(v[c]);
        } else {
#pragma unroll
          for (int c = 0; c < CPW / 32; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c][i] = 0u;
        }
#pragma unroll
        for (int c = 0; c < CPW / 32; ++c)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            put4(pp * CPW + c * 32 + 4 * j, __uint_as_float(v[c][4 * j]), __uint_as_float(v[c][4 * j + 1]),
                 __uint_as_float(v[c][4 * j + 2]), __uint_as_float(v[c][4 * j + 3]));
      } else {
        float v[8];
#pragma unroll
        for (int c = 0; c < CPW / 8; ++c) {
          if (acc_ok) tmem_ld8(t_row + c * 8, v);
          else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
          }
          put4(pp * CPW + c * 8, v[0], v[1], v[2], v[3]);
          put4(pp * CPW + c * 8 + 4, v[4], v[5], v[6], v[7]);
        }
      }
    }
    tc_fence_before();                     // this warp's TMEM loads are ordered before the release below
    if (S > 1) fence_proxy_async_smem();   // the outgoing blocks are read by the copy engine
    epi_sync();
    if (S > 1) {
      if (threadIdx.x == 64) {
        const uint32_t blk = (uint32_t)(rows * EP * 4);
        for (int o = 0; o < S; ++o) {
          if (o == rank) continue;
          const int so = o < rank ? o : o - 1;
          bulk_copy_to_peer(mapa_shared(smem_u32(slab) + (uint32_t)rank * blk, (uint32_t)o),
                            smem_u32(outgoing) + (uint32_t)so * blk, blk, mapa_shared(smem_u32(&b.recv), (uint32_t)o));
        }
      }
      // every other CTA's partials of this CTA's rows
      mbar_wait_bounded<true>(&b.recv, 0, abort_flag, a.st);
    }

    // one warp per row: rows ew, ew + 16, ... of this CTA's `rows`, R at a time (independent chains of
    // reductions side by side)
    const bool softmax = a.score == MOE_SCORE_SOFTMAX;
    const bool late_choice = softmax && a.sel_bias != nullptr;
    constexpr int R = EPT >= 8 ? 1 : 2;     // (two rows of 256 columns do not fit the registers)
    constexpr float LOG2E = 1.4426950408889634f;
    float imp[EPT], bias_j[EPT], sbias_j[EPT];
    bool colv[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      imp[j] = 0.0f;
      colv[j] = e < E;
      bias_j[j] = (a.bias && colv[j]) ? __ldg(a.bias + e) : 0.0f;
      sbias_j[j] = (a.sel_bias && colv[j]) ? __ldg(a.sel_bias + e) : 0.0f;
    }
    const int swz = lane >> 2, sub = lane & 3;
#pragma unroll 1
    for (int base = ew; base < rows; base += EPI_WARPS * R) {
      float h[R][EPT], sc[R][EPT];
      uint32_t key[R][EPT], ex[R][EPT];
      bool live[R];
      int64_t tr[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int lr = base + EPI_WARPS * r;
        const int lc = lr < rows ? lr : base;                 // a row past `rows` recomputes `base`, unstored
        tr[r] = (int64_t)m0 + rank * rows + lr;
        live[r] = lr < rows && tr[r] < a.T;                   // warp-uniform
        // the S partials of this row: the same permutation in every slot (rows is a multiple of 8)
        const float *rp = slab + lc * EP + ((swz ^ (lc & 7)) << 2) + sub;
        float m = -FLT_MAX;
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          float acc = rp[32 * j];
          for (int src = 1; src < S; ++src) acc += rp[src * rows * EP + 32 * j];
          h[r][j] = acc + bias_j[j];
          if (colv[j]) m = fmaxf(m, h[r][j]);
        }
        sc[r][0] = m;   // the lane's maximum, until the softmax below
      }
      if (softmax) {
        // M: the row maximum (a warp maximum over order-preserving keys); p = 2^((h - M) log2 e) / Z with
        // Z = the lanes' sums in column order, then a butterfly (both lanes of a pair add the same two
        // values, so every lane ends with the same Z), and one correctly rounded reciprocal of Z
        float M[R], z[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
          M[r] = cand_key_value((unsigned long long)__reduce_max_sync(0xffffffffu, logit_key(sc[r][0])) << 32);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          z[r] = 0.0f;
#pragma unroll
          for (int j = 0; j < EPT; ++j) {
            sc[r][j] = colv[j] ? exp2f((h[r][j] - M[r]) * LOG2E) : 0.0f;
            z[r] += sc[r][j];
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int r = 0; r < R; ++r) z[r] += __shfl_xor_sync(0xffffffffu, z[r], o);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const float inv = __frcp_rn(z[r]);
#pragma unroll
          for (int j = 0; j < EPT; ++j) sc[r][j] *= inv;
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int j = 0; j < EPT; ++j) sc[r][j] = colv[j] ? elem_score(h[r][j], a.score) : 0.0f;
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float *prow = a.probs ? a.probs + tr[r] * E : nullptr;
#pragma unroll
        for (int j = 0; j < EPT; ++j) {
          // softmax without a correction bias chooses by logit (the same order as by p, without p's rounding)
          const float sel = late_choice || !softmax ? (a.sel_bias ? sc[r][j] + sbias_j[j] : h[r][j]) : h[r][j];
          key[r][j] = colv[j] ? logit_key(sel) : 0u;
          ex[r][j] = (uint32_t)(lane + 32 * j);
          if (live[r] && colv[j]) {
            imp[j] += sc[r][j];
            if (prow) prow[lane + 32 * j] = sc[r][j];
          }
        }
        // the lane's candidates sorted by key, descending, ties to the lower expert
        sort_desc<EPT>(key[r], sc[r], ex[r]);
      }
      // k rounds over the lanes' list heads: the largest key (one max reduction), the lowest expert holding
      // it (one min reduction); the lane that holds it moves to its next candidate
      int my_e[R];
      float my_g[R], psum[R];
#pragma unroll
      for (int r = 0; r < R; ++r) { my_e[r] = 0; my_g[r] = 0.0f; psum[r] = 0.0f; }
#pragma unroll 1
      for (int i = 0; i < k; ++i) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t wmax = __reduce_max_sync(0xffffffffu, key[r][0]);
          const uint32_t mine = (key[r][0] == wmax && wmax != 0u) ? ex[r][0] : 0xFFFFFFFFu;
          const uint32_t em = __reduce_min_sync(0xffffffffu, mine);
          // (no key left only if NaN logits emptied the lists: expert 0, gate 0, not counted)
          const bool found = wmax != 0u;
          const uint32_t e = found ? em : 0u;
          const float g = found ? __shfl_sync(0xffffffffu, sc[r][0], (int)(e & 31u)) : 0.0f;
          if (found && ex[r][0] == e) pop_front<EPT>(key[r], sc[r], ex[r]);
          psum[r] += g;
          if (lane == i) { my_e[r] = (int)e; my_g[r] = g; }
          if (lane == 0 && found && live[r] && i < a.k_route) atomicAdd(&b.cnt2[e >> 1], (e & 1u) ? 65536u : 1u);
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (live[r] && lane < k) {
          a.idx[tr[r] * k + lane] = my_e[r];
          a.gate[tr[r] * k + lane] = a.renorm ? my_g[r] / psum[r] : my_g[r];
        }
    }
    // this CTA's per-expert sums: the warps' partial sums added in warp order, as integers into the accumulators
    epi_sync();                            // every row has been read: the slab is free
#pragma unroll
    for (int j = 0; j < EPT; ++j) imp_w[ew * EP + lane + 32 * j] = imp[j];
    epi_sync();
    for (int c = threadIdx.x - 64; c < EP; c += 32 * EPI_WARPS) {
      if (c < E) {
        float sm = 0.0f;
        for (int w2 = 0; w2 < EPI_WARPS; ++w2) sm += imp_w[w2 * EP + c];
        // sm <= 128 rows x a score <= 1 (softmax, sigmoid) or <= 2^64 (sqrt softplus of an
        // fp32 logit): llrint of sm * 2^32 is exact to 2^-33 while sm < 2^31
        const unsigned long long qv = (unsigned long long)llrint((double)sm * 4294967296.0);
        if (qv) atomicAdd(a.acc_imp + c, qv);
        const int n = (int)((b.cnt2[c >> 1] >> (16 * (c & 1))) & 0xFFFFu);
        if (n) atomicAdd(a.acc_load + c, n);
      }
    }
  }

  // The last CTA to finish converts the accumulated importance and load,
  // sums the aux terms as a fixed-shape tree over 256 slots, and clears the
  // accumulators and the counter for the next call.
  {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) b.last = atomicAdd(a.counter, 1u) == gridDim.x * gridDim.y - 1;
    __syncthreads();
    if (b.last) {
      __threadfence();
      for (int e = threadIdx.x; e < 256; e += THREADS) {
        float v = 0.0f;
        if (e < E) {
          const unsigned long long qv = __ldcg(a.acc_imp + e);
          const int c = __ldcg(a.acc_load + e);
          const float sm = (float)((double)qv * (1.0 / 4294967296.0));
          a.acc_imp[e] = 0ull;
          a.acc_load[e] = 0;
          a.importance[e] = sm;
          a.load[e] = c;
          v = ((float)c / ((float)a.T * (float)a.k_route)) * (sm / (float)a.T);
        }
        term[e] = v;
      }
      __syncthreads();
      for (int w = 128; w > 0; w >>= 1) {
        for (int e = threadIdx.x; e < w; e += THREADS) term[e] += term[e + w];
        __syncthreads();
      }
      if (threadIdx.x == 0) {
        if (a.aux) *a.aux = a.alpha * (float)E * term[0];
        *a.counter = 0u;
      }
    }
  }
  __syncthreads();
  // no CTA leaves while a copy into or out of its shared memory may be in flight (every CTA has waited for
  // its incoming blocks before this point)
  if (S > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}
}  // namespace rf

template <typename K>
cudaError_t set_smem(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename XT, int EPT>
cudaError_t run_simt(const RouterArgs &a, const StatsOut &so, int nblk, cudaStream_t stream) {
  constexpr size_t smem = simt_router_smem_bytes<EPT>();
  static cudaError_t attr = set_smem(router_simt_kernel<XT, EPT>, smem);
  if (attr != cudaSuccess) return attr;
  return launch_kernel(router_simt_kernel<XT, EPT>, dim3(nblk), dim3(256), smem, stream, a, so);
}

template <int EP>
cudaError_t run_fused(const CUtensorMap &mx, const CUtensorMap &mw, const rf::Args &ra, int m_tiles,
                      cudaStream_t stream) {
  if ((size_t)ra.stages * rf::Geo<EP>::STAGE_BYTES < rf::Geo<EP>::epi_bytes(ra.S)) return cudaErrorInvalidConfiguration;
  static cudaError_t attr = set_smem(rf::router_fused_kernel<EP>, rf::SMEM_LIMIT);
  if (attr != cudaSuccess) return attr;
  const size_t smem = rf::smem_bytes<EP>(ra.stages);
  if (ra.S > 1)
    return launch_kernel_cluster(rf::router_fused_kernel<EP>, ra.S, dim3(ra.S, m_tiles), dim3(rf::THREADS), smem,
                                 stream, mx, mw, ra);
  return launch_kernel(rf::router_fused_kernel<EP>, dim3(1, m_tiles), dim3(rf::THREADS), smem, stream, mx, mw, ra);
}

int epad_of(int E) { return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256; }

template <int EP> int fused_stages() {
  const size_t fixed = 1024 + sizeof(rf::Bars);
  int st = (int)((rf::SMEM_LIMIT - fixed) / rf::Geo<EP>::STAGE_BYTES);
  return st > rf::MAX_STAGES ? rf::MAX_STAGES : st;
}

}  // namespace

int router_blocks(const Shape &sh) { return (sh.T + RT - 1) / RT; }

RouterPlan router_plan(const Shape &sh) {
  RouterPlan p;
  p.tensor_cores = sh.dtype == MOE_BF16;
  p.ep = epad_of(sh.E);
  p.m_tiles = (sh.T + rf::BM - 1) / rf::BM;
  // d split over a cluster of S CTAs while the grid stays within one wave
  // and every CTA keeps at least one 64-deep K step
  const int nk = (sh.d + rf::BK - 1) / rf::BK;
  // (for 256 expert columns the ring holds the incoming and outgoing partials of at most four CTAs)
  const int smax = p.ep == 256 ? 4 : rf::SMAX;
  int S = 1;
  while (2 * S <= smax && p.m_tiles * 2 * S <= sm_count() && 2 * S <= nk) S *= 2;
  p.cluster = S;
  return p;
}

// b_e += gamma * sign(mean(load) - load_e), decided in integers:
// sign(sum(load) - E load_e) (the mean is sum / E). One block.
__global__ void __launch_bounds__(256) select_bias_update_kernel(const int32_t *load, int E, float gamma,
                                                                 float *sel_bias) {
  __shared__ long long part[256];
  long long sum = 0;
  for (int e = threadIdx.x; e < E; e += 256) sum += load[e];
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  const long long total = part[0];
  for (int e = threadIdx.x; e < E; e += 256) {
    const long long diff = total - (long long)E * load[e];
    const float step = diff > 0 ? gamma : (diff < 0 ? -gamma : 0.0f);
    sel_bias[e] = sel_bias[e] + step;
  }
}

cudaError_t launch_select_bias_update(const Shape &sh, const int32_t *load, float gamma, float *sel_bias,
                                      cudaStream_t stream) {
  return launch_kernel(select_bias_update_kernel, dim3(1), dim3(256), 0, stream, load, sh.E, gamma, sel_bias);
}

cudaError_t launch_router(const Shape &sh, const void *x, const float *w_r, const float *bias, const float *sel_bias,
                          float *probs, int32_t *idx, float *gate, float *importance, int32_t *load, float *aux,
                          void *ws, cudaStream_t stream) {
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  unsigned long long *acc_imp = reinterpret_cast<unsigned long long *>(w + L.router_acc);
  int32_t *acc_load = reinterpret_cast<int32_t *>(w + L.router_acc + 8 * (size_t)sh.E);
  unsigned int *counter = reinterpret_cast<unsigned int *>(w + L.status + 64);
  const RouterPlan plan = router_plan(sh);
  cudaError_t e;
  if (!plan.tensor_cores) {
    RouterArgs a;
    a.x = x; a.w_r = w_r; a.bias = bias; a.probs = probs; a.idx = idx; a.gate = gate;
    a.acc_imp = acc_imp;
    a.acc_load = acc_load;
    a.T = sh.T; a.d = sh.d; a.E = sh.E; a.k = sh.k; a.renorm = sh.renorm; a.k_route = sh.k_route;
    StatsOut so;
    so.alpha = sh.alpha; so.importance = importance; so.load = load; so.aux = aux; so.counter = counter;
    const int nblk = router_blocks(sh);
    if (sh.E <= 32) e = run_simt<float, 1>(a, so, nblk, stream);
    else if (sh.E <= 64) e = run_simt<float, 2>(a, so, nblk, stream);
    else if (sh.E <= 128) e = run_simt<float, 4>(a, so, nblk, stream);
    else e = run_simt<float, 8>(a, so, nblk, stream);
    return e;
  }
  bf16 *parts = reinterpret_cast<bf16 *>(w + L.router_parts);
  const int64_t n = (int64_t)plan.ep * sh.d;
  int sgrid = (int)((n / 4 + 255) / 256);
  if (sgrid > 4 * sm_count()) sgrid = 4 * sm_count();
  e = launch_kernel(router_split_kernel, dim3(sgrid), dim3(256), 0, stream, w_r, sh.E, plan.ep, sh.d, parts);
  if (e != cudaSuccess) return e;
  CUtensorMap mx, mw;
  if (!make_map_2d(&mx, x, sh.d, sh.T, 64, rf::BM) || !make_map_2d(&mw, parts, sh.d, 3 * plan.ep, 64, plan.ep))
    return cudaErrorInvalidValue;
  rf::Args ra;
  ra.T = sh.T; ra.E = sh.E; ra.k = sh.k; ra.renorm = sh.renorm; ra.S = plan.cluster;
  ra.k_route = sh.k_route;
  ra.nk = (sh.d + rf::BK - 1) / rf::BK;
  ra.score = sh.score;
  ra.bias = bias; ra.sel_bias = sel_bias; ra.probs = probs; ra.idx = idx; ra.gate = gate;
  ra.acc_imp = acc_imp; ra.acc_load = acc_load;
  ra.alpha = sh.alpha; ra.importance = importance; ra.load = load; ra.aux = aux; ra.counter = counter;
  ra.st = reinterpret_cast<DeviceStatus *>(w + L.status);
  switch (plan.ep) {
    case 32: ra.stages = fused_stages<32>(); return run_fused<32>(mx, mw, ra, plan.m_tiles, stream);
    case 64: ra.stages = fused_stages<64>(); return run_fused<64>(mx, mw, ra, plan.m_tiles, stream);
    case 128: ra.stages = fused_stages<128>(); return run_fused<128>(mx, mw, ra, plan.m_tiles, stream);
    default: ra.stages = fused_stages<256>(); return run_fused<256>(mx, mw, ra, plan.m_tiles, stream);
  }
}

}  // namespace moe
