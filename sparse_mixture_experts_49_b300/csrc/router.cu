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
// into TMEM and, in its epilogue, one thread per token does softmax, top-k
// and the statistics straight from TMEM. When there are few token tiles, the
// experts' columns are split over a cluster of up to four CTAs, which swap
// only per-token records (local maximum, local sum of exponentials, top-k
// candidates) through distributed shared memory. fp32 layers use a
// register-tiled CUDA-core kernel, one warp per token for the selection.
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
  const int64_t n = (int64_t)EP * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / d);
    const float w = (e < E) ? w_r[i] : 0.0f;
    const bf16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);          // exact
    const bf16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);        // exact
    parts[i] = hi;
    parts[n + i] = mid;
    parts[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

namespace rf {
constexpr int BM = 128;        // tokens per CTA (TMEM lanes)
constexpr int BK = 64;         // K per stage (one 128-byte swizzled row of bf16)
constexpr int EPI_WARPS = 16;  // 4 per TMEM lane quarter, each on a quarter of the CTA's columns
constexpr int THREADS = 64 + 32 * EPI_WARPS;   // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-17 epilogue
constexpr int KMAX = 8;        // top-k candidates kept per row
constexpr int SMAX = 4;        // CTAs per cluster (expert-column split)
constexpr int MAX_STAGES = 8;
constexpr int SMEM_LIMIT = 232448;

template <int NC> struct Geo {
  static constexpr int A_BYTES = BM * BK * 2;      // x tile
  static constexpr int B_BYTES = NC * BK * 2;      // one bf16 part of this CTA's W_r rows
  static constexpr int STAGE_BYTES = A_BYTES + 3 * B_BYTES;
  static constexpr int TMEM_COLS = NC;             // NC >= 32, a power of two
};

// One row as one CTA of a cluster sees it (its NC expert columns): the k
// best (selection key, expert) pairs, packed so that a larger value is the
// larger key, ties to the lower expert; the score of each; the local max m
// and sum of exp(h - m) z (softmax scores).
struct Cand {
  unsigned long long c[KMAX];
  float sc[KMAX];
  float m, z;
};
struct __align__(8) Bars {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int last;          // this CTA finished last
};

struct Args {
  int T, E, EP, k, renorm, S, nk, stages, score;
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

__host__ __device__ constexpr size_t recv_bytes(int S) { return S > 1 ? (size_t)S * BM * sizeof(Cand) : 0; }
template <int NC> size_t smem_bytes(int S, int stages) {
  return 1024 + (size_t)stages * Geo<NC>::STAGE_BYTES + recv_bytes(S) + sizeof(Bars);
}

__device__ __forceinline__ unsigned long long pack_cand(float key, int e) {
  return ((unsigned long long)logit_key(key) << 32) | (unsigned)(0xFFFF - e);
}
__device__ __forceinline__ int cand_expert(unsigned long long c) { return 0xFFFF - (int)(c & 0xFFFFu); }
// Inverse of logit_key (a -0.0 key comes back as +0.0).
__device__ __forceinline__ float cand_key_value(unsigned long long c) {
  const uint32_t key = (uint32_t)(c >> 32);
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
// p = exp(h - M) / Z: the one expression both the probabilities and the gates use.
__device__ __forceinline__ float prob_of(float h, float M, float Z) { return expf(h - M) / Z; }
// The elementwise scores: sigmoid, and sqrt(softplus) with
// softplus(h) = max(h, 0) + log1p(exp(-|h|)) (no overflow for large h).
__device__ __forceinline__ float elem_score(float h, int score) {
  if (score == MOE_SCORE_SIGMOID) return 1.0f / (1.0f + expf(-h));
  return sqrtf(fmaxf(h, 0.0f) + log1pf(expf(-fabsf(h))));
}

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Named barrier of the four epilogue warps.

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity))
    if (global_timer_ns() - t0 > 200000000ull) break;
}

// A thread's candidate list in registers: the KMAX best selection keys seen
// so far, descending, with the score of each. Branch-free insertion (the
// same compare-and-swap chain for every lane, whatever its keys), so that a
// warp never splits on which of its rows took a new candidate.
struct RegList {
  unsigned long long c[KMAX];
  float s[KMAX];
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) { c[j] = 0ull; s[j] = 0.0f; }
  }
  __device__ __forceinline__ void offer(unsigned long long v, float vs, int k) {
    if (k == 1) {   // uniform over the kernel: the maximum alone
      if (v > c[0]) { c[0] = v; s[0] = vs; }
      return;
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const bool gt = v > c[j];
      const unsigned long long cj = c[j];
      const float sj = s[j];
      c[j] = gt ? v : cj;
      s[j] = gt ? vs : sj;
      v = gt ? cj : v;
      vs = gt ? sj : vs;
    }
  }
};

__device__ __forceinline__ void put_record(Cand &rc, const RegList &l, float m, float z) {
#pragma unroll
  for (int j = 0; j < KMAX; ++j) { rc.c[j] = l.c[j]; rc.sc[j] = l.s[j]; }
  rc.m = m;
  rc.z = z;
}
// This row's record into slot [rank][r] of every CTA of the cluster.
__device__ __forceinline__ void send_record(Cand *recv, int rank, int r, int S, const RegList &l, float m, float z) {
  const uint32_t mine = smem_u32(&recv[rank * BM + r]);
  for (int dst = 0; dst < S; ++dst) {
    const uint32_t ra = mapa_shared(mine, (uint32_t)dst);
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      st_cluster_u64(ra + 8u * j, l.c[j]);
      st_cluster_f32(ra + 8u * KMAX + 4u * j, l.s[j]);
    }
    st_cluster_f32(ra + 12u * KMAX, m);
    st_cluster_f32(ra + 12u * KMAX + 4u, z);
  }
}
// The k best of n sorted records recs[i * stride] (distinct experts: no equal
// keys) into l, and the softmax statistics they combine to: M = max m,
// Z = sum z exp(m - M) in record order.
__device__ __forceinline__ void merge_records(const Cand *recs, int stride, int n, int k, RegList &l, float &M,
                                              float &Z) {
  M = -FLT_MAX;
  for (int i = 0; i < n; ++i) M = fmaxf(M, recs[i * stride].m);
  Z = 0.0f;
  for (int i = 0; i < n; ++i) Z += recs[i * stride].z * expf(recs[i * stride].m - M);
  uint32_t heads = 0;   // each list's next position, 8 bits per list
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    unsigned long long best = 0ull;
    float bs = 0.0f;
    int from = 0;
    for (int i = 0; i < n; ++i) {
      const int hd = (int)((heads >> (8 * i)) & 0xFFu);
      if (j < k && hd < k) {
        const unsigned long long v = recs[i * stride].c[hd];
        if (v > best) { best = v; bs = recs[i * stride].sc[hd]; from = i; }
      }
    }
    l.c[j] = best;
    l.s[j] = bs;
    heads += 1u << (8 * from);
  }
}
// Named barrier of the sixteen epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * EPI_WARPS) : "memory"); }

// Logits, scores, top-k and statistics of 128 tokens, with the experts'
// columns split over the S CTAs of a cluster (NC = EP / S each).
//   warp 0: TMA of the x tile and of the hi/mid/lo parts of this CTA's W_r
//           rows, one 64-deep K step per stage;
//   warp 1: 3 x 4 tcgen05 MMAs (M 128, N NC, K 16) per stage into one fp32
//           TMEM accumulator;
//   warps 2-5: one token row per thread, read from TMEM. Softmax scores:
//           pass 1 the local maximum (and, without a correction bias, the
//           top-k candidates by logit), pass 2 the sum of exp(h - m); the
//           cluster's CTAs swap these per-row records over distributed shared
//           memory, each forms M = max m and Z = sum z exp(m - M) in CTA order
//           and merges the candidates. Elementwise scores: pass 1 the
//           candidates by logit (by score + bias with a correction bias) with
//           their scores. Pass 3 writes the scores of its columns (staged
//           through shared memory so each store instruction covers one
//           128-byte row piece), sums them per expert, and, for softmax scores
//           with a correction bias, forms the candidates by p + b and swaps
//           them in a second exchange. The row's experts and gates come from
//           the merged candidates (CTA `rank` writes the rows r with
//           r % S == rank).
template <int NC>
__global__ void __launch_bounds__(THREADS, 1)
    router_fused_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const Args a) {
  using G = Geo<NC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *tiles = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const int S = a.S;
  Cand *recv = reinterpret_cast<Cand *>(tiles + (size_t)a.stages * G::STAGE_BYTES);   // [S][BM]
  Bars &b = *reinterpret_cast<Bars *>(reinterpret_cast<uint8_t *>(recv) + recv_bytes(S));
  volatile int *abort_flag = &b.abort_flag;
  // Used only after this CTA's MMAs have completed, in the then idle ring:
  Cand *part_rec = reinterpret_cast<Cand *>(tiles);                          // [4 column parts][BM]
  float *stage_out = reinterpret_cast<float *>(part_rec + 4 * BM);           // [16 warps][32 rows][32]
  float *imp_w = stage_out + EPI_WARPS * 32 * 32;                            // [4 row quarters][NC]
  int *cnt = reinterpret_cast<int *>(imp_w + 4 * NC);                        // [EP]
  float *term = reinterpret_cast<float *>(cnt + 256);                        // [256]
  float2 *fin = reinterpret_cast<float2 *>(term + 256);                      // [BM] the rows' M and Z

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = S > 1 ? (int)cluster_ctarank() : 0;
  const int m0 = blockIdx.y * BM;
  const int col0 = rank * NC;
  const int E = a.E, k = a.k;
  const bool softmax = a.score == MOE_SCORE_SOFTMAX;
  // softmax scores with a correction bias choose on p + b, known only after
  // the first exchange: a second one follows pass 3
  const bool late_choice = softmax && a.sel_bias != nullptr;
  const int cluster_syncs = S > 1 ? (late_choice ? 3 : 1) : 0;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    for (int i = 0; i < a.stages; ++i) { mbar_init(&b.full[i], 1); mbar_init(&b.empty[i], 1); }
    mbar_init(&b.acc_full, 1);
    mbar_init(&b.drain, 1);
    b.abort_flag = 0;
    fence_barrier_init();
  } else if (warp == 1) {
    tmem_alloc(&b.tmem_base, G::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_parity = 0;
      for (int ks = 0; ks < a.nk; ++ks) {
        if (!mbar_wait_bounded(&b.empty[stage], phase ^ 1, abort_flag, a.st)) break;
        uint8_t *a_s = tiles + (size_t)stage * G::STAGE_BYTES;
        mbar_arrive_expect_tx(&b.full[stage], G::STAGE_BYTES);
        const int k0 = ks * BK;
        tma_load_2d(a_s, &tmX, &b.full[stage], k0, m0, pol_x);
#pragma unroll
        for (int part = 0; part < 3; ++part)
          tma_load_2d(a_s + G::A_BYTES + part * G::B_BYTES, &tmW, &b.full[stage], k0, part * a.EP + col0, pol_w);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == a.stages) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag)
        for (int i = 0; i < a.stages; ++i)
          if (issued & (1u << i)) drain_wait(&b.full[i], (issued_parity >> i) & 1);
    }
    __syncwarp();
    for (int i = 0; i < cluster_syncs; ++i) cluster_sync_all();
  } else if (warp == 1) {
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, NC, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ks = 0; ks < a.nk; ++ks) {
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
                        IDESC, (ks > 0 || part > 0 || kk > 0) ? 1u : 0u);
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
    for (int i = 0; i < cluster_syncs; ++i) cluster_sync_all();
  } else {
    // Warp w reads TMEM lane quarter q = w % 4 (rows 32 q .. 32 q + 31, one
    // per lane) and column part pp of the CTA's NC columns (CP wide).
    constexpr int CP = NC / 4;
    constexpr int SC = CP < 32 ? CP : 32;   // staging width of pass 3
    const int q = warp & 3;
    const int pp = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const int t = m0 + r;
    const bool live = t < a.T;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(pp * CP);
    const int ecol0 = col0 + pp * CP;       // this thread's first expert
    const float *bias = a.bias, *sel_bias = a.sel_bias;
    float m = -FLT_MAX, z = 0.0f;
    RegList cl;
    cl.clear();
    // warp-uniform: the TMEM loads below are warp-collective
    const bool acc_ok =
        __all_sync(0xffffffffu, mbar_wait_bounded(&b.acc_full, 0, abort_flag, a.st) ? 1 : 0) != 0;
    float v[8];
    if (acc_ok) {
      tc_fence_after();
      // pass 1: the maximum (softmax) and the candidates that need no global statistics
      if (softmax) {
#pragma unroll 1
        for (int c = 0; c < CP / 8; ++c) {
          tmem_ld8(t_row + c * 8, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = ecol0 + c * 8 + i;
            if (e < E) {
              const float h = v[i] + (bias ? __ldg(bias + e) : 0.0f);
              m = fmaxf(m, h);
              if (!late_choice) cl.offer(pack_cand(h, e), 0.0f, k);
            }
          }
        }
        // pass 2: sum of exp(h - m)
#pragma unroll 1
        for (int c = 0; c < CP / 8; ++c) {
          tmem_ld8(t_row + c * 8, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = ecol0 + c * 8 + i;
            if (e < E) z += expf(v[i] + (bias ? __ldg(bias + e) : 0.0f) - m);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < CP / 8; ++c) {
          tmem_ld8(t_row + c * 8, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int e = ecol0 + c * 8 + i;
            if (e < E) {
              const float h = v[i] + (bias ? __ldg(bias + e) : 0.0f);
              const float sv = elem_score(h, a.score);
              cl.offer(pack_cand(sel_bias ? sv + __ldg(sel_bias + e) : h, e), sv, k);
            }
          }
        }
      }
    }
    // merge the four column parts of each row (warps of part 0, one thread per row), then the cluster's CTAs
    put_record(part_rec[pp * BM + r], cl, m, z);
    epi_sync();
    float M = -FLT_MAX, Z = 0.0f;
    if (pp == 0) {
      merge_records(part_rec + r, BM, 4, k, cl, M, Z);
      if (S > 1) send_record(recv, rank, r, S, cl, M, Z);
    }
    if (S > 1) {
      cluster_sync_all();   // every CTA's records are in
      if (pp == 0) {
        RegList ml;
        float M2, Z2;
        merge_records(recv + r, BM, S, k, ml, M2, Z2);
        if (!late_choice) cl = ml;
        M = M2;
        Z = Z2;
      }
    }
    if (pp == 0) fin[r] = make_float2(M, Z);
    for (int e = threadIdx.x - 64; e < a.EP; e += 32 * EPI_WARPS) cnt[e] = 0;
    epi_sync();
    M = fin[r].x;
    Z = fin[r].y;
    if (late_choice) cl.clear();
    // pass 3: the scores of this thread's columns; per 32 x SC block, each
    // lane writes its row into the warp's 128-byte swizzled staging rows (8
    // columns at a time), then lane j < SC takes column j row by row: one
    // coalesced store of the block's row piece per row, and the column's sum
    // over the block's live rows.
    float *stg = stage_out + (warp - 2) * 32 * 32;
#pragma unroll 1
    for (int c = 0; c < CP / SC; ++c) {
#pragma unroll 1
      for (int sub = 0; sub < SC / 8; ++sub) {
        if (acc_ok) tmem_ld8(t_row + c * SC + sub * 8, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = ecol0 + c * SC + sub * 8 + i;
          float sv = 0.0f;
          if (acc_ok && live && e < E) {
            const float h = v[i] + (bias ? __ldg(bias + e) : 0.0f);
            sv = softmax ? prob_of(h, M, Z) : elem_score(h, a.score);
            if (late_choice) cl.offer(pack_cand(sv + __ldg(sel_bias + e), e), sv, k);
          }
          v[i] = sv;
        }
        *reinterpret_cast<float4 *>(stg + lane * 32 + (((2 * sub) ^ (lane & 7)) << 2)) =
            make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(stg + lane * 32 + (((2 * sub + 1) ^ (lane & 7)) << 2)) =
            make_float4(v[4], v[5], v[6], v[7]);
      }
      __syncwarp();
      if (lane < SC) {
        const int e = ecol0 + c * SC + lane;
        float colsum = 0.0f;
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
          const float pv = stg[rr * 32 + ((((lane >> 2) ^ (rr & 7))) << 2) + (lane & 3)];
          const int tt = m0 + q * 32 + rr;
          if (tt < a.T) {
            colsum += pv;
            if (a.probs && e < E) a.probs[(int64_t)tt * E + e] = pv;
          }
        }
        imp_w[q * NC + pp * CP + c * SC + lane] = colsum;
      }
      __syncwarp();
    }
    if (late_choice) {
      // softmax scores with a correction bias: the candidates by p + b, merged over the parts and the cluster
      epi_sync();   // every part's first records have been read
      put_record(part_rec[pp * BM + r], cl, M, Z);
      epi_sync();
      if (pp == 0) {
        float Mx, Zx;
        merge_records(part_rec + r, BM, 4, k, cl, Mx, Zx);
      }
      if (S > 1) {
        cluster_sync_all();   // every CTA has read the first records
        if (pp == 0) send_record(recv, rank, r, S, cl, M, Z);
        cluster_sync_all();   // the second records are in
        if (pp == 0) {
          float Mx, Zx;
          merge_records(recv + r, BM, S, k, cl, Mx, Zx);
        }
      }
    }
    // the row's experts and gates
    if (pp == 0 && acc_ok && live && (r % S) == rank) {
      float gv[KMAX];
      float psum = 0.0f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        gv[j] = 0.0f;
        if (j < k) {
          // softmax scores chosen by logit: p from the logit the key carries
          gv[j] = (softmax && !late_choice) ? prob_of(cand_key_value(cl.c[j]), M, Z) : cl.s[j];
          psum += gv[j];
        }
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k) {
          const int e = cand_expert(cl.c[j]);
          a.idx[(int64_t)t * k + j] = e;
          a.gate[(int64_t)t * k + j] = a.renorm ? gv[j] / psum : gv[j];
          if (j < a.k_route) atomicAdd(&cnt[e], 1);
        }
      }
    }
    epi_sync();
    // this CTA's per-expert sums: importance over its 128 rows (row quarters
    // in a fixed order) and loads, added as integers into the accumulators
    for (int c = threadIdx.x - 64; c < NC; c += 32 * EPI_WARPS) {
      const int e = col0 + c;
      if (e < E) {
        const float sm = imp_w[c] + imp_w[NC + c] + imp_w[2 * NC + c] + imp_w[3 * NC + c];
        // sm <= 128 rows x a score <= 1 (softmax, sigmoid) or <= 2^64 (sqrt softplus of an
        // fp32 logit): llrint of sm * 2^32 is exact to 2^-33 while sm < 2^31
        const unsigned long long qv = (unsigned long long)llrint((double)sm * 4294967296.0);
        if (qv) atomicAdd(a.acc_imp + e, qv);
      }
    }
    for (int e = threadIdx.x - 64; e < E; e += 32 * EPI_WARPS)
      if (cnt[e]) atomicAdd(a.acc_load + e, cnt[e]);
    tc_fence_before();   // this warp's TMEM loads are ordered before the release below
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

// Shared memory the epilogue uses inside the idle ring: four column parts' records, sixteen warps' staging
// blocks, the per-expert sums and counts, the aux tree and the rows' M and Z.
template <int NC> constexpr size_t epilogue_ring_bytes() {
  return 4 * rf::BM * sizeof(rf::Cand) + rf::EPI_WARPS * 32 * 32 * 4 + 4 * NC * 4 + 256 * 4 + 256 * 4 + rf::BM * 8;
}

template <int NC>
cudaError_t run_fused(const CUtensorMap &mx, const CUtensorMap &mw, const rf::Args &ra, int m_tiles,
                      cudaStream_t stream) {
  if ((size_t)ra.stages * rf::Geo<NC>::STAGE_BYTES < epilogue_ring_bytes<NC>()) return cudaErrorInvalidConfiguration;
  static cudaError_t attr = set_smem(rf::router_fused_kernel<NC>, rf::SMEM_LIMIT);
  if (attr != cudaSuccess) return attr;
  const size_t smem = rf::smem_bytes<NC>(ra.S, ra.stages);
  if (ra.S > 1)
    return launch_kernel_cluster(rf::router_fused_kernel<NC>, ra.S, dim3(ra.S, m_tiles), dim3(rf::THREADS), smem,
                                 stream, mx, mw, ra);
  return launch_kernel(rf::router_fused_kernel<NC>, dim3(1, m_tiles), dim3(rf::THREADS), smem, stream, mx, mw, ra);
}

int epad_of(int E) { return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256; }

template <int NC> int fused_stages(int S) {
  const size_t fixed = 1024 + rf::recv_bytes(S) + sizeof(rf::Bars);
  int st = (int)((rf::SMEM_LIMIT - fixed) / rf::Geo<NC>::STAGE_BYTES);
  return st > rf::MAX_STAGES ? rf::MAX_STAGES : st;
}

}  // namespace

int router_blocks(const Shape &sh) { return (sh.T + RT - 1) / RT; }

RouterPlan router_plan(const Shape &sh) {
  RouterPlan p;
  p.tensor_cores = sh.dtype == MOE_BF16;
  p.ep = epad_of(sh.E);
  p.m_tiles = (sh.T + rf::BM - 1) / rf::BM;
  // expert columns split over a cluster of S CTAs while the grid stays
  // within one wave and every CTA keeps at least 32 columns
  int S = 1;
  while (2 * S <= rf::SMAX && p.m_tiles * 2 * S <= sm_count() && p.ep / (2 * S) >= 32) S *= 2;
  p.cluster = S;
  p.nc = p.ep / S;
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
  int sgrid = (int)((n + 255) / 256);
  if (sgrid > 4 * sm_count()) sgrid = 4 * sm_count();
  e = launch_kernel(router_split_kernel, dim3(sgrid), dim3(256), 0, stream, w_r, sh.E, plan.ep, sh.d, parts);
  if (e != cudaSuccess) return e;
  CUtensorMap mx, mw;
  if (!make_map_2d(&mx, x, sh.d, sh.T, 64, rf::BM) || !make_map_2d(&mw, parts, sh.d, 3 * plan.ep, 64, plan.nc))
    return cudaErrorInvalidValue;
  rf::Args ra;
  ra.T = sh.T; ra.E = sh.E; ra.EP = plan.ep; ra.k = sh.k; ra.renorm = sh.renorm; ra.S = plan.cluster;
  ra.k_route = sh.k_route;
  ra.nk = (sh.d + rf::BK - 1) / rf::BK;
  ra.score = sh.score;
  ra.bias = bias; ra.sel_bias = sel_bias; ra.probs = probs; ra.idx = idx; ra.gate = gate;
  ra.acc_imp = acc_imp; ra.acc_load = acc_load;
  ra.alpha = sh.alpha; ra.importance = importance; ra.load = load; ra.aux = aux; ra.counter = counter;
  ra.st = reinterpret_cast<DeviceStatus *>(w + L.status);
  switch (plan.nc) {
    case 32: ra.stages = fused_stages<32>(ra.S); return run_fused<32>(mx, mw, ra, plan.m_tiles, stream);
    case 64: ra.stages = fused_stages<64>(ra.S); return run_fused<64>(mx, mw, ra, plan.m_tiles, stream);
    case 128: ra.stages = fused_stages<128>(ra.S); return run_fused<128>(mx, mw, ra, plan.m_tiles, stream);
    default: ra.stages = fused_stages<256>(ra.S); return run_fused<256>(mx, mw, ra, plan.m_tiles, stream);
  }
}

}  // namespace moe
