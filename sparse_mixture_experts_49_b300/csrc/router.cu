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
// additions. A tcgen05 kernel (128 tokens x all experts per CTA, K split
// across CTAs when there are few token tiles) writes fp32 partial logits;
// a selection kernel sums the partials in a fixed order and does softmax and
// top-k. fp32 layers use a register-tiled CUDA-core kernel instead.
//
// Selection: one warp per token, softmax in fp32 with the row maximum
// subtracted, then k rounds of a warp arg-max (descending logit, ties to the
// lower index: a max reduction over order keys of the logits, then a min
// reduction over the expert indices holding the maximum). Importance and load are summed per block in a fixed order;
// each block then adds its sums into per-expert accumulators in the
// workspace: the loads as 32-bit integers, the importance as 64-bit fixed
// point (units of 2^-32). Integer addition is associative, so the totals do
// not depend on the order in which blocks arrive and the statistics are
// bitwise reproducible. The last block to finish converts the totals, forms
// the aux loss with a fixed-shape tree and clears the accumulators.
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
        atomicAdd(&cnt[my_e[g]], 1);
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
    v = ((float)c / ((float)a.T * (float)a.k)) * (s / (float)a.T);
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

namespace rt {
constexpr int BM = 128;
constexpr int BK = 64;
template <int EP> struct Geo {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = EP * BK * 2;  // one part
  static constexpr int STAGE_BYTES = A_BYTES + 3 * B_BYTES;
  static constexpr int STAGES = EP >= 256 ? 2 : (EP >= 128 ? 3 : 4);
  static constexpr int TMEM_COLS = EP < 32 ? 32 : EP;
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
};
struct __align__(8) Bars {
  uint64_t full[4];
  uint64_t empty[4];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
struct Args {
  int T, E, kb_per_split, KB;
  float *partial;   // [splits, T, EP]
  DeviceStatus *st;
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity))
    if (global_timer_ns() - t0 > 200000000ull) break;
}

// Partial logits of 128 tokens x all experts over the CTA's K range. Warp 0
// loads (x tile once, then the hi/mid/lo parts of W_r), warp 1 issues
// 3 x 4 MMAs per 64-deep K step into one TMEM accumulator, warps 2-5 store it.
template <int EP>
__global__ void __launch_bounds__(192, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const Args a) {
  using G = Geo<EP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *tiles = smem_raw + ((1024 - (raw & 1023)) & 1023);
  Bars &b = *reinterpret_cast<Bars *>(tiles + (size_t)G::STAGES * G::STAGE_BYTES);
  volatile int *abort_flag = &b.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    for (int i = 0; i < G::STAGES; ++i) { mbar_init(&b.full[i], 1); mbar_init(&b.empty[i], 1); }
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
  const int m0 = blockIdx.x * BM;
  const int kb0 = blockIdx.y * a.kb_per_split;
  const int kb1 = min(a.KB, kb0 + a.kb_per_split);
  const int nk = max(0, kb1 - kb0);

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_x = policy_evict_first();
      const uint64_t pol_w = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_parity = 0;
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait_bounded(&b.empty[stage], phase ^ 1, abort_flag, a.st)) break;
        uint8_t *a_s = tiles + (size_t)stage * G::STAGE_BYTES;
        mbar_arrive_expect_tx(&b.full[stage], G::STAGE_BYTES);
        const int k0 = (kb0 + ks) * BK;
        tma_load_2d(a_s, &tmX, &b.full[stage], k0, m0, pol_x);
#pragma unroll
        for (int part = 0; part < 3; ++part)
          tma_load_2d(a_s + G::A_BYTES + part * G::B_BYTES, &tmW, &b.full[stage], k0, part * EP, pol_w);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == G::STAGES) { stage = 0; phase ^= 1; }
      }
      if (*abort_flag)
        for (int i = 0; i < G::STAGES; ++i)
          if (issued & (1u << i)) drain_wait(&b.full[i], (issued_parity >> i) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, EP, 0, 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int ks = 0; ks < nk; ++ks) {
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
      if (++stage == G::STAGES) { stage = 0; phase ^= 1; }
    }
    if (ok && lane == 0) tc_commit(&b.acc_full);
    __syncwarp();
    if (*abort_flag) {
      if (lane == 0) tc_commit(&b.drain);
      __syncwarp();
      drain_wait(&b.drain, 0);
    }
  } else {
    // Each warp owns 32 rows. TMEM gives a thread one row; a 32 x 33 shared
    // transpose (in the now idle stage buffers) turns that into 128-byte
    // coalesced row stores. Partial rows have stride EP (padding columns are 0).
    const int q = warp & 3;
    if (nk > 0 && mbar_wait_bounded(&b.acc_full, 0, abort_flag, a.st)) {
      tc_fence_after();
      float *tr = reinterpret_cast<float *>(tiles) + q * (32 * 33);
      float v[32];
      const int row0 = m0 + q * 32;
      float *dst = a.partial + ((int64_t)blockIdx.y * a.T + row0) * EP;
#pragma unroll 1
      for (int c = 0; c < EP / 32; ++c) {
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) tr[lane * 33 + i] = v[i];
        __syncwarp();
#pragma unroll 8
        for (int r = 0; r < 32; ++r)
          if (row0 + r < a.T) dst[(int64_t)r * EP + c * 32 + lane] = tr[r * 33 + lane];
        __syncwarp();
      }
      tc_fence_before();
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, G::TMEM_COLS);
  }
}
}  // namespace rt

// Logits = sum of the split partials in split order (+ bias), then selection
// of 32 tokens per block. Partial rows have stride EP; every thread loads its
// float4 chunks of all splits before adding, so the loads overlap.
constexpr int RT_TC = 32;  // tokens per selection block (measured: 32 beats 64 and 128; 16 is faster
                           // for 16384 tokens but slower for the 8192-token switch-base layer)
template <int EPT>
__global__ void __launch_bounds__(256) router_select_kernel(const float *partial, int splits, const RouterArgs a,
                                                            const StatsOut so) {
  constexpr int EP = 32 * EPT;
  constexpr int Q = EP / 4;              // float4 per row
  constexpr int CH = RT_TC * Q / 256;    // float4 chunks per thread
  extern __shared__ float sm[];
  float *lg = sm;                      // [RT_TC][EP + 1]
  float *impw = lg + RT_TC * (EP + 1); // [8][EP]
  int *cnt = reinterpret_cast<int *>(impw + 8 * EP);
  const int t0 = blockIdx.x * RT_TC;
  const int E = a.E;
  float4 acc[CH];
#pragma unroll
  for (int c = 0; c < CH; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < splits; ++s) {
    float4 v[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = threadIdx.x + 256 * c, tl = i / Q, e4 = i - tl * Q, t = t0 + tl;
      v[c] = (t < a.T) ? __ldcs(reinterpret_cast<const float4 *>(partial + ((int64_t)s * a.T + t) * EP) + e4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      acc[c].x += v[c].x; acc[c].y += v[c].y; acc[c].z += v[c].z; acc[c].w += v[c].w;
    }
  }
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int i = threadIdx.x + 256 * c, tl = i / Q, e = (i - tl * Q) * 4;
    const float vv[4] = {acc[c].x, acc[c].y, acc[c].z, acc[c].w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      lg[tl * (EP + 1) + e + u] = vv[u] + ((a.bias != nullptr && e + u < E) ? a.bias[e + u] : 0.0f);
  }
  for (int e = threadIdx.x; e < EP; e += 256) cnt[e] = 0;
  __syncthreads();
  select_block<EPT, RT_TC / 8>(lg, impw, cnt, a, t0);
  finish_if_last(a, so.alpha, so.importance, so.load, so.aux, so.counter);
}

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

template <int EPT>
cudaError_t run_select(const float *partial, int splits, const RouterArgs &a, const StatsOut &so, int nblk,
                       cudaStream_t stream) {
  constexpr size_t smem = select_smem_bytes<EPT, RT_TC>();
  static cudaError_t attr = set_smem(router_select_kernel<EPT>, smem);
  if (attr != cudaSuccess) return attr;
  return launch_kernel(router_select_kernel<EPT>, dim3(nblk), dim3(256), smem, stream, partial, splits, a, so);
}

template <int EP>
cudaError_t run_tc(const CUtensorMap &mx, const CUtensorMap &mw, const rt::Args &ta, int m_tiles, int splits,
                   cudaStream_t stream) {
  static cudaError_t attr = set_smem(rt::router_tc_kernel<EP>, rt::Geo<EP>::SMEM);
  if (attr != cudaSuccess) return attr;
  return launch_kernel(rt::router_tc_kernel<EP>, dim3(m_tiles, splits), dim3(192), rt::Geo<EP>::SMEM, stream, mx, mw,
                    ta);
}

int epad_of(int E) { return E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256; }

}  // namespace

int router_blocks(const Shape &sh) {
  const int per = sh.dtype == MOE_BF16 ? RT_TC : RT;
  return (sh.T + per - 1) / per;
}

RouterPlan router_plan(const Shape &sh) {
  RouterPlan p;
  p.tensor_cores = sh.dtype == MOE_BF16;
  p.ep = epad_of(sh.E);
  p.m_tiles = (sh.T + rt::BM - 1) / rt::BM;
  const int KB = (sh.d + rt::BK - 1) / rt::BK;
  int splits = kRouterTargetCtas / p.m_tiles;
  if (splits < 1) splits = 1;
  if (splits > KB) splits = KB;
  p.kb_per_split = (KB + splits - 1) / splits;
  p.splits = (KB + p.kb_per_split - 1) / p.kb_per_split;
  return p;
}

cudaError_t launch_router(const Shape &sh, const void *x, const float *w_r, const float *bias, float *probs,
                          int32_t *idx, float *gate, float *importance, int32_t *load, float *aux, void *ws,
                          cudaStream_t stream) {
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  RouterArgs a;
  a.x = x; a.w_r = w_r; a.bias = bias; a.probs = probs; a.idx = idx; a.gate = gate;
  a.acc_imp = reinterpret_cast<unsigned long long *>(w + L.router_acc);
  a.acc_load = reinterpret_cast<int32_t *>(w + L.router_acc + 8 * (size_t)sh.E);
  a.T = sh.T; a.d = sh.d; a.E = sh.E; a.k = sh.k; a.renorm = sh.renorm;
  const int nblk = router_blocks(sh);
  const RouterPlan plan = router_plan(sh);
  StatsOut so;
  so.alpha = sh.alpha; so.importance = importance; so.load = load; so.aux = aux;
  so.counter = reinterpret_cast<unsigned int *>(w + L.status + 64);
  cudaError_t e;
  if (!plan.tensor_cores) {
    if (sh.E <= 32) e = run_simt<float, 1>(a, so, nblk, stream);
    else if (sh.E <= 64) e = run_simt<float, 2>(a, so, nblk, stream);
    else if (sh.E <= 128) e = run_simt<float, 4>(a, so, nblk, stream);
    else e = run_simt<float, 8>(a, so, nblk, stream);
    return e;
  }
  bf16 *parts = reinterpret_cast<bf16 *>(w + L.router_parts);
  float *partial = reinterpret_cast<float *>(w + L.router_partial);
  const int64_t n = (int64_t)plan.ep * sh.d;
  int sgrid = (int)((n + 255) / 256);
  if (sgrid > 4 * sm_count()) sgrid = 4 * sm_count();
  e = launch_kernel(router_split_kernel, dim3(sgrid), dim3(256), 0, stream, w_r, sh.E, plan.ep, sh.d, parts);
  if (e != cudaSuccess) return e;
  CUtensorMap mx, mw;
  if (!make_map_2d(&mx, x, sh.d, sh.T, 64, 128) || !make_map_2d(&mw, parts, sh.d, 3 * plan.ep, 64, plan.ep))
    return cudaErrorInvalidValue;
  rt::Args ta;
  ta.T = sh.T; ta.E = sh.E; ta.kb_per_split = plan.kb_per_split; ta.KB = (sh.d + rt::BK - 1) / rt::BK;
  ta.partial = partial;
  ta.st = reinterpret_cast<DeviceStatus *>(w + L.status);
  switch (plan.ep) {
    case 32: e = run_tc<32>(mx, mw, ta, plan.m_tiles, plan.splits, stream); break;
    case 64: e = run_tc<64>(mx, mw, ta, plan.m_tiles, plan.splits, stream); break;
    case 128: e = run_tc<128>(mx, mw, ta, plan.m_tiles, plan.splits, stream); break;
    default: e = run_tc<256>(mx, mw, ta, plan.m_tiles, plan.splits, stream); break;
  }
  if (e != cudaSuccess) return e;
  if (sh.E <= 32) return run_select<1>(partial, plan.splits, a, so, nblk, stream);
  if (sh.E <= 64) return run_select<2>(partial, plan.splits, a, so, nblk, stream);
  if (sh.E <= 128) return run_select<4>(partial, plan.splits, a, so, nblk, stream);
  return run_select<8>(partial, plan.splits, a, so, nblk, stream);
}

}  // namespace moe
