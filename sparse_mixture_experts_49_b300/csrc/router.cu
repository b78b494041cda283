// Router of the MoE layer: fp32 logits h = W_r x (+ b), softmax over the E
// experts, top-k with gates, and the per-expert balance statistics.
//
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散": eq. (1) (softmax router), eq. (2) (gates = p of the selected experts),
// eq. (4) and its numpy sketch (f = selected fraction, P = mean probability,
// aux = alpha N sum f P), section 学習を安定させる3つの工夫 (the router runs in
// float32 even when the rest is bf16).
//
// One block handles 64 tokens against all E <= 256 experts: a register-tiled
// fp32 GEMM over d (8 tokens x E/32 experts per thread), then one warp per
// token for the softmax and the top-k (descending logit, ties to the lower
// index). Importance and load are reduced per block in a fixed order and
// finished by a second kernel, so the statistics are bitwise reproducible.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int RT = ROUTER_TOKENS;  // 64 tokens per block
constexpr int RBK = 16;            // d-slice per smem stage

struct RouterArgs {
  const void *x;
  const float *w_r;
  const float *bias;
  float *probs;
  int32_t *idx;
  float *gate;
  float *part_imp;    // [blocks, E]
  int32_t *part_load; // [blocks, E]
  int T, d, E, k, renorm;
};

template <typename XT> __device__ __forceinline__ void load4(const XT *p, float *o);
template <> __device__ __forceinline__ void load4<float>(const float *p, float *o) {
  float4 v = *reinterpret_cast<const float4 *>(p);
  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
template <> __device__ __forceinline__ void load4<bf16>(const bf16 *p, float *o) {
  uint2 u = *reinterpret_cast<const uint2 *>(p);
  o[0] = __uint_as_float(u.x << 16); o[1] = __uint_as_float(u.x & 0xFFFF0000u);
  o[2] = __uint_as_float(u.y << 16); o[3] = __uint_as_float(u.y & 0xFFFF0000u);
}

template <int EPT> constexpr size_t router_smem_bytes() {
  constexpr int EP = 32 * EPT;
  return sizeof(float) * ((size_t)RBK * RT + (size_t)RBK * EP + (size_t)RT * (EP + 1) + 8 * EP) +
         sizeof(int) * EP;
}

template <typename XT, int EPT>
__global__ void __launch_bounds__(256) router_kernel(const RouterArgs a) {
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

  // logits (+ fixed bias) to shared memory
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

  float imp[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) imp[j] = 0.0f;

  for (int i = 0; i < 8; ++i) {
    const int tl = warp * 8 + i, t = t0 + tl;
    if (t >= a.T) break;
    float h[EPT], p[EPT];
    float m = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      h[j] = (e < E) ? lg[tl * (EP + 1) + e] : -FLT_MAX;
      m = fmaxf(m, h[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.0f;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      p[j] = (e < E) ? expf(h[j] - m) : 0.0f;
      z += p[j];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float inv = 1.0f / z;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      p[j] = p[j] * inv;
      if (e < E) {
        if (a.probs) a.probs[(int64_t)t * E + e] = p[j];
        imp[j] += p[j];
      }
    }
    // top-k: k rounds of a warp arg-max over the not yet selected experts
    uint32_t taken = 0;
    int my_e = 0;
    float my_p = 0.0f, psum = 0.0f;
    for (int r = 0; r < a.k; ++r) {
      float bh = -FLT_MAX;
      int be = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const int e = lane + 32 * j;
        if (e < E && !((taken >> j) & 1u) && (h[j] > bh || (h[j] == bh && e < be))) { bh = h[j]; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, bh, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (oh > bh || (oh == bh && oe < be)) { bh = oh; be = oe; }
      }
      float pv = 0.0f;
#pragma unroll
      for (int j = 0; j < EPT; ++j)
        if (lane + 32 * j == be) { pv = p[j]; taken |= 1u << j; }
      const float pe = __shfl_sync(0xffffffffu, pv, be & 31);
      psum += pe;
      if (lane == r) { my_e = be; my_p = pe; }
    }
    if (lane < a.k) {
      a.idx[(int64_t)t * a.k + lane] = my_e;
      a.gate[(int64_t)t * a.k + lane] = a.renorm ? my_p / psum : my_p;
      atomicAdd(&cnt[my_e], 1);
    }
  }
#pragma unroll
  for (int j = 0; j < EPT; ++j) impw[warp * EP + lane + 32 * j] = imp[j];
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += impw[w * EP + e];
    a.part_imp[(int64_t)blockIdx.x * E + e] = s;
    a.part_load[(int64_t)blockIdx.x * E + e] = cnt[e];
  }
}

__global__ void __launch_bounds__(256) router_finish_kernel(const float *part_imp, const int32_t *part_load,
                                                            int nblk, int T, int E, int k, float alpha,
                                                            float *importance, int32_t *load, float *aux) {
  __shared__ float term[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = warp; e < E; e += 8) {
    float s = 0.0f;
    int c = 0;
    for (int b = lane; b < nblk; b += 32) {
      s += part_imp[(int64_t)b * E + e];
      c += part_load[(int64_t)b * E + e];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, o);
      c += __shfl_xor_sync(0xffffffffu, c, o);
    }
    if (lane == 0) {
      importance[e] = s;
      load[e] = c;
      term[e] = ((float)c / ((float)T * (float)k)) * (s / (float)T);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && aux != nullptr) {
    float acc = 0.0f;
    for (int e = 0; e < E; ++e) acc += term[e];
    *aux = alpha * (float)E * acc;
  }
}

template <typename XT, int EPT>
cudaError_t run(const RouterArgs &a, int nblk, cudaStream_t stream) {
  constexpr size_t smem = router_smem_bytes<EPT>();
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(router_kernel<XT, EPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  router_kernel<XT, EPT><<<nblk, 256, smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename XT>
cudaError_t run_dtype(const RouterArgs &a, int nblk, cudaStream_t stream) {
  if (a.E <= 32) return run<XT, 1>(a, nblk, stream);
  if (a.E <= 64) return run<XT, 2>(a, nblk, stream);
  if (a.E <= 128) return run<XT, 4>(a, nblk, stream);
  return run<XT, 8>(a, nblk, stream);
}

}  // namespace

int router_blocks(const Shape &sh) { return (sh.T + RT - 1) / RT; }

cudaError_t launch_router(const Shape &sh, const void *x, const float *w_r, const float *bias, float *probs,
                          int32_t *idx, float *gate, float *importance, int32_t *load, float *aux, void *ws,
                          cudaStream_t stream) {
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  RouterArgs a;
  a.x = x; a.w_r = w_r; a.bias = bias; a.probs = probs; a.idx = idx; a.gate = gate;
  a.part_imp = reinterpret_cast<float *>(w + L.router_imp);
  a.part_load = reinterpret_cast<int32_t *>(w + L.router_load);
  a.T = sh.T; a.d = sh.d; a.E = sh.E; a.k = sh.k; a.renorm = sh.renorm;
  const int nblk = router_blocks(sh);
  cudaError_t e = sh.dtype == MOE_BF16 ? run_dtype<bf16>(a, nblk, stream) : run_dtype<float>(a, nblk, stream);
  if (e != cudaSuccess) return e;
  router_finish_kernel<<<1, 256, 0, stream>>>(a.part_imp, a.part_load, nblk, sh.T, sh.E, sh.k, sh.alpha,
                                              importance, load, aux);
  return cudaGetLastError();
}

}  // namespace moe
