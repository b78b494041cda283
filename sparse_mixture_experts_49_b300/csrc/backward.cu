// Router part of the backward pass: gradient at the router logits, then the
// two GEMMs for dW_r and the router's contribution to dX. For bf16 layers the
// GEMMs run on the tensor cores from exact bf16 parts of dh and W_r (a value
// v in fp32 is h1 + h2 + h3 with h1 = bf16(v), h2 = bf16(v - h1),
// h3 = bf16(v - h1 - h2), every subtraction exact), so the products keep
// fp32 accuracy; fp32 layers use the CUDA-core fp32 GEMM.
//
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散": eq. (2) multiplies each selected expert's output by p_i, which is how
// the router receives a gradient; eq. (4) adds alpha N sum_i f_i P_i, where f
// comes from the argmax (no gradient) and P_i = mean_t p_i (gradient
// alpha N f_i / T on every p_{t,i}); eq. (1) is the softmax whose Jacobian
// maps dp to dh = p * (dp - <p, dp>). With the router variants' elementwise
// scores ([Wiki] "Mixture-of-Experts", section 横断的知見) dh = s'(h) dp.
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {

cudaError_t router_weight_grads(const Shape &sh, const float *dh, const void *x, const float *w_r, float *dw_r,
                                float *dxr, cudaStream_t stream);

namespace {

// Exact split of an fp32 value into three bf16 parts.
struct Parts3 {
  bf16 h[3];
};
__device__ __forceinline__ Parts3 split3(float v) {
  Parts3 q;
  q.h[0] = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(q.h[0]);
  q.h[1] = __float2bfloat16_rn(r1);
  q.h[2] = __float2bfloat16_rn(r1 - __bfloat162float(q.h[1]));
  return q;
}

// Which part of dh (A) and of W_r (B) each of the six EP-wide K blocks of the
// dX_r GEMM pairs: (1,1) (1,2) (2,1) (1,3) (2,2) (3,1). Blocks 3..5 are
// h1, h2, h3 in order, which the dW_r GEMM reads as its A operand.
__constant__ int kPartA[6] = {0, 0, 1, 0, 1, 2};
__constant__ int kPartB[6] = {0, 1, 0, 2, 1, 0};

// Warp per token; lane holds experts lane, lane + 32, ... When a6 is given
// (bf16 layers) the row of dh is also written as the six part blocks
// a6[t, b * EP + e] (zero for e >= E), offs2 = {0, T} and the bounds of the
// G token ranges of the dW_r split (multiples of 64 rows).
template <int EPT>
__global__ void __launch_bounds__(256) router_dh_kernel(const float *probs, const int32_t *idx, const float *gate,
                                                        const int32_t *load, const float *dg, int T, int E, int k,
                                                        int renorm, float alpha, int score, int k_route, float *dh,
                                                        bf16 *a6, int EP, int32_t *offs2, int G) {
  if (a6 && blockIdx.x == 0) {
    if (threadIdx.x < 2) offs2[threadIdx.x] = threadIdx.x ? T : 0;
    if (threadIdx.x <= G) {
      const int64_t b = ((int64_t)threadIdx.x * T / G + 63) / 64 * 64;
      offs2[2 + threadIdx.x] = (int32_t)(b < T ? b : T);
    }
  }
  const int lane = threadIdx.x & 31;
  // alpha E f_e / T = this * load_e (f counts the k_route routing columns: 1 with rerouting)
  const float aux_scale = alpha * (float)E / ((float)T * (float)T * (float)k_route);
  float base[EPT];
#pragma unroll
  for (int j = 0; j < EPT; ++j) {
    const int e = lane + 32 * j;
    base[j] = (e < E) ? aux_scale * (float)load[e] : 0.0f;
  }
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    // per selected slot: (expert, dg, gate) held by lanes < k
    int se = -1;
    float sdg = 0.0f, sg = 0.0f, sp = 0.0f;
    if (lane < k) {
      se = idx[(int64_t)t * k + lane];
      if (se >= 0 && se < E) {
        sdg = dg[(int64_t)t * k + lane];
        sg = gate[(int64_t)t * k + lane];
        sp = probs[(int64_t)t * E + se];
      } else {
        se = -1;  // an index the dispatch rejected: no gradient flows through it
      }
    }
    float S = 0.0f, corr = 0.0f;
    if (renorm) {
      for (int j = 0; j < k; ++j) {
        S += __shfl_sync(0xffffffffu, sp, j);
        corr += __shfl_sync(0xffffffffu, sdg, j) * __shfl_sync(0xffffffffu, sg, j);
      }
    }
    float p[EPT], dp[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      p[j] = (e < E) ? probs[(int64_t)t * E + e] : 0.0f;
      dp[j] = base[j];
    }
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, se, j);
      const float g = __shfl_sync(0xffffffffu, sdg, j);
      const float add = renorm ? (g - corr) / S : g;
#pragma unroll
      for (int q = 0; q < EPT; ++q)
        if (lane + 32 * q == ej) dp[q] += add;
    }
    float s = 0.0f;
    if (score == MOE_SCORE_SOFTMAX) {
#pragma unroll
      for (int j = 0; j < EPT; ++j) s = fmaf(p[j], dp[j], s);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    }
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      float v;
      if (score == MOE_SCORE_SOFTMAX) {
        v = p[j] * (dp[j] - s);                       // softmax Jacobian
      } else if (score == MOE_SCORE_SIGMOID) {
        v = p[j] * (1.0f - p[j]) * dp[j];             // sigmoid' = s (1 - s)
      } else {
        // sqrt(softplus)'(h) = sigmoid(h) / (2 s), and sigmoid(h) = 1 - exp(-softplus(h)) = 1 - exp(-s^2)
        v = p[j] > 0.0f ? (-expm1f(-p[j] * p[j])) / (2.0f * p[j]) * dp[j] : 0.0f;
      }
      if (e < E) dh[(int64_t)t * E + e] = v;
      if (a6 && e < EP) {
        const Parts3 q = split3(e < E ? v : 0.0f);
        bf16 *row = a6 + (int64_t)t * 6 * EP + e;
#pragma unroll
        for (int b = 0; b < 6; ++b) row[b * EP] = q.h[kPartA[b]];
      }
    }
  }
}

// W_r [E, d] fp32 -> b6 [6 EP, d] bf16: block b holds part kPartB[b] (rows >= E zero).
__global__ void __launch_bounds__(256) router_wsplit6_kernel(const float *w_r, int E, int EP, int d, bf16 *b6) {
  const int64_t n = (int64_t)EP * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / d);
    const Parts3 q = split3(e < E ? w_r[i] : 0.0f);
#pragma unroll
    for (int b = 0; b < 6; ++b) b6[b * n + i] = q.h[kPartB[b]];
  }
}

// dW_r[e] = sum over the G token ranges g (in order) of (h1^T x)[e] + (h2^T x)[e] + (h3^T x)[e], rows of
// c3 [G][3 EP][d].
__global__ void __launch_bounds__(256) router_dwr_sum_kernel(const float *c3, int E, int EP, int d, int G,
                                                             float *dw_r) {
  const int64_t n = (int64_t)E * d;
  const int64_t part = (int64_t)EP * d;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n / 4; i += (int64_t)gridDim.x * blockDim.x) {
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < G; ++g) {
      const float *cg = c3 + (int64_t)g * 3 * part;
      const float4 a = reinterpret_cast<const float4 *>(cg)[i];
      const float4 b = reinterpret_cast<const float4 *>(cg + part)[i];
      const float4 c = reinterpret_cast<const float4 *>(cg + 2 * part)[i];
      r.x += a.x + b.x + c.x; r.y += a.y + b.y + c.y; r.z += a.z + b.z + c.z; r.w += a.w + b.w + c.w;
    }
    reinterpret_cast<float4 *>(dw_r)[i] = r;
  }
}

int grid_for(int64_t n) {
  const int64_t g = (n + 255) / 256;
  const int cap = 4 * sm_count();
  return (int)(g < cap ? (g > 0 ? g : 1) : cap);
}

// Expert-choice routing's logit gradient (see expert_choice.cu): warp per
// token; lane holds experts lane + 32 j. A chosen (t, e) carries the gradient
// at its gate, dg_row of its row e C + (rank of t among expert e's chosen
// tokens: membership bitmap word prefix + popcount below t); dh = p (dp -
// <p, dp>) (eq. (1); no auxiliary term). Writes dh, and for bf16 layers its
// six exact part blocks and the dW_r split bounds as router_dh_kernel does.
template <int EPT>
__global__ void __launch_bounds__(256) router_dh_ec_kernel(const float *probs, const uint32_t *bm,
                                                           const int32_t *bm_prefix, const float *dg_row, int T, int E,
                                                           int Ce, float *dh, bf16 *a6, int EP, int32_t *offs2, int G) {
  if (a6 && blockIdx.x == 0) {
    if (threadIdx.x < 2) offs2[threadIdx.x] = threadIdx.x ? T : 0;
    if (threadIdx.x <= G) {
      const int64_t b = ((int64_t)threadIdx.x * T / G + 63) / 64 * 64;
      offs2[2 + threadIdx.x] = (int32_t)(b < T ? b : T);
    }
  }
  const int lane = threadIdx.x & 31;
  const int W = (T + 31) / 32;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    const int w = t >> 5;
    const uint32_t below = (1u << (t & 31)) - 1u;
    float p[EPT], dp[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      p[j] = 0.0f;
      dp[j] = 0.0f;
      if (e < E) {
        p[j] = probs[(int64_t)t * E + e];
        const uint32_t word = bm[(int64_t)e * W + w];
        if ((word >> (t & 31)) & 1u) dp[j] = dg_row[(int64_t)e * Ce + bm_prefix[(int64_t)e * W + w] + __popc(word & below)];
      }
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < EPT; ++j) s = fmaf(p[j], dp[j], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      const float v = p[j] * (dp[j] - s);
      if (e < E) dh[(int64_t)t * E + e] = v;
      if (a6 && e < EP) {
        const Parts3 q = split3(e < E ? v : 0.0f);
        bf16 *row = a6 + (int64_t)t * 6 * EP + e;
#pragma unroll
        for (int b = 0; b < 6; ++b) row[b * EP] = q.h[kPartA[b]];
      }
    }
  }
}

}  // namespace

// dW_r = dh^T x and dX_r = dh W_r from the logit gradient (and, for bf16
// layers, its part blocks and split bounds the logit-gradient kernel wrote).
static cudaError_t router_grads_from_dh(const Shape &sh, const void *x, const float *w_r, const float *dh,
                                        float *dw_r, float *dxr, void *ws, cudaStream_t stream) {
  const bool tc = sh.dtype == MOE_BF16;
  if (!tc) return router_weight_grads(sh, dh, x, w_r, dw_r, dxr, stream);
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  const int EP = router_plan(sh).ep;
  bf16 *a6 = reinterpret_cast<bf16 *>(w + L.rg_a6);
  bf16 *b6 = reinterpret_cast<bf16 *>(w + L.rg_b6);
  float *c3 = reinterpret_cast<float *>(w + L.rg_c3);
  int32_t *offs2 = reinterpret_cast<int32_t *>(w + L.rg_offs);
  const int G = router_grad_splits(sh);
  cudaError_t err = launch_kernel(router_wsplit6_kernel, dim3(grid_for((int64_t)EP * sh.d)), dim3(256), 0, stream, w_r,
                                  sh.E, EP, sh.d, b6);
  if (err != cudaSuccess) return err;
  err = tc_router_grads(sh, EP, a6, b6, x, offs2, offs2 + 2, G, dxr, c3, reinterpret_cast<DeviceStatus *>(w + L.status),
                        stream);
  if (err != cudaSuccess) return err;
  return launch_kernel(router_dwr_sum_kernel, dim3(grid_for((int64_t)sh.E * sh.d / 4)), dim3(256), 0, stream, c3, sh.E,
                       EP, sh.d, G, dw_r);
}

cudaError_t launch_router_backward_ec(const Shape &sh, const void *x, const float *w_r, const float *probs,
                                      const uint32_t *bm, const int32_t *bm_prefix, const float *dg_row, float *dh,
                                      float *dw_r, float *dxr, void *ws, cudaStream_t stream) {
  const bool tc = sh.dtype == MOE_BF16;
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  const int EP = router_plan(sh).ep;
  bf16 *a6 = tc ? reinterpret_cast<bf16 *>(w + L.rg_a6) : nullptr;
  int32_t *offs2 = reinterpret_cast<int32_t *>(w + L.rg_offs);
  const int G = tc ? router_grad_splits(sh) : 0;
  int grid = (sh.T + 7) / 8;
  if (grid > sm_count() * 8) grid = sm_count() * 8;
  const int Ce = (int)(sh.rows / sh.E);
  cudaError_t err;
#define MOE_DH_EC(EPT)                                                                                                  \
  err = launch_kernel(router_dh_ec_kernel<EPT>, dim3(grid), dim3(256), 0, stream, probs, bm, bm_prefix, dg_row, sh.T, sh.E, \
                      Ce, dh, a6, EP, offs2, G)
  if (sh.E <= 32) MOE_DH_EC(1);
  else if (sh.E <= 64) MOE_DH_EC(2);
  else if (sh.E <= 128) MOE_DH_EC(4);
  else MOE_DH_EC(8);
#undef MOE_DH_EC
  if (err != cudaSuccess) return err;
  return router_grads_from_dh(sh, x, w_r, dh, dw_r, dxr, ws, stream);
}

cudaError_t launch_router_backward(const Shape &sh, const void *x, const float *w_r, const float *probs,
                                   const int32_t *idx, const float *gate, const int32_t *load, const float *dg,
                                   float *dh, float *dw_r, float *dxr, void *ws, cudaStream_t stream) {
  const bool tc = sh.dtype == MOE_BF16;
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  const int EP = router_plan(sh).ep;
  bf16 *a6 = tc ? reinterpret_cast<bf16 *>(w + L.rg_a6) : nullptr;
  bf16 *b6 = reinterpret_cast<bf16 *>(w + L.rg_b6);
  float *c3 = reinterpret_cast<float *>(w + L.rg_c3);
  int32_t *offs2 = reinterpret_cast<int32_t *>(w + L.rg_offs);
  const int G = tc ? router_grad_splits(sh) : 0;
  int grid = (sh.T + 7) / 8;
  if (grid > sm_count() * 8) grid = sm_count() * 8;
  cudaError_t err;
#define MOE_DH(EPT)                                                                                            \
  err = launch_kernel(router_dh_kernel<EPT>, dim3(grid), dim3(256), 0, stream, probs, idx, gate, load, dg, sh.T, sh.E, \
                   sh.k, sh.renorm, sh.alpha, sh.score, sh.k_route, dh, a6, EP, offs2, G)
  if (sh.E <= 32) MOE_DH(1);
  else if (sh.E <= 64) MOE_DH(2);
  else if (sh.E <= 128) MOE_DH(4);
  else MOE_DH(8);
#undef MOE_DH
  if (err != cudaSuccess) return err;
  (void)b6;
  (void)c3;
  return router_grads_from_dh(sh, x, w_r, dh, dw_r, dxr, ws, stream);
}

}  // namespace moe
