// Router part of the backward pass: gradient at the router logits, then the
// two fp32 GEMMs for dW_r and the router's contribution to dX.
//
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散": eq. (2) multiplies each selected expert's output by p_i, which is how
// the router receives a gradient; eq. (4) adds alpha N sum_i f_i P_i, where f
// comes from the argmax (no gradient) and P_i = mean_t p_i (gradient
// alpha N f_i / T on every p_{t,i}); eq. (1) is the softmax whose Jacobian
// maps dp to dh = p * (dp - <p, dp>).
#include "common.cuh"
#include "kernels.h"

namespace moe {

cudaError_t router_weight_grads(const Shape &sh, const float *dh, const void *x, const float *w_r, float *dw_r,
                                float *dxr, cudaStream_t stream);

namespace {

// Warp per token; lane holds experts lane, lane + 32, ...
template <int EPT>
__global__ void __launch_bounds__(256) router_dh_kernel(const float *probs, const int32_t *idx, const float *gate,
                                                        const int32_t *load, const float *dg, int T, int E, int k,
                                                        int renorm, float alpha, float *dh) {
  const int lane = threadIdx.x & 31;
  const float aux_scale = alpha * (float)E / ((float)T * (float)T * (float)k);  // alpha E f_e / T = this * load_e
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
#pragma unroll
    for (int j = 0; j < EPT; ++j) s = fmaf(p[j], dp[j], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = lane + 32 * j;
      if (e < E) dh[(int64_t)t * E + e] = p[j] * (dp[j] - s);
    }
  }
}

}  // namespace

cudaError_t launch_router_backward(const Shape &sh, const void *x, const float *w_r, const float *probs,
                                   const int32_t *idx, const float *gate, const int32_t *load, const float *dg,
                                   float *dh, float *dw_r, float *dxr, cudaStream_t stream) {
  int sms = 148;
  {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  int grid = (sh.T + 7) / 8;
  if (grid > sms * 8) grid = sms * 8;
#define MOE_DH(EPT)                                                                                         \
  router_dh_kernel<EPT><<<grid, 256, 0, stream>>>(probs, idx, gate, load, dg, sh.T, sh.E, sh.k, sh.renorm, \
                                                  sh.alpha, dh)
  if (sh.E <= 32) MOE_DH(1);
  else if (sh.E <= 64) MOE_DH(2);
  else if (sh.E <= 128) MOE_DH(4);
  else MOE_DH(8);
#undef MOE_DH
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return router_weight_grads(sh, dh, x, w_r, dw_r, dxr, stream);
}

}  // namespace moe
