// Grouped GEMM on the CUDA cores in plain fp32 (no TF32), for the fp32 layer
// (the expert FFNs, forward and backward) and for the router's gradient GEMMs,
// which stay in fp32 for every layer dtype ("Mixture of Experts (MoE) を1から
// 解説 — Switch Transformerのルーティングと負荷分散", section
// 学習を安定させる3つの工夫: the router is computed in float32).
//
// Operands are addressed through strides so one kernel serves every
// orientation: A(m, k) = A[m*sam + k*sak], B_e(n, k) = B[e*sbe + n*sbn + k*sbk],
// C(m, n) = C[e*sce + m*scm + n*scn]. Grouped-M mode runs the rows of group e
// (offsets[e] .. offsets[e+1]) against B_e; grouped-K mode sums over the rows
// of group e into C_e (weight gradients). 64 x 64 tiles, 16-deep k slices,
// 4 x 4 outputs per thread.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

struct SimtArgs {
  const void *A, *B;
  void *C, *C2;
  const void *aux;
  int64_t sam, sak, sbe, sbn, sbk, scm, scn, sce, sc2m, saux;
  int M, N, K, F;
  const int32_t *offsets;  // nullptr: one group covering all rows
  int groups;
};

constexpr int TM = 64, TN = 64, TK = 16;

template <typename T>
__device__ __forceinline__ float ld(const void *p, int64_t i) {
  return to_f32<T>(reinterpret_cast<const T *>(p)[i]);
}

template <typename TA, typename TB, typename TC, int GROUP_K, int EPI>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const SimtArgs a) {
  constexpr bool DUAL = (EPI == EPI_SWIGLU);
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float Bu[DUAL ? TK : 1][TN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int e = blockIdx.z;
  const int n0 = blockIdx.x * TN;
  int64_t m0, mlim, klo, khi;
  if (GROUP_K) {
    klo = a.offsets ? a.offsets[e] : 0;
    khi = a.offsets ? a.offsets[e + 1] : a.K;
    m0 = (int64_t)blockIdx.y * TM;
    mlim = a.M;
  } else {
    const int64_t rlo = a.offsets ? a.offsets[e] : 0;
    mlim = a.offsets ? a.offsets[e + 1] : a.M;
    m0 = rlo + (int64_t)blockIdx.y * TM;
    if (m0 >= mlim) return;
    klo = 0;
    khi = a.K;
  }
  const int64_t boff = GROUP_K ? 0 : (int64_t)e * a.sbe;
  const bool a_kfast = (a.sak == 1), b_kfast = (a.sbk == 1);

  float acc[4][4], accu[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = accu[i][j] = 0.0f;

  for (int64_t k0 = klo; k0 < khi; k0 += TK) {
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int i = tid + 256 * l;
      const int mm = a_kfast ? (i >> 4) : (i & 63), kk = a_kfast ? (i & 15) : (i >> 6);
      const int64_t m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < mlim && k < khi) ? ld<TA>(a.A, m * a.sam + k * a.sak) : 0.0f;
      const int nn = b_kfast ? (i >> 4) : (i & 63), kb = b_kfast ? (i & 15) : (i >> 6);
      const int64_t n = n0 + nn, kq = k0 + kb;
      const bool bv = (n < a.N && kq < khi);
      Bs[kb][nn] = bv ? ld<TB>(a.B, boff + n * a.sbn + kq * a.sbk) : 0.0f;
      if (DUAL) Bu[kb][nn] = bv ? ld<TB>(a.B, boff + (n + a.F) * a.sbn + kq * a.sbk) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4], uv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[j] = Bs[kk][tx * 4 + j];
        if (DUAL) uv[j] = Bu[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (DUAL) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
        }
    }
    __syncthreads();
  }

  TC *C = reinterpret_cast<TC *>(a.C) + (GROUP_K ? (int64_t)e * a.sce : 0);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty * 4 + i;
    if (m >= mlim) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      float v = acc[i][j];
      if (EPI == EPI_RELU) v = fmaxf(v, 0.0f);
      if (EPI == EPI_SWIGLU) {
        const float g = v, u = accu[i][j];
        v = silu_f(g) * u;
        if (a.C2) {
          TC *c2 = reinterpret_cast<TC *>(a.C2);
          c2[m * a.sc2m + n] = from_f32<TC>(g);
          c2[m * a.sc2m + a.F + n] = from_f32<TC>(u);
        }
      }
      if (EPI == EPI_RELU_BWD) v = (ld<TC>(a.aux, m * a.saux + n) > 0.0f) ? v : 0.0f;
      if (EPI == EPI_SWIGLU_BWD) {
        const float g = ld<TC>(a.aux, m * a.saux + n), u = ld<TC>(a.aux, m * a.saux + a.F + n);
        const float sg = 1.0f / (1.0f + expf(-g));
        C[m * a.scm + a.F + n] = from_f32<TC>(v * g * sg);
        v = v * u * (sg * (1.0f + g * (1.0f - sg)));
      }
      C[m * a.scm + n * a.scn] = from_f32<TC>(v);
    }
  }
}

template <typename TA, typename TB, typename TC, int GROUP_K, int EPI>
cudaError_t run(const SimtArgs &a, int64_t max_rows, cudaStream_t stream) {
  dim3 grid((a.N + TN - 1) / TN, (unsigned)((GROUP_K ? a.M : max_rows) + TM - 1) / TM, a.groups);
  if (grid.y == 0) return cudaSuccess;
  return launch_kernel(simt_gemm_kernel<TA, TB, TC, GROUP_K, EPI>, grid, dim3(256), 0, stream, a);
}

}  // namespace

cudaError_t simt_expert_forward(const Shape &sh, const void *x_perm, const int32_t *offsets, const void *w1,
                                const void *w2, void *pre_act, void *h, void *y_perm, cudaStream_t stream) {
  SimtArgs a{};
  a.offsets = offsets; a.groups = sh.E; a.F = sh.F;
  a.A = x_perm; a.sam = sh.d; a.sak = 1;
  a.B = w1; a.sbe = (int64_t)sh.R1 * sh.d; a.sbn = sh.d; a.sbk = 1;
  a.C = h; a.scm = sh.F; a.scn = 1;
  a.C2 = pre_act; a.sc2m = 2 * (int64_t)sh.F;
  a.N = sh.F; a.K = sh.d;
  cudaError_t err = sh.act == MOE_ACT_SWIGLU ? run<float, float, float, 0, EPI_SWIGLU>(a, sh.rows, stream)
                                             : run<float, float, float, 0, EPI_RELU>(a, sh.rows, stream);
  if (err != cudaSuccess) return err;
  SimtArgs b{};
  b.offsets = offsets; b.groups = sh.E; b.F = sh.F;
  b.A = h; b.sam = sh.F; b.sak = 1;
  b.B = w2; b.sbe = (int64_t)sh.d * sh.F; b.sbn = sh.F; b.sbk = 1;
  b.C = y_perm; b.scm = sh.d; b.scn = 1;
  b.N = sh.d; b.K = sh.F;
  return run<float, float, float, 0, EPI_STORE>(b, sh.rows, stream);
}

cudaError_t simt_expert_backward(const Shape &sh, const int32_t *offsets, const void *x_perm, const void *w1,
                                 const void *w2, const void *pre_act, const void *h, const void *dyp, void *da,
                                 void *dxp, void *dw1, void *dw2, cudaStream_t stream) {
  cudaError_t err;
  {  // dH = dYp W2_e, activation backward -> dA
    SimtArgs a{};
    a.offsets = offsets; a.groups = sh.E; a.F = sh.F;
    a.A = dyp; a.sam = sh.d; a.sak = 1;
    a.B = w2; a.sbe = (int64_t)sh.d * sh.F; a.sbn = 1; a.sbk = sh.F;
    a.C = da; a.scm = sh.R1; a.scn = 1;
    a.N = sh.F; a.K = sh.d;
    if (sh.act == MOE_ACT_SWIGLU) {
      a.aux = pre_act; a.saux = 2 * (int64_t)sh.F;
      err = run<float, float, float, 0, EPI_SWIGLU_BWD>(a, sh.rows, stream);
    } else {
      a.aux = h; a.saux = sh.F;
      err = run<float, float, float, 0, EPI_RELU_BWD>(a, sh.rows, stream);
    }
    if (err != cudaSuccess) return err;
  }
  {  // dW2_e = dYp_e^T H_e
    SimtArgs a{};
    a.offsets = offsets; a.groups = sh.E;
    a.A = dyp; a.sam = 1; a.sak = sh.d;
    a.B = h; a.sbn = 1; a.sbk = sh.F;
    a.C = dw2; a.sce = (int64_t)sh.d * sh.F; a.scm = sh.F; a.scn = 1;
    a.M = sh.d; a.N = sh.F;
    err = run<float, float, float, 1, EPI_STORE>(a, 0, stream);
    if (err != cudaSuccess) return err;
  }
  {  // dXp = dA W1_e
    SimtArgs a{};
    a.offsets = offsets; a.groups = sh.E;
    a.A = da; a.sam = sh.R1; a.sak = 1;
    a.B = w1; a.sbe = (int64_t)sh.R1 * sh.d; a.sbn = 1; a.sbk = sh.d;
    a.C = dxp; a.scm = sh.d; a.scn = 1;
    a.N = sh.d; a.K = sh.R1;
    err = run<float, float, float, 0, EPI_STORE>(a, sh.rows, stream);
    if (err != cudaSuccess) return err;
  }
  {  // dW1_e = dA_e^T X_e
    SimtArgs a{};
    a.offsets = offsets; a.groups = sh.E;
    a.A = da; a.sam = 1; a.sak = sh.R1;
    a.B = x_perm; a.sbn = 1; a.sbk = sh.d;
    a.C = dw1; a.sce = (int64_t)sh.R1 * sh.d; a.scm = sh.d; a.scn = 1;
    a.M = sh.R1; a.N = sh.d;
    err = run<float, float, float, 1, EPI_STORE>(a, 0, stream);
  }
  return err;
}

// Router gradients: dW_r = dh^T x ([E, d], sum over tokens) and dXr = dh W_r ([T, d]).
cudaError_t router_weight_grads(const Shape &sh, const float *dh, const void *x, const float *w_r, float *dw_r,
                                float *dxr, cudaStream_t stream) {
  SimtArgs a{};
  a.offsets = nullptr; a.groups = 1;
  a.A = dh; a.sam = 1; a.sak = sh.E;
  a.B = x; a.sbn = 1; a.sbk = sh.d;
  a.C = dw_r; a.scm = sh.d; a.scn = 1;
  a.M = sh.E; a.N = sh.d; a.K = sh.T;
  cudaError_t err = sh.dtype == MOE_BF16 ? run<float, bf16, float, 1, EPI_STORE>(a, 0, stream)
                                         : run<float, float, float, 1, EPI_STORE>(a, 0, stream);
  if (err != cudaSuccess) return err;
  SimtArgs b{};
  b.offsets = nullptr; b.groups = 1;
  b.A = dh; b.sam = sh.E; b.sak = 1;
  b.B = w_r; b.sbn = 1; b.sbk = sh.d;
  b.C = dxr; b.scm = sh.d; b.scn = 1;
  b.M = sh.T; b.N = sh.d; b.K = sh.E;
  return run<float, float, float, 0, EPI_STORE>(b, sh.T, stream);
}

}  // namespace moe
