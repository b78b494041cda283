// Combine of the MoE layer and the two token-side kernels of its backward pass.
//
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散", eq. (2): y = sum over the selected experts of p_i E_i(x); section
// エキスパートには「定員」がある: a token over capacity skips the expert and
// passes through the residual connection. The layer output is
// out = x + sum over kept (t, j) of g[t, j] * y_perm[row(t, j)], accumulated in
// fp32 and rounded once; a token with nothing kept returns x bit for bit.
// Without the residual (add_residual = 0) the sum starts from zero, and the
// backward's dX from zero instead of dY.
//
// All three kernels give one warp to a token and stream its rows with
// 16-byte vector accesses, so they run at HBM speed.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

// Rows and gates of token t's k assignments, in registers (row = -1 when dropped).
template <int KMAX>
__device__ __forceinline__ void token_rows(int t, int k, const int32_t *__restrict__ idx,
                                           const int32_t *__restrict__ slot, const int32_t *__restrict__ offsets,
                                           const float *__restrict__ gate, int (&row)[KMAX], float (&g)[KMAX]) {
  const int lane = threadIdx.x & 31;
  int r = -1;
  float gv = 0.0f;
  if (lane < k) {
    const int s = slot[(int64_t)t * k + lane];
    const int e = idx[(int64_t)t * k + lane];
    if (gate) gv = gate[(int64_t)t * k + lane];
    if (s >= 0) r = offsets[e] + s;
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    row[j] = __shfl_sync(0xffffffffu, r, j);
    g[j] = __shfl_sync(0xffffffffu, gv, j);
  }
}

template <typename XT, int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const XT *__restrict__ x, const XT *__restrict__ y_perm,
                                                      const int32_t *__restrict__ idx, const float *__restrict__ gate,
                                                      const int32_t *__restrict__ slot,
                                                      const int32_t *__restrict__ offsets, int T, int d, int k,
                                                      int residual, XT *__restrict__ out) {
  constexpr int V = Vec16<XT>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = d / V;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    int row[KMAX];
    float g[KMAX];
    token_rows<KMAX>(t, k, idx, slot, offsets, gate, row, g);
    const XT *xr = x + (int64_t)t * d;
    XT *orow = out + (int64_t)t * d;
    // NB vectors per lane per pass, all their loads issued before any is used
    constexpr int NB = KMAX <= 2 ? 4 : (KMAX <= 4 ? 2 : 1);
    for (int v0 = lane; v0 < nvec; v0 += 32 * NB) {
      uint4 raw[NB][KMAX + 1];
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const int v = v0 + 32 * q;
        if (v >= nvec) break;
        raw[q][0] = residual ? *reinterpret_cast<const uint4 *>(xr + v * V) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (row[j] >= 0) raw[q][j + 1] = *reinterpret_cast<const uint4 *>(y_perm + (int64_t)row[j] * d + v * V);
      }
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const int v = v0 + 32 * q;
        if (v >= nvec) break;
        float acc[V], y[V];
        Vec16<XT>::unpack(raw[q][0], acc);
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (row[j] < 0) continue;
          Vec16<XT>::unpack(raw[q][j + 1], y);
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(g[j], y[i], acc[i]);
        }
        Vec16<XT>::store(orow + v * V, acc);
      }
    }
  }
}

// dg[t, j] = <dY_t, y_perm[row]> and dYp[row] = g[t, j] dY_t for kept pairs; dg = 0 otherwise.
// All k rows of a 16-byte chunk are loaded before any is used.
template <typename XT, int KMAX>
__global__ void __launch_bounds__(256) combine_backward_kernel(const XT *__restrict__ dy, const XT *__restrict__ y_perm,
                                                               const int32_t *__restrict__ idx,
                                                               const float *__restrict__ gate,
                                                               const int32_t *__restrict__ slot,
                                                               const int32_t *__restrict__ offsets, int T, int d, int k,
                                                               XT *__restrict__ dyp, float *__restrict__ dg) {
  constexpr int V = Vec16<XT>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = d / V;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    int row[KMAX];
    float g[KMAX];
    token_rows<KMAX>(t, k, idx, slot, offsets, gate, row, g);
    float dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = 0.0f;
    const XT *dr = dy + (int64_t)t * d;
    for (int v = lane; v < nvec; v += 32) {
      uint4 raw[KMAX + 1];
      raw[0] = *reinterpret_cast<const uint4 *>(dr + v * V);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (row[j] >= 0) raw[j + 1] = *reinterpret_cast<const uint4 *>(y_perm + (int64_t)row[j] * d + v * V);
      float gv[V], y[V], o[V];
      Vec16<XT>::unpack(raw[0], gv);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (row[j] < 0) continue;
        Vec16<XT>::unpack(raw[j + 1], y);
        float sacc = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) {
          sacc = fmaf(gv[i], y[i], sacc);
          o[i] = g[j] * gv[i];
        }
        dot[j] += sacc;
        Vec16<XT>::store(dyp + (int64_t)row[j] * d + v * V, o);
      }
    }
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      float sacc = dot[j];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, o);
      if (lane == j && row[j] >= 0) mine = sacc;
    }
    if (lane < k) dg[(int64_t)t * k + lane] = mine;
  }
}

// dX_t = dY_t + sum over kept rows of dXp[row] + dXr_t (router path, fp32), rounded once; all k
// rows of a chunk are loaded before the sum.
template <typename XT, int KMAX>
__global__ void __launch_bounds__(256) unpermute_kernel(const XT *__restrict__ dy, const XT *__restrict__ dxp,
                                                        const float *__restrict__ dxr, const int32_t *__restrict__ idx,
                                                        const int32_t *__restrict__ slot,
                                                        const int32_t *__restrict__ offsets, int T, int d, int k,
                                                        int residual, XT *__restrict__ dx) {
  constexpr int V = Vec16<XT>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = d / V;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    int row[KMAX];
    float g[KMAX];
    token_rows<KMAX>(t, k, idx, slot, offsets, nullptr, row, g);
    for (int v = lane; v < nvec; v += 32) {
      uint4 raw[KMAX + 1];
      raw[0] = residual ? *reinterpret_cast<const uint4 *>(dy + (int64_t)t * d + v * V) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (row[j] >= 0) raw[j + 1] = *reinterpret_cast<const uint4 *>(dxp + (int64_t)row[j] * d + v * V);
      float r[V];
      Vec16<float>::load(dxr + (int64_t)t * d + v * V, r);
      if (V == 8) Vec16<float>::load(dxr + (int64_t)t * d + v * V + 4, r + 4);
      float acc[V], y[V];
      Vec16<XT>::unpack(raw[0], acc);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (row[j] < 0) continue;
        Vec16<XT>::unpack(raw[j + 1], y);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += y[i];
      }
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += r[i];
      Vec16<XT>::store(dx + (int64_t)t * d + v * V, acc);
    }
  }
}

int token_grid(int T) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  int grid = (T + 7) / 8;
  return grid > sms * 8 ? sms * 8 : grid;
}

}  // namespace

template <typename XT, int KMAX>
cudaError_t run_combine(const Shape &sh, const void *x, const void *y_perm, const int32_t *idx, const float *gate,
                        const int32_t *slot, const int32_t *offsets, void *out, cudaStream_t stream) {
  return launch_kernel(combine_kernel<XT, KMAX>, dim3(token_grid(sh.T)), dim3(256), 0, stream, (const XT *)x,
                    (const XT *)y_perm, idx, gate, slot, offsets, sh.T, sh.d, sh.k, sh.residual, (XT *)out);
}

template <typename XT>
cudaError_t run_combine_k(const Shape &sh, const void *x, const void *y_perm, const int32_t *idx, const float *gate,
                          const int32_t *slot, const int32_t *offsets, void *out, cudaStream_t stream) {
  if (sh.k == 1) return run_combine<XT, 1>(sh, x, y_perm, idx, gate, slot, offsets, out, stream);
  if (sh.k == 2) return run_combine<XT, 2>(sh, x, y_perm, idx, gate, slot, offsets, out, stream);
  if (sh.k <= 4) return run_combine<XT, 4>(sh, x, y_perm, idx, gate, slot, offsets, out, stream);
  return run_combine<XT, 8>(sh, x, y_perm, idx, gate, slot, offsets, out, stream);
}

cudaError_t launch_combine(const Shape &sh, const void *x, const void *y_perm, const int32_t *idx,
                           const float *gate, const int32_t *slot, const int32_t *offsets, void *out,
                           cudaStream_t stream) {
  if (sh.dtype == MOE_BF16) return run_combine_k<bf16>(sh, x, y_perm, idx, gate, slot, offsets, out, stream);
  return run_combine_k<float>(sh, x, y_perm, idx, gate, slot, offsets, out, stream);
}

template <typename XT, int KMAX>
cudaError_t run_combine_backward(const Shape &sh, const void *dy, const void *y_perm, const int32_t *idx,
                                 const float *gate, const int32_t *slot, const int32_t *offsets, void *dyp, float *dg,
                                 cudaStream_t stream) {
  return launch_kernel(combine_backward_kernel<XT, KMAX>, dim3(token_grid(sh.T)), dim3(256), 0, stream, (const XT *)dy,
                       (const XT *)y_perm, idx, gate, slot, offsets, sh.T, sh.d, sh.k, (XT *)dyp, dg);
}

template <typename XT>
cudaError_t run_combine_backward_k(const Shape &sh, const void *dy, const void *y_perm, const int32_t *idx,
                                   const float *gate, const int32_t *slot, const int32_t *offsets, void *dyp,
                                   float *dg, cudaStream_t stream) {
  if (sh.k == 1) return run_combine_backward<XT, 1>(sh, dy, y_perm, idx, gate, slot, offsets, dyp, dg, stream);
  if (sh.k == 2) return run_combine_backward<XT, 2>(sh, dy, y_perm, idx, gate, slot, offsets, dyp, dg, stream);
  if (sh.k <= 4) return run_combine_backward<XT, 4>(sh, dy, y_perm, idx, gate, slot, offsets, dyp, dg, stream);
  return run_combine_backward<XT, 8>(sh, dy, y_perm, idx, gate, slot, offsets, dyp, dg, stream);
}

cudaError_t launch_combine_backward(const Shape &sh, const void *dy, const void *y_perm, const int32_t *idx,
                                    const float *gate, const int32_t *slot, const int32_t *offsets, void *dyp,
                                    float *dg, cudaStream_t stream) {
  if (sh.dtype == MOE_BF16)
    return run_combine_backward_k<bf16>(sh, dy, y_perm, idx, gate, slot, offsets, dyp, dg, stream);
  return run_combine_backward_k<float>(sh, dy, y_perm, idx, gate, slot, offsets, dyp, dg, stream);
}

template <typename XT, int KMAX>
cudaError_t run_unpermute(const Shape &sh, const void *dy, const void *dxp, const float *dxr, const int32_t *idx,
                          const int32_t *slot, const int32_t *offsets, void *dx, cudaStream_t stream) {
  return launch_kernel(unpermute_kernel<XT, KMAX>, dim3(token_grid(sh.T)), dim3(256), 0, stream, (const XT *)dy,
                       (const XT *)dxp, dxr, idx, slot, offsets, sh.T, sh.d, sh.k, sh.residual, (XT *)dx);
}

template <typename XT>
cudaError_t run_unpermute_k(const Shape &sh, const void *dy, const void *dxp, const float *dxr, const int32_t *idx,
                            const int32_t *slot, const int32_t *offsets, void *dx, cudaStream_t stream) {
  if (sh.k == 1) return run_unpermute<XT, 1>(sh, dy, dxp, dxr, idx, slot, offsets, dx, stream);
  if (sh.k == 2) return run_unpermute<XT, 2>(sh, dy, dxp, dxr, idx, slot, offsets, dx, stream);
  if (sh.k <= 4) return run_unpermute<XT, 4>(sh, dy, dxp, dxr, idx, slot, offsets, dx, stream);
  return run_unpermute<XT, 8>(sh, dy, dxp, dxr, idx, slot, offsets, dx, stream);
}

cudaError_t launch_unpermute(const Shape &sh, const void *dy, const void *dxp, const float *dxr,
                             const int32_t *idx, const int32_t *slot, const int32_t *offsets, void *dx,
                             cudaStream_t stream) {
  if (sh.dtype == MOE_BF16) return run_unpermute_k<bf16>(sh, dy, dxp, dxr, idx, slot, offsets, dx, stream);
  return run_unpermute_k<float>(sh, dy, dxp, dxr, idx, slot, offsets, dx, stream);
}

}  // namespace moe
