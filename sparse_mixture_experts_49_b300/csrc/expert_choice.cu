// Expert-choice routing: the experts pick their tokens instead of the tokens
// picking experts ("Mixture-of-Experts" (notes.yuuk.io), section 横断的知見,
// names it among the algorithm-level routing changes; the same page's top-k
// vocabulary fixes the rest).
//
// Read with the rest of the layer: the scores are the softmax of eq. (1) of
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散", p [T, E]; expert e takes the Ce = min(C, T) tokens with the largest
// p[:, e] (descending, ties to the lower token index) and keeps them in
// ascending token order as its group of rows e Ce .. e Ce + Ce - 1; the gate
// of a chosen (t, e) is p[t, e]; out_t = x_t + sum over the experts that
// chose t of p[t, e] E_e(x_t). A token can be chosen by any number of
// experts, or by none. The expert GEMMs are the grouped GEMM with groups of
// Ce rows each.
//
// Kernels:
//   ec_select_kernel      one CTA per expert: a radix select of the Ce-th
//                         largest score key over the expert's column (4
//                         passes of 8 bits over the keys in shared memory),
//                         the ties at the threshold taken in token order, a
//                         membership bitmap of the chosen tokens (one bit
//                         per token, ballot per 32 tokens) and its word
//                         prefixes; each chosen token's row is the word
//                         prefix plus the popcount below it;
//   ec_membership_kernel  the same bitmap and prefixes rebuilt from the
//                         rows' tokens (for the combine and the backward
//                         pass, which take the routing as an input);
//   ec_gather_kernel      x_perm[row] = x[row_token[row]];
//   ec_combine_kernel     warp per token: its chosen experts in index order
//                         (a ballot over its membership bits), the gated sum
//                         of their rows in fp32, rounded once;
//   ec_combine_backward_kernel   warp per row: dYp = g dY_t, dg = <dY_t, y>;
//   ec_unpermute_kernel   warp per token: dX = dY + sum of its rows' dXp +
//                         the router part.
// No atomics decide any order: every result is reproducible bit for bit.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {

namespace {

constexpr int SEL_THREADS = 512;

// Order key of a score (every key > 0; -0.0 counts as +0.0).
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Writes the expert's membership words (bitmap over T tokens) and their
// exclusive popcount prefixes from the words in shared memory.
__device__ __forceinline__ void store_words(const uint32_t *words, int W, uint32_t *bm, int32_t *prefix,
                                            int *scratch) {
  // block-wide exclusive scan of the words' popcounts, in word order
  const int tid = threadIdx.x;
  const int per = (W + blockDim.x - 1) / blockDim.x;
  int local = 0;
  for (int i = 0; i < per; ++i) {
    const int w = tid * per + i;
    if (w < W) local += __popc(words[w]);
  }
  scratch[tid] = local;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int i = 0; i < (int)blockDim.x; ++i) {
      const int c = scratch[i];
      scratch[i] = run;
      run += c;
    }
  }
  __syncthreads();
  int run = scratch[tid];
  for (int i = 0; i < per; ++i) {
    const int w = tid * per + i;
    if (w < W) {
      bm[w] = words[w];
      prefix[w] = run;
      run += __popc(words[w]);
    }
  }
}

// One CTA per expert e: the Ce tokens with the largest p[:, e].
__global__ void __launch_bounds__(SEL_THREADS) ec_select_kernel(const float *__restrict__ probs, int T, int E, int Ce,
                                                                int32_t *row_token, float *row_gate,
                                                                int32_t *expert_offsets, uint32_t *bm_all,
                                                                int32_t *prefix_all) {
  extern __shared__ uint32_t sm[];
  uint32_t *keys = sm;                         // [T]
  const int W = (T + 31) / 32;
  uint32_t *words = keys + T;                  // [W]
  __shared__ int hist[256];
  __shared__ int scratch[SEL_THREADS];
  __shared__ uint32_t s_prefix, s_need;
  __shared__ int warp_ties[SEL_THREADS / 32];
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int t = tid; t < T; t += SEL_THREADS) keys[t] = score_key(probs[(int64_t)t * E + e]);
  if (tid == 0) { s_prefix = 0u; s_need = (uint32_t)Ce; }
  __syncthreads();
  // radix select, most significant byte first: after the four passes s_prefix
  // is the Ce-th largest key and s_need the number of tokens with exactly that
  // key to take (the keys above it are all taken)
  uint32_t mask = 0u;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += SEL_THREADS) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int t = tid; t < T; t += SEL_THREADS)
      if ((keys[t] & mask) == prefix) atomicAdd(&hist[(keys[t] >> shift) & 255u], 1);
    __syncthreads();
    if (tid == 0) {
      uint32_t need = s_need;
      int bin = 255;
      for (; bin > 0; --bin) {
        if ((uint32_t)hist[bin] >= need) break;
        need -= (uint32_t)hist[bin];
      }
      s_prefix = prefix | ((uint32_t)bin << shift);
      s_need = need;
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t kstar = s_prefix;
  const uint32_t need = s_need;
  // membership in token order: 32 tokens per warp per step, ties ranked by a
  // running count over the steps (warp prefix, then block prefix)
  uint32_t ties_before = 0;
  for (int base = 0; base < T; base += SEL_THREADS) {
    const int t = base + tid;
    const uint32_t key = t < T ? keys[t] : 0u;
    const bool tie = t < T && key == kstar;
    const uint32_t tb = __ballot_sync(0xffffffffu, tie);
    if (lane == 0) warp_ties[warp] = __popc(tb);
    __syncthreads();
    uint32_t before = ties_before;
    for (int w = 0; w < warp; ++w) before += warp_ties[w];
    before += __popc(tb & ((1u << lane) - 1u));
    const bool take = t < T && (key > kstar || (tie && before < need));
    const uint32_t wb = __ballot_sync(0xffffffffu, take);
    if (lane == 0 && (base >> 5) + warp < W) words[(base >> 5) + warp] = wb;
    for (int w = 0; w < SEL_THREADS / 32; ++w) ties_before += warp_ties[w];
    __syncthreads();
  }
  uint32_t *bm = bm_all + (int64_t)e * W;
  int32_t *prefix = prefix_all + (int64_t)e * W;
  store_words(words, W, bm, prefix, scratch);
  __syncthreads();
  // each chosen token's row: e Ce + word prefix + popcount below it in its word
  for (int t = tid; t < T; t += SEL_THREADS) {
    const uint32_t word = words[t >> 5];
    if ((word >> (t & 31)) & 1u) {
      const int pos = prefix[t >> 5] + __popc(word & ((1u << (t & 31)) - 1u));
      row_token[(int64_t)e * Ce + pos] = t;
      row_gate[(int64_t)e * Ce + pos] = probs[(int64_t)t * E + e];
    }
  }
  if (tid == 0) expert_offsets[e] = e * Ce;
  if (e == 0 && tid == 0) expert_offsets[E] = E * Ce;
}

// One CTA per expert: the membership bitmap and prefixes from the rows' tokens.
__global__ void __launch_bounds__(SEL_THREADS) ec_membership_kernel(const int32_t *__restrict__ row_token, int T,
                                                                    int Ce, uint32_t *bm_all, int32_t *prefix_all) {
  extern __shared__ uint32_t words[];          // [W]
  __shared__ int scratch[SEL_THREADS];
  const int e = blockIdx.x, tid = threadIdx.x;
  const int W = (T + 31) / 32;
  for (int w = tid; w < W; w += SEL_THREADS) words[w] = 0u;
  __syncthreads();
  for (int i = tid; i < Ce; i += SEL_THREADS) {
    const int t = row_token[(int64_t)e * Ce + i];
    if (t >= 0 && t < T) atomicOr(&words[t >> 5], 1u << (t & 31));
  }
  __syncthreads();
  store_words(words, W, bm_all + (int64_t)e * W, prefix_all + (int64_t)e * W, scratch);
}

template <typename XT>
__global__ void __launch_bounds__(256) ec_gather_kernel(const XT *__restrict__ x, const int32_t *__restrict__ row_token,
                                                        int64_t rows, int d, XT *__restrict__ x_perm) {
  constexpr int V = Vec16<XT>::N;
  const int nvec = d / V;
  const int64_t units = rows * nvec;
  for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < units; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = u / nvec;
    const int v = (int)(u - row * nvec);
    const int t = __ldg(row_token + row);
    *reinterpret_cast<uint4 *>(x_perm + row * d + (int64_t)v * V) =
        *reinterpret_cast<const uint4 *>(x + (int64_t)t * d + (int64_t)v * V);
  }
}

// The rows of token t's chosen experts, in expert order, written to the
// warp's list (row, gate); returns their number.
__device__ __forceinline__ int token_rows_ec(int t, int E, int Ce, int W, const uint32_t *__restrict__ bm,
                                             const int32_t *__restrict__ prefix, const float *__restrict__ row_gate,
                                             int *lrow, float *lgate) {
  const int lane = threadIdx.x & 31;
  const int w = t >> 5;
  const uint32_t bit = 1u << (t & 31);
  int n = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    int row = -1;
    if (e < E) {
      const uint32_t word = bm[(int64_t)e * W + w];
      if (word & bit) row = e * Ce + prefix[(int64_t)e * W + w] + __popc(word & (bit - 1u));
    }
    const uint32_t mine = __ballot_sync(0xffffffffu, row >= 0);
    const int at = n + __popc(mine & ((1u << lane) - 1u));
    if (row >= 0) {
      lrow[at] = row;
      if (lgate) lgate[at] = row_gate[row];
    }
    n += __popc(mine);
  }
  __syncwarp();
  return n;
}

template <typename XT>
__global__ void __launch_bounds__(256) ec_combine_kernel(const XT *__restrict__ x, const XT *__restrict__ y_perm,
                                                         const float *__restrict__ row_gate,
                                                         const uint32_t *__restrict__ bm,
                                                         const int32_t *__restrict__ prefix, int T, int d, int E, int Ce,
                                                         int residual, XT *__restrict__ out) {
  constexpr int V = Vec16<XT>::N;
  __shared__ int s_row[8][256];
  __shared__ float s_gate[8][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = d / V, W = (T + 31) / 32;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    const int n = token_rows_ec(t, E, Ce, W, bm, prefix, row_gate, s_row[warp], s_gate[warp]);
    for (int v = lane; v < nvec; v += 32) {
      float acc[V], y[V];
      if (residual) Vec16<XT>::load(x + (int64_t)t * d + v * V, acc);
      else {
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.0f;
      }
      for (int j = 0; j < n; ++j) {
        Vec16<XT>::load(y_perm + (int64_t)s_row[warp][j] * d + v * V, y);
        const float g = s_gate[warp][j];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = fmaf(g, y[i], acc[i]);
      }
      Vec16<XT>::store(out + (int64_t)t * d + v * V, acc);
    }
    __syncwarp();
  }
}

template <typename XT>
__global__ void __launch_bounds__(256) ec_combine_backward_kernel(const XT *__restrict__ dy,
                                                                  const XT *__restrict__ y_perm,
                                                                  const int32_t *__restrict__ row_token,
                                                                  const float *__restrict__ row_gate, int64_t rows,
                                                                  int d, XT *__restrict__ dyp, float *__restrict__ dg_row) {
  constexpr int V = Vec16<XT>::N;
  const int lane = threadIdx.x & 31;
  const int nvec = d / V;
  for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; row < rows;
       row += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int t = row_token[row];
    const float g = row_gate[row];
    float dot = 0.0f;
    for (int v = lane; v < nvec; v += 32) {
      float a[V], y[V], o[V];
      Vec16<XT>::load(dy + (int64_t)t * d + v * V, a);
      Vec16<XT>::load(y_perm + row * d + v * V, y);
#pragma unroll
      for (int i = 0; i < V; ++i) {
        dot = fmaf(a[i], y[i], dot);
        o[i] = g * a[i];
      }
      Vec16<XT>::store(dyp + row * d + v * V, o);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) dg_row[row] = dot;
  }
}

template <typename XT>
__global__ void __launch_bounds__(256) ec_unpermute_kernel(const XT *__restrict__ dy, const XT *__restrict__ dxp,
                                                           const float *__restrict__ dxr,
                                                           const uint32_t *__restrict__ bm,
                                                           const int32_t *__restrict__ prefix, int T, int d, int E,
                                                           int Ce, int residual, XT *__restrict__ dx) {
  constexpr int V = Vec16<XT>::N;
  __shared__ int s_row[8][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = d / V, W = (T + 31) / 32;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    const int n = token_rows_ec(t, E, Ce, W, bm, prefix, nullptr, s_row[warp], nullptr);
    for (int v = lane; v < nvec; v += 32) {
      float acc[V], y[V], r[V];
      if (residual) Vec16<XT>::load(dy + (int64_t)t * d + v * V, acc);
      else {
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.0f;
      }
      for (int j = 0; j < n; ++j) {
        Vec16<XT>::load(dxp + (int64_t)s_row[warp][j] * d + v * V, y);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += y[i];
      }
      Vec16<float>::load(dxr + (int64_t)t * d + v * V, r);
      if (V == 8) Vec16<float>::load(dxr + (int64_t)t * d + v * V + 4, r + 4);
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] += r[i];
      Vec16<XT>::store(dx + (int64_t)t * d + v * V, acc);
    }
    __syncwarp();
  }
}

int warp_grid(int64_t items) {
  int64_t g = (items + 7) / 8;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (g > cap) g = cap;
  return (int)(g > 0 ? g : 1);
}

size_t select_smem(int T) { return sizeof(uint32_t) * ((size_t)T + (size_t)(T + 31) / 32); }

}  // namespace

cudaError_t launch_ec_select(const Shape &sh, const float *probs, int32_t *row_token, float *row_gate,
                             int32_t *expert_offsets, uint32_t *bm, int32_t *prefix, cudaStream_t stream) {
  static cudaError_t attr = cudaFuncSetAttribute(ec_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)select_smem(kExpertChoiceMaxTokens));
  if (attr != cudaSuccess) return attr;
  return launch_kernel(ec_select_kernel, dim3(sh.E), dim3(SEL_THREADS), select_smem(sh.T), stream, probs, sh.T, sh.E,
                       (int)(sh.rows / sh.E), row_token, row_gate, expert_offsets, bm, prefix);
}

cudaError_t launch_ec_membership(const Shape &sh, const int32_t *row_token, uint32_t *bm, int32_t *prefix,
                                 cudaStream_t stream) {
  return launch_kernel(ec_membership_kernel, dim3(sh.E), dim3(SEL_THREADS), sizeof(uint32_t) * ((sh.T + 31) / 32),
                       stream, row_token, sh.T, (int)(sh.rows / sh.E), bm, prefix);
}

cudaError_t launch_ec_gather(const Shape &sh, const void *x, const int32_t *row_token, void *x_perm,
                             cudaStream_t stream) {
  const int vec = sh.dtype == MOE_BF16 ? 8 : 4;
  int64_t g = (sh.rows * (sh.d / vec) + 255) / 256;
  if (g > 16LL * sm_count()) g = 16LL * sm_count();
  if (sh.dtype == MOE_BF16)
    return launch_kernel(ec_gather_kernel<bf16>, dim3((unsigned)(g > 0 ? g : 1)), dim3(256), 0, stream,
                         (const bf16 *)x, row_token, sh.rows, sh.d, (bf16 *)x_perm);
  return launch_kernel(ec_gather_kernel<float>, dim3((unsigned)(g > 0 ? g : 1)), dim3(256), 0, stream,
                       (const float *)x, row_token, sh.rows, sh.d, (float *)x_perm);
}

cudaError_t launch_ec_combine(const Shape &sh, const void *x, const void *y_perm, const float *row_gate,
                              const uint32_t *bm, const int32_t *prefix, void *out, cudaStream_t stream) {
  const int Ce = (int)(sh.rows / sh.E);
  if (sh.dtype == MOE_BF16)
    return launch_kernel(ec_combine_kernel<bf16>, dim3(warp_grid(sh.T)), dim3(256), 0, stream, (const bf16 *)x,
                         (const bf16 *)y_perm, row_gate, bm, prefix, sh.T, sh.d, sh.E, Ce, sh.residual, (bf16 *)out);
  return launch_kernel(ec_combine_kernel<float>, dim3(warp_grid(sh.T)), dim3(256), 0, stream, (const float *)x,
                       (const float *)y_perm, row_gate, bm, prefix, sh.T, sh.d, sh.E, Ce, sh.residual, (float *)out);
}

cudaError_t launch_ec_combine_backward(const Shape &sh, const void *dy, const void *y_perm, const int32_t *row_token,
                                       const float *row_gate, void *dyp, float *dg_row, cudaStream_t stream) {
  if (sh.dtype == MOE_BF16)
    return launch_kernel(ec_combine_backward_kernel<bf16>, dim3(warp_grid(sh.rows)), dim3(256), 0, stream,
                         (const bf16 *)dy, (const bf16 *)y_perm, row_token, row_gate, sh.rows, sh.d, (bf16 *)dyp, dg_row);
  return launch_kernel(ec_combine_backward_kernel<float>, dim3(warp_grid(sh.rows)), dim3(256), 0, stream,
                       (const float *)dy, (const float *)y_perm, row_token, row_gate, sh.rows, sh.d, (float *)dyp,
                       dg_row);
}

cudaError_t launch_ec_unpermute(const Shape &sh, const void *dy, const void *dxp, const float *dxr, const uint32_t *bm,
                                const int32_t *prefix, void *dx, cudaStream_t stream) {
  const int Ce = (int)(sh.rows / sh.E);
  if (sh.dtype == MOE_BF16)
    return launch_kernel(ec_unpermute_kernel<bf16>, dim3(warp_grid(sh.T)), dim3(256), 0, stream, (const bf16 *)dy,
                         (const bf16 *)dxp, dxr, bm, prefix, sh.T, sh.d, sh.E, Ce, sh.residual, (bf16 *)dx);
  return launch_kernel(ec_unpermute_kernel<float>, dim3(warp_grid(sh.T)), dim3(256), 0, stream, (const float *)dy,
                       (const float *)dxp, dxr, bm, prefix, sh.T, sh.d, sh.E, Ce, sh.residual, (float *)dx);
}

}  // namespace moe
