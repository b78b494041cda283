// Dispatch of the MoE layer: expert capacity, token-order slots, dropped
// tokens, and the packing of kept tokens into per-expert row groups.
//
// "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティングと負荷
// 分散", section エキスパートには「定員」がある: every expert takes at most
// C = expert capacity tokens (eq. (3)); tokens over capacity skip the expert
// and pass through the residual. The kept token-expert pairs are compacted
// into contiguous variable-size groups ("LRMoE: Demand-Side Load
// Re-Calibration for Efficient MoE Training on Memory-Constrained Nodes",
// section この記事のポイント).
//
// Slots are the rank of a token among the tokens that chose the same expert,
// in ascending token order. They are computed without atomics deciding any
// order, so the result is exact and reproducible:
//   1. per block of 256 tokens, a bitmap present[e][token] in shared memory
//      and its per-expert popcounts;
//   2. per expert, an exclusive scan of those counts over blocks;
//   3. per block, rank = block base + popcount of the bitmap below the token,
//      slot = rank if rank < C else -1; kept = min(load, C) and the group
//      offsets (exclusive scan over experts) are recomputed per block;
//   4. a separate wide grid copies each token's row to its kept rows with
//      16-byte vector loads and stores.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int DT = DISPATCH_TOKENS;   // 256 tokens per block
constexpr int WORDS = DT / 32;        // bitmap words per expert

// Marks (token, expert) pairs of this block's tokens; returns nothing, fills `present`.
// A pair with an expert outside [0, E) or a repeat within one token is left out
// and, when `st` is given, recorded.
__device__ __forceinline__ void build_bitmap(uint32_t *present, const int32_t *idx, int T, int E, int k, int t0,
                                             DeviceStatus *st) {
  for (int i = threadIdx.x; i < E * WORDS; i += blockDim.x) present[i] = 0;
  __syncthreads();
  const int t = t0 + threadIdx.x;
  if (t < T) {
    const uint32_t bit = 1u << (threadIdx.x & 31);
    for (int j = 0; j < k; ++j) {
      const int e = idx[(int64_t)t * k + j];
      if (e < 0 || e >= E) {
        if (st) record_error(st, MOE_DEVERR_BAD_EXPERT, t);
        continue;
      }
      const uint32_t old = atomicOr(&present[e * WORDS + (threadIdx.x >> 5)], bit);
      if ((old & bit) && st) record_error(st, MOE_DEVERR_DUP_EXPERT, t);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(DT) dispatch_count_kernel(const int32_t *idx, int T, int E, int k,
                                                            int32_t *block_counts, DeviceStatus *st) {
  extern __shared__ uint32_t present[];
  build_bitmap(present, idx, T, E, k, blockIdx.x * DT, st);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) c += __popc(present[e * WORDS + w]);
    block_counts[(int64_t)blockIdx.x * E + e] = c;
  }
}

// One block per expert: exclusive scan of the per-block counts over blocks.
__global__ void __launch_bounds__(256) dispatch_scan_kernel(const int32_t *block_counts, int nblk, int E,
                                                            int32_t *block_base, int32_t *load) {
  __shared__ int warp_sums[8];
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int carry = 0;
  for (int b0 = 0; b0 < nblk; b0 += 256) {
    const int b = b0 + threadIdx.x;
    const int v = (b < nblk) ? block_counts[(int64_t)b * E + e] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int s = warp_sums[w];
      if (w < warp) before += s;
      total += s;
    }
    if (b < nblk) block_base[(int64_t)b * E + e] = carry + before + incl - v;
    carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) load[e] = carry;
}

__global__ void __launch_bounds__(DT) dispatch_assign_kernel(const int32_t *idx, int T, int E, int k, int64_t C,
                                                             const int32_t *block_base, const int32_t *load,
                                                             int32_t *slot, int32_t *kept_out,
                                                             int32_t *offsets_out, int32_t *row_token) {
  extern __shared__ uint32_t present[];          // [E][WORDS]
  __shared__ int pre[256 * WORDS];               // popcount prefix per (expert, word)
  __shared__ int off[257];
  __shared__ int warp_sums[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // group offsets: exclusive scan over experts of kept = min(load, C)
  {
    const int e = threadIdx.x;
    int kept = 0;
    if (e < E) {
      const int l = load[e];
      kept = (C >= 0 && (int64_t)l > C) ? (int)C : l;
    }
    int incl = kept;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    if (e < E) off[e] = before + incl - kept;
    if (e == E - 1) off[E] = before + incl;
    if (blockIdx.x == 0 && e < E) kept_out[e] = kept;
    __syncthreads();
    if (blockIdx.x == 0) {
      if (threadIdx.x < E) offsets_out[threadIdx.x] = off[threadIdx.x];
      if (threadIdx.x == 0) offsets_out[E] = off[E];
    }
  }

  const int t0 = blockIdx.x * DT;
  build_bitmap(present, idx, T, E, k, t0, nullptr);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
      pre[e * WORDS + w] = run;
      run += __popc(present[e * WORDS + w]);
    }
  }
  __syncthreads();

  const int t = t0 + threadIdx.x;
  if (t >= T) return;
  const int word = threadIdx.x >> 5;
  const uint32_t below = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(int64_t)t * k + j];
    int s = -1;
    bool ok = (e >= 0 && e < E);
    for (int jj = 0; ok && jj < j; ++jj) ok = idx[(int64_t)t * k + jj] != e;  // repeats count as dropped
    if (ok) {
      const int local = pre[e * WORDS + word] + __popc(present[e * WORDS + word] & below);
      const int64_t rank = (int64_t)block_base[(int64_t)blockIdx.x * E + e] + local;
      if (C < 0 || rank < C) {
        s = (int)rank;
        row_token[off[e] + s] = t;
      }
    }
    slot[(int64_t)t * k + j] = s;
  }
}

// Warp per token: read the row once, write it to each kept row.
template <typename XT>
__global__ void __launch_bounds__(256) dispatch_gather_kernel(const XT *x, const int32_t *idx, const int32_t *slot,
                                                              const int32_t *offsets, int T, int d, int k,
                                                              XT *x_perm) {
  const int lane = threadIdx.x & 31;
  const int nvec = d / Vec16<XT>::N;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
    int row = -1;
    if (lane < k) {
      const int s = slot[(int64_t)t * k + lane];
      if (s >= 0) row = offsets[idx[(int64_t)t * k + lane]] + s;
    }
    int rows[8];
    int nr = 0;
    for (int j = 0; j < k; ++j) {
      const int r = __shfl_sync(0xffffffffu, row, j);
      if (r >= 0) rows[nr++] = r;
    }
    if (nr == 0) continue;
    const XT *src = x + (int64_t)t * d;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = *reinterpret_cast<const uint4 *>(src + v * Vec16<XT>::N);
      for (int j = 0; j < nr; ++j)
        *reinterpret_cast<uint4 *>(x_perm + (int64_t)rows[j] * d + v * Vec16<XT>::N) = u;
    }
  }
}

}  // namespace

int dispatch_blocks(const Shape &sh) { return (sh.T + DT - 1) / DT; }

cudaError_t launch_dispatch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot, int32_t *kept,
                            int32_t *offsets, int32_t *row_token, void *x_perm, void *ws, cudaStream_t stream) {
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  DeviceStatus *st = reinterpret_cast<DeviceStatus *>(w + L.status);
  int32_t *counts = reinterpret_cast<int32_t *>(w + L.disp_counts);
  int32_t *base = reinterpret_cast<int32_t *>(w + L.disp_base);
  int32_t *load = reinterpret_cast<int32_t *>(w + L.disp_load);
  const int nblk = dispatch_blocks(sh);
  const size_t bm = sizeof(uint32_t) * (size_t)sh.E * WORDS;
  dispatch_count_kernel<<<nblk, DT, bm, stream>>>(idx, sh.T, sh.E, sh.k, counts, st);
  dispatch_scan_kernel<<<sh.E, 256, 0, stream>>>(counts, nblk, sh.E, base, load);
  dispatch_assign_kernel<<<nblk, DT, bm, stream>>>(idx, sh.T, sh.E, sh.k, sh.C, base, load, slot, kept, offsets,
                                                   row_token);
  int sms = 148;
  {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  const int warps_needed = sh.T;
  int grid = (warps_needed + 7) / 8;
  if (grid > sms * 8) grid = sms * 8;
  if (sh.dtype == MOE_BF16)
    dispatch_gather_kernel<bf16><<<grid, 256, 0, stream>>>((const bf16 *)x, idx, slot, offsets, sh.T, sh.d, sh.k,
                                                           (bf16 *)x_perm);
  else
    dispatch_gather_kernel<float><<<grid, 256, 0, stream>>>((const float *)x, idx, slot, offsets, sh.T, sh.d,
                                                            sh.k, (float *)x_perm);
  return cudaGetLastError();
}

// The same launch sequence as launch_dispatch, with the scratch arrays given
// explicitly (used by the workspace-free entry point).
cudaError_t launch_dispatch_with_scratch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot,
                                         int32_t *kept, int32_t *offsets, int32_t *row_token, void *x_perm,
                                         int32_t *counts, int32_t *base, int32_t *load, DeviceStatus *st,
                                         cudaStream_t stream) {
  const int nblk = dispatch_blocks(sh);
  const size_t bm = sizeof(uint32_t) * (size_t)sh.E * WORDS;
  dispatch_count_kernel<<<nblk, DT, bm, stream>>>(idx, sh.T, sh.E, sh.k, counts, st);
  dispatch_scan_kernel<<<sh.E, 256, 0, stream>>>(counts, nblk, sh.E, base, load);
  dispatch_assign_kernel<<<nblk, DT, bm, stream>>>(idx, sh.T, sh.E, sh.k, sh.C, base, load, slot, kept, offsets,
                                                   row_token);
  int sms = 148;
  {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  int grid = (sh.T + 7) / 8;
  if (grid > sms * 8) grid = sms * 8;
  if (sh.dtype == MOE_BF16)
    dispatch_gather_kernel<bf16><<<grid, 256, 0, stream>>>((const bf16 *)x, idx, slot, offsets, sh.T, sh.d, sh.k,
                                                           (bf16 *)x_perm);
  else
    dispatch_gather_kernel<float><<<grid, 256, 0, stream>>>((const float *)x, idx, slot, offsets, sh.T, sh.d,
                                                            sh.k, (float *)x_perm);
  return cudaGetLastError();
}

}  // namespace moe
