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
// order, so the result is exact and reproducible. Two launches:
//   1. per block of 256 tokens, a bitmap present[e][token] in shared memory
//      and its per-expert popcounts; the last block to finish scans those
//      counts over blocks for every expert (block bases, one warp per expert
//      and 32 blocks per shuffle scan), and derives kept = min(load, C) and
//      the group offsets (exclusive scan over experts);
//      The same kernel writes each pair's rank inside its block (popcount of
//      the bitmap below the token) into slot;
//   2. per block of 32 tokens, rank = block base + that rank, slot = rank if
//      rank < C else -1, and the copy of the token's row to each of its kept
//      rows with 16-byte loads and stores (small blocks spread the copy over
//      eight times more SMs; each thread keeps eight 16-byte loads in flight).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int DT = DISPATCH_TOKENS;   // 256 tokens per counting block
constexpr int WORDS = DT / 32;        // bitmap words per expert
constexpr int SUB = 32;               // tokens per placing block

// Marks (token, expert) pairs of the 256 tokens from t0 (one per thread).
// A pair with an expert outside [0, E) or a repeat within one token is left
// out and, when `st` is given, recorded.
__device__ __forceinline__ void build_bitmap(uint32_t *present, const int32_t *__restrict__ idx, int T, int E,
                                             int k, int t0, DeviceStatus *st) {
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

// Per-block expert counts and each pair's rank inside its block (written to
// local_rank, which is the caller's slot array); the last block scans the
// counts into block bases and writes kept[] and the group offsets.
__global__ void __launch_bounds__(DT) dispatch_count_kernel(const int32_t *__restrict__ idx, int T, int E, int k,
                                                            int64_t C, int32_t *block_counts, int32_t *block_base,
                                                            int32_t *kept_out, int32_t *offsets_out,
                                                            int32_t *__restrict__ local_rank, unsigned int *counter,
                                                            DeviceStatus *st) {
  extern __shared__ uint32_t present[];
  __shared__ bool last;
  __shared__ int warp_sums[8];
  build_bitmap(present, idx, T, E, k, blockIdx.x * DT, st);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) c += __popc(present[e * WORDS + w]);
    block_counts[(int64_t)blockIdx.x * E + e] = c;
  }
  {
    // rank of each of this thread's pairs among the block's tokens that chose
    // the same expert (popcount of the bitmap below the token), or -1 for a
    // pair the bitmap left out (bad index, or a repeat within the token)
    const int t = blockIdx.x * DT + threadIdx.x;
    const int word = threadIdx.x >> 5;
    const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
    if (t < T) {
      for (int j = 0; j < k; ++j) {
        const int e = idx[(int64_t)t * k + j];
        bool ok = (e >= 0 && e < E);
        for (int jj = 0; ok && jj < j; ++jj) ok = idx[(int64_t)t * k + jj] != e;
        int r = -1;
        if (ok) {
          r = __popc(present[e * WORDS + word] & below);
          for (int w = 0; w < word; ++w) r += __popc(present[e * WORDS + w]);
        }
        local_rank[(int64_t)t * k + j] = r;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Block bases: per expert, an exclusive scan of the blocks' counts in block
  // order. A warp scans one expert at a time, 32 blocks per step; the loads of
  // all the warp's experts are issued before any is scanned.
  __shared__ int total[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = (int)gridDim.x;
  constexpr int EPW = 256 / (DT / 32);  // experts per warp at most (E <= 256, 8 warps)
  int carry[EPW];
#pragma unroll
  for (int i = 0; i < EPW; ++i) carry[i] = 0;
  for (int b0 = 0; b0 < nb; b0 += 32) {
    const int b = b0 + lane;
    int c[EPW];
#pragma unroll
    for (int i = 0; i < EPW; ++i) {
      const int e = warp + 8 * i;
      c[i] = (e < E && b < nb) ? __ldcg(block_counts + (int64_t)b * E + e) : 0;
    }
#pragma unroll
    for (int i = 0; i < EPW; ++i) {
      const int e = warp + 8 * i;
      if (e >= E) break;
      int incl = c[i];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (b < nb) block_base[(int64_t)b * E + e] = carry[i] + incl - c[i];
      carry[i] += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
#pragma unroll
  for (int i = 0; i < EPW; ++i) {
    const int e = warp + 8 * i;
    if (e < E && lane == 0) total[e] = carry[i];
  }
  __syncthreads();
  // kept = min(load, C) and the group offsets (exclusive scan over experts)
  const int e = threadIdx.x;
  const int run = (e < E) ? total[e] : 0;
  const int kept = (e < E) ? ((C >= 0 && (int64_t)run > C) ? (int)C : run) : 0;
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
  if (e < E) {
    kept_out[e] = kept;
    offsets_out[e] = before + incl - kept;
  }
  if (e == E - 1) offsets_out[E] = before + incl;
  if (threadIdx.x == 0) *counter = 0u;
}

// Slots, row owners and the row copies for 32 tokens: rank = block base +
// the rank inside the 256-token block that the counting kernel left in slot;
// slot = rank if rank < C else -1. KMAX >= k bounds the unrolled row stores.
template <typename XT, int KMAX>
__global__ void __launch_bounds__(DT) dispatch_place_kernel(const XT *__restrict__ x, const int32_t *__restrict__ idx,
                                                            int T, int d, int E, int k, int64_t C,
                                                            const int32_t *__restrict__ block_base,
                                                            const int32_t *__restrict__ offsets,
                                                            int32_t *__restrict__ slot, int32_t *__restrict__ row_token,
                                                            XT *__restrict__ x_perm, XT *__restrict__ out_dropped) {
  __shared__ int rows[SUB][8];
  __shared__ int has_rows[SUB];
  const int64_t tbase = (int64_t)blockIdx.x * SUB;
  {
    // one thread per (token, j) pair of the block's 32 tokens
    const int tl = threadIdx.x >> 3, j = threadIdx.x & 7;
    const int64_t t = tbase + tl;
    int r = -1;
    if (j < k && t < T) {
      const int64_t at = t * k + j;
      const int local = slot[at];
      int s = -1;
      if (local >= 0) {
        const int e = idx[at];
        const int64_t rank = (int64_t)block_base[(t / DT) * E + e] + local;
        if (C < 0 || rank < C) {
          s = (int)rank;
          r = offsets[e] + s;
          row_token[r] = (int)t;
        }
      }
      slot[at] = s;
    }
    rows[tl][j] = r;
    const unsigned any = __ballot_sync(0xffffffffu, r >= 0);
    if (j == 0) has_rows[tl] = (any >> (threadIdx.x & 24)) & 0xffu ? 1 : 0;
  }
  __syncthreads();
  // copy: (token, 16-byte chunk) items spread over the block, 8 loads in flight per thread;
  // a kept token's row goes to its rows of x_perm (if given), a token with no
  // kept assignment goes to out_dropped (if given)
  if (x_perm == nullptr && out_dropped == nullptr) return;
  constexpr int V = Vec16<XT>::N;
  const int nvec = d / V;
  const int items = SUB * nvec;
  for (int i0 = 0; i0 < items; i0 += 8 * DT) {
    uint4 u[8];
    int q[8], v[8];
    bool want[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int it = i0 + b * DT + threadIdx.x;
      q[b] = it / nvec;
      v[b] = it - q[b] * nvec;
      want[b] = it < items && tbase + q[b] < T &&
                (has_rows[q[b]] ? x_perm != nullptr : out_dropped != nullptr);
      if (want[b]) u[b] = *reinterpret_cast<const uint4 *>(x + (tbase + q[b]) * d + (int64_t)v[b] * V);
    }
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (!want[b]) continue;
      if (!has_rows[q[b]]) {
        *reinterpret_cast<uint4 *>(out_dropped + (tbase + q[b]) * d + (int64_t)v[b] * V) = u[b];
        continue;
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const int r = rows[q[b]][j];   // -1 for j >= k
        if (r >= 0) *reinterpret_cast<uint4 *>(x_perm + (int64_t)r * d + (int64_t)v[b] * V) = u[b];
      }
    }
  }
}

}  // namespace

int dispatch_blocks(const Shape &sh) { return (sh.T + DT - 1) / DT; }

// The dispatch launch sequence with its scratch given explicitly: per-block
// counts and bases [blocks, E], a zero-initialised completion counter, the
// error word.
cudaError_t launch_dispatch_with_scratch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot,
                                         int32_t *kept, int32_t *offsets, int32_t *row_token, void *x_perm,
                                         void *out_dropped, int32_t *counts, int32_t *base, unsigned int *counter,
                                         DeviceStatus *st, cudaStream_t stream) {
  const int nblk = dispatch_blocks(sh);
  const size_t bm = sizeof(uint32_t) * (size_t)sh.E * WORDS;
  cudaError_t e = launch_kernel(dispatch_count_kernel, dim3(nblk), dim3(DT), bm, stream, idx, sh.T, sh.E, sh.k, sh.C,
                             counts, base, kept, offsets, slot, counter, st);
  if (e != cudaSuccess) return e;
  const int nsub = (sh.T + SUB - 1) / SUB;
  if (sh.dtype == MOE_BF16) {
#define MOE_PLACE(KM)                                                                                             \
  return launch_kernel(dispatch_place_kernel<bf16, KM>, dim3(nsub), dim3(DT), 0, stream, (const bf16 *)x, idx, sh.T, \
                       sh.d, sh.E, sh.k, sh.C, base, offsets, slot, row_token, (bf16 *)x_perm, (bf16 *)out_dropped)
    if (sh.k == 1) MOE_PLACE(1);
    if (sh.k == 2) MOE_PLACE(2);
    if (sh.k <= 4) MOE_PLACE(4);
    MOE_PLACE(8);
#undef MOE_PLACE
  }
  return launch_kernel(dispatch_place_kernel<float, 8>, dim3(nsub), dim3(DT), 0, stream, (const float *)x, idx, sh.T,
                       sh.d, sh.E, sh.k, sh.C, base, offsets, slot, row_token, (float *)x_perm, (float *)out_dropped);
}

cudaError_t launch_dispatch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot, int32_t *kept,
                            int32_t *offsets, int32_t *row_token, void *x_perm, void *out_dropped, void *ws,
                            cudaStream_t stream) {
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  return launch_dispatch_with_scratch(sh, x, idx, slot, kept, offsets, row_token, x_perm, out_dropped,
                                      reinterpret_cast<int32_t *>(w + L.disp_counts),
                                      reinterpret_cast<int32_t *>(w + L.disp_base),
                                      reinterpret_cast<unsigned int *>(w + L.status + 128),
                                      reinterpret_cast<DeviceStatus *>(w + L.status), stream);
}

}  // namespace moe
