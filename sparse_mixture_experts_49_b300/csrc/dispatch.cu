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
//      counts over blocks for every expert (block bases, one thread per
//      expert with 32 loads in flight), and derives kept = min(load, C) and
//      the group offsets (exclusive scan over experts). The same kernel
//      writes each pair's rank inside its block (popcount of the bitmap below
//      the token) into slot, as -2 - rank;
//   2. a grid-stride loop over (token, 512-byte chunk) units, one warp per
//      unit and four units in flight per warp: per (token, j) pair, rank =
//      block base + that rank, slot = rank if rank < C else -1, the row owner
//      of each kept pair, and the copy of the token's row to its kept rows.
//      The loop keeps the 1-read-to-k-writes traffic spread evenly over every
//      SM whatever the number of tokens.
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {

namespace {

#ifndef MOE_DISPATCH_COPY_BLOCKS_PER_SM
#define MOE_DISPATCH_COPY_BLOCKS_PER_SM 16  // copy grid cap (measured on the B300: 16 > 8 > 4)
#endif

constexpr int DT = DISPATCH_TOKENS;   // 256 tokens per counting block
constexpr int WORDS = DT / 32;        // bitmap words per expert

// Per-block expert counts and each pair's rank inside its block (written to
// local_rank, which is the caller's slot array, as -2 - rank; -1 for a pair
// left out); the last block scans the counts into block bases and writes
// kept[] and the group offsets.
//
// One thread per token of the block: its k experts are read once; a pair
// with an expert outside [0, E) or a repeat of an earlier pair of the same
// token is left out (rank -1) and, when `st` is given, recorded. The kept
// pairs set bit (token) of present[e]; a pair's rank is the number of set
// bits of present[e] below its token (word prefix + popcount in the word).
// KMAX >= k bounds the unrolled per-token loops.
// kc <= k: the columns counted (the first kc); with rerouting (kc = 1, k = 2)
// the last block writes kept_out = the first round's kept counts and no
// offsets (offsets_out null): the second round's kernel completes them.
template <int KMAX>
__global__ void __launch_bounds__(DT) dispatch_count_kernel(const int32_t *__restrict__ idx, int T, int E, int k,
                                                            int kc, int64_t C, int32_t *block_counts,
                                                            int32_t *block_base, int32_t *kept_out,
                                                            int32_t *offsets_out, int32_t *__restrict__ local_rank,
                                                            unsigned int *counter, DeviceStatus *st) {
  extern __shared__ uint32_t present[];             // [E][WORDS] bitmap, then [E][WORDS] word prefixes
  int *prefix = reinterpret_cast<int *>(present + E * WORDS);
  __shared__ bool last;
  __shared__ int warp_sums[8];
  __shared__ int total[256];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x * DT + tid;
  const bool live = t < T;
  int ev[KMAX];
  unsigned ok = 0;  // bit j: pair j is counted
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    ev[j] = (live && j < k) ? idx[(int64_t)t * k + j] : -1;
    if (live && j < k) {
      bool good = ev[j] >= 0 && ev[j] < E;
      if (!good && st) record_error(st, MOE_DEVERR_BAD_EXPERT, t);
#pragma unroll
      for (int jj = 0; jj < j; ++jj)
        if (good && ev[jj] == ev[j]) {
          good = false;
          if (st) record_error(st, MOE_DEVERR_DUP_EXPERT, t);
        }
      ok |= (good ? 1u : 0u) << j;
    }
  }
  for (int i = tid; i < E * WORDS; i += DT) present[i] = 0;
  __syncthreads();
  const uint32_t bit = 1u << lane;
#pragma unroll
  for (int j = 0; j < KMAX; ++j)
    if (j < kc && ((ok >> j) & 1u)) atomicOr(&present[ev[j] * WORDS + warp], bit);
  __syncthreads();
  for (int e = tid; e < E; e += DT) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
      prefix[e * WORDS + w] = c;
      c += __popc(present[e * WORDS + w]);
    }
    block_counts[(int64_t)blockIdx.x * E + e] = c;
  }
  __syncthreads();
  if (live) {
    const uint32_t below = bit - 1u;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= kc) break;
      int r = -1;  // -2 - rank for a counted pair (see the placing kernel)
      if ((ok >> j) & 1u) r = -2 - (prefix[ev[j] * WORDS + warp] + __popc(present[ev[j] * WORDS + warp] & below));
      local_rank[(int64_t)t * k + j] = r;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // Block bases: per expert (one thread each), an exclusive scan of the
  // blocks' counts in block order; 32 loads in flight per step.
  const int nb = (int)gridDim.x;
  if (tid < E) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      int c[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) c[i] = (b0 + i < nb) ? __ldcg(block_counts + (int64_t)(b0 + i) * E + tid) : 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (b0 + i < nb) block_base[(int64_t)(b0 + i) * E + tid] = run;
        run += c[i];
      }
    }
    total[tid] = run;
  }
  __syncthreads();
  // kept = min(load, C) and the group offsets (exclusive scan over experts)
  const int e = tid;
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
    if (offsets_out) offsets_out[e] = before + incl - kept;
  }
  if (e == E - 1 && offsets_out) offsets_out[E] = before + incl;
  if (tid == 0) *counter = 0u;
}

// No-Token-Left-Behind, second round ([Switch] section 論文の限界と、まだ分か
// っていないこと: overflow goes to the token's second candidate). Runs after
// the first-choice count (k = 2 columns, the first counted): a token whose
// first-choice rank (block base + its rank inside the block, from slot[t, 0])
// reaches C is a round-2 candidate of its second choice idx[t, 1]. Per block
// of 256 tokens, a bitmap of the candidates per expert gives each its rank
// inside the block (slot[t, 1] = -2 - rank; -1 for a non-candidate) and the
// block's counts; the last block scans the counts over blocks into bases,
// keeps min(candidates, C - kept1) per expert and writes kept = kept1 + kept2
// and the group offsets.
__global__ void __launch_bounds__(DT) dispatch_reroute_kernel(const int32_t *__restrict__ idx, int T, int E,
                                                              int64_t C, const int32_t *block_base1,
                                                              const int32_t *kept1, int32_t *slot,
                                                              int32_t *block_counts2, int32_t *block_base2,
                                                              int32_t *kept_out, int32_t *offsets_out,
                                                              unsigned int *counter) {
  extern __shared__ uint32_t present[];             // [E][WORDS] bitmap, then [E][WORDS] word prefixes
  int *prefix = reinterpret_cast<int *>(present + E * WORDS);
  __shared__ bool last;
  __shared__ int warp_sums[8];
  __shared__ int total[256];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x * DT + tid;
  int e2 = -1;
  if (t < T && C >= 0) {
    const int enc = slot[(int64_t)t * 2];
    const int e1 = idx[(int64_t)t * 2], e = idx[(int64_t)t * 2 + 1];
    if (enc <= -2 && e >= 0 && e < E && e != e1) {
      const int64_t rank1 = (int64_t)block_base1[(int64_t)blockIdx.x * E + e1] + (-2 - enc);
      if (rank1 >= C) e2 = e;
    }
  }
  for (int i = tid; i < E * WORDS; i += DT) present[i] = 0;
  __syncthreads();
  const uint32_t bit = 1u << lane;
  if (e2 >= 0) atomicOr(&present[e2 * WORDS + warp], bit);
  __syncthreads();
  for (int e = tid; e < E; e += DT) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < WORDS; ++w) {
      prefix[e * WORDS + w] = c;
      c += __popc(present[e * WORDS + w]);
    }
    block_counts2[(int64_t)blockIdx.x * E + e] = c;
  }
  __syncthreads();
  if (t < T)
    slot[(int64_t)t * 2 + 1] =
        e2 >= 0 ? -2 - (prefix[e2 * WORDS + warp] + __popc(present[e2 * WORDS + warp] & (bit - 1u))) : -1;
  __threadfence();
  __syncthreads();
  if (tid == 0) last = atomicAdd(counter, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  const int nb = (int)gridDim.x;
  if (tid < E) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      int c[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) c[i] = (b0 + i < nb) ? __ldcg(block_counts2 + (int64_t)(b0 + i) * E + tid) : 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (b0 + i < nb) block_base2[(int64_t)(b0 + i) * E + tid] = run;
        run += c[i];
      }
    }
    total[tid] = run;
  }
  __syncthreads();
  const int e = tid;
  int kept = 0;
  if (e < E) {
    const int k1 = __ldcg(kept1 + e);
    const int64_t room = C < 0 ? 0 : C - k1;
    kept = k1 + (int)((int64_t)total[e] < room ? total[e] : room);
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
  if (e < E) {
    kept_out[e] = kept;
    offsets_out[e] = before + incl - kept;
  }
  if (e == E - 1) offsets_out[E] = before + incl;
  if (tid == 0) *counter = 0u;
}

// Slots, row owners and row copies: a grid-stride loop over (token,
// 512-byte chunk) units, one unit per warp and four units in flight per warp
// (16-byte loads). Lanes j < k resolve the token's pairs: slot[t, j] holds
// -2 - r (r = rank inside the token's 256-token block) until the unit of
// chunk 0 replaces it with the final slot (rank = block base + r; slot =
// rank if rank < C else -1) and writes the kept pair's row owner. Units of
// other chunks may read either form and derive the same row, offsets[e] +
// slot. The chunk goes to each kept row of x_perm (if given), or to
// out_dropped (if given) when the token kept none (zeros instead of the
// chunk when zero_dropped: the layer without its residual). KMAX >= k bounds the
// unrolled row stores.
template <typename XT, int KMAX>
__global__ void __launch_bounds__(256) dispatch_place_kernel(
    const XT *__restrict__ x, const int32_t *__restrict__ idx, int T, int d, int E, int k, int64_t C,
    const int32_t *__restrict__ block_base, const int32_t *__restrict__ offsets, int32_t *slot,
    int32_t *__restrict__ row_token, XT *__restrict__ x_perm, XT *__restrict__ out_dropped, int zero_dropped,
    const int32_t *__restrict__ block_base2, const int32_t *__restrict__ kept1) {
  constexpr int V = Vec16<XT>::N;
  constexpr int U = 4;  // units in flight per warp
  const int lane = threadIdx.x & 31;
  const int nvec = d / V;
  const int nchunk = (nvec + 31) / 32;
  const int64_t units = (int64_t)T * nchunk;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const bool copy = x_perm != nullptr || out_dropped != nullptr;
  for (int64_t u0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u0 < units; u0 += U * nwarps) {
    uint4 val[U];
    int row[U], tok[U], vv[U], chunk[U], sl[U], ex[U];
    // x chunks first (they do not depend on the slots), then slot and expert
    // of the lanes' pairs, then block bases and group offsets
#pragma unroll
    for (int b = 0; b < U; ++b) {
      const int64_t u = u0 + b * nwarps;
      const bool in = u < units;
      tok[b] = in ? (int)(u / nchunk) : 0;
      chunk[b] = in ? (int)(u - (int64_t)tok[b] * nchunk) : 0;
      vv[b] = in ? chunk[b] * 32 + lane : nvec;
      if (copy && vv[b] < nvec) val[b] = *reinterpret_cast<const uint4 *>(x + (int64_t)tok[b] * d + (int64_t)vv[b] * V);
      sl[b] = -1;
      ex[b] = 0;
      if (in && lane < k) {
        const int64_t at = (int64_t)tok[b] * k + lane;
        sl[b] = slot[at];
        ex[b] = idx[at];
      }
    }
#pragma unroll
    for (int b = 0; b < U; ++b) {
      row[b] = -1;
      if (sl[b] != -1) {
        const int e = ex[b];
        int s2 = sl[b];
        if (s2 <= -2) {
          // rerouting's second column: a round-2 rank, placed after the expert's round-1 rows
          const bool second = kept1 != nullptr && lane == 1;
          const int64_t rank = (second ? (int64_t)kept1[e] + block_base2[(tok[b] / DT) * E + e]
                                       : (int64_t)block_base[(tok[b] / DT) * E + e]) + (-2 - s2);
          s2 = (C < 0 || rank < C) ? (int)rank : -1;
          if (chunk[b] == 0) {
            slot[(int64_t)tok[b] * k + lane] = s2;
            if (s2 >= 0) row_token[offsets[e] + s2] = tok[b];
          }
        }
        if (s2 >= 0) row[b] = offsets[e] + s2;
      }
    }
    if (!copy) continue;
#pragma unroll
    for (int b = 0; b < U; ++b) {
      const bool kept_any = __ballot_sync(0xffffffffu, row[b] >= 0) != 0u;
      const bool lv = vv[b] < nvec;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        const int r = __shfl_sync(0xffffffffu, row[b], j);  // -1 for j >= k
        if (lv && r >= 0 && x_perm) *reinterpret_cast<uint4 *>(x_perm + (int64_t)r * d + (int64_t)vv[b] * V) = val[b];
      }
      if (lv && !kept_any && out_dropped)
        *reinterpret_cast<uint4 *>(out_dropped + (int64_t)tok[b] * d + (int64_t)vv[b] * V) =
            zero_dropped ? make_uint4(0u, 0u, 0u, 0u) : val[b];
    }
  }
}

}  // namespace

int dispatch_blocks(const Shape &sh) { return (sh.T + DT - 1) / DT; }

// Resident blocks per SM of the placing kernel for this layer's dtype and k
// (queried once per instantiation).
template <typename XT, int KMAX> static int place_occupancy() {
  static int n = -1;
  if (n < 0) {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, dispatch_place_kernel<XT, KMAX>, 256, 0) != cudaSuccess) {
      (void)cudaGetLastError();
      v = 0;
    }
    n = v > 0 ? v : 1;
  }
  return n;
}
static int place_blocks_per_sm(const Shape &sh) {
  if (sh.dtype != MOE_BF16) return place_occupancy<float, 8>();
  if (sh.k == 1) return place_occupancy<bf16, 1>();
  if (sh.k == 2) return place_occupancy<bf16, 2>();
  if (sh.k <= 4) return place_occupancy<bf16, 4>();
  return place_occupancy<bf16, 8>();
}

// The dispatch launch sequence with its scratch given explicitly: per-block
// counts and bases [blocks, E], a zero-initialised completion counter, the
// error word.
cudaError_t launch_dispatch_with_scratch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot,
                                         int32_t *kept, int32_t *offsets, int32_t *row_token, void *x_perm,
                                         void *out_dropped, int32_t *counts, int32_t *base, unsigned int *counter,
                                         DeviceStatus *st, cudaStream_t stream, const RerouteScratch *rr) {
  const int nblk = dispatch_blocks(sh);
  const size_t bm = 2 * sizeof(uint32_t) * (size_t)sh.E * WORDS;  // bitmap + word prefixes
  if (sh.reroute && rr == nullptr) return cudaErrorInvalidValue;
  // rerouting: the first round counts the first column, keeps kept1 apart and leaves the offsets to the second
  const int kc = sh.reroute ? 1 : sh.k;
  int32_t *kept_round1 = sh.reroute ? rr->kept1 : kept;
  int32_t *offsets_round1 = sh.reroute ? nullptr : offsets;
  cudaError_t e;
#define MOE_COUNT(KM)                                                                                            \
  e = launch_kernel(dispatch_count_kernel<KM>, dim3(nblk), dim3(DT), bm, stream, idx, sh.T, sh.E, sh.k, kc, sh.C, \
                    counts, base, kept_round1, offsets_round1, slot, counter, st)
  if (sh.k == 1) MOE_COUNT(1);
  else if (sh.k == 2) MOE_COUNT(2);
  else if (sh.k <= 4) MOE_COUNT(4);
  else MOE_COUNT(8);
#undef MOE_COUNT
  if (e != cudaSuccess) return e;
  if (sh.reroute) {
    e = launch_kernel(dispatch_reroute_kernel, dim3(nblk), dim3(DT), bm, stream, idx, sh.T, sh.E, sh.C,
                      (const int32_t *)base, (const int32_t *)rr->kept1, slot, rr->counts2, rr->base2, kept, offsets,
                      rr->counter2);
    if (e != cudaSuccess) return e;
  }
  const int32_t *base2 = sh.reroute ? rr->base2 : nullptr;
  const int32_t *kept1 = sh.reroute ? rr->kept1 : nullptr;
  // Grid of the grid-stride loop (blocks of 8 warps, four units per warp per
  // pass): one wave of resident blocks when the work fits in two such waves
  // (latency-bound small layers), else MOE_DISPATCH_COPY_BLOCKS_PER_SM blocks
  // per SM (measured faster for the large layers).
  const int vec = sh.dtype == MOE_BF16 ? 8 : 4;
  const int64_t units = (int64_t)sh.T * ((sh.d / vec + 31) / 32);
  int64_t g = (units + 31) / 32;
  const int64_t wave = (int64_t)place_blocks_per_sm(sh) * sm_count();
  if (g <= 2 * wave) {
    if (g > wave) g = wave;
  } else if (g > (int64_t)MOE_DISPATCH_COPY_BLOCKS_PER_SM * sm_count()) {
    g = (int64_t)MOE_DISPATCH_COPY_BLOCKS_PER_SM * sm_count();
  }
  const dim3 grid((unsigned)(g > 0 ? g : 1));
  if (sh.dtype == MOE_BF16) {
#define MOE_PLACE(KM)                                                                                            \
  return launch_kernel(dispatch_place_kernel<bf16, KM>, grid, dim3(256), 0, stream, (const bf16 *)x, idx, sh.T,   \
                       sh.d, sh.E, sh.k, sh.C, base, offsets, slot, row_token, (bf16 *)x_perm, (bf16 *)out_dropped,   \
                       sh.residual ? 0 : 1, base2, kept1)
    if (sh.k == 1) MOE_PLACE(1);
    if (sh.k == 2) MOE_PLACE(2);
    if (sh.k <= 4) MOE_PLACE(4);
    MOE_PLACE(8);
#undef MOE_PLACE
  }
  return launch_kernel(dispatch_place_kernel<float, 8>, grid, dim3(256), 0, stream, (const float *)x, idx, sh.T,
                       sh.d, sh.E, sh.k, sh.C, base, offsets, slot, row_token, (float *)x_perm, (float *)out_dropped,
                       sh.residual ? 0 : 1, base2, kept1);
}

cudaError_t launch_dispatch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot, int32_t *kept,
                            int32_t *offsets, int32_t *row_token, void *x_perm, void *out_dropped, void *ws,
                            cudaStream_t stream) {
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  RerouteScratch rr;
  rr.counts2 = reinterpret_cast<int32_t *>(w + L.disp_counts2);
  rr.base2 = reinterpret_cast<int32_t *>(w + L.disp_base2);
  rr.kept1 = reinterpret_cast<int32_t *>(w + L.disp_kept1);
  rr.counter2 = reinterpret_cast<unsigned int *>(w + L.status + 160);
  return launch_dispatch_with_scratch(sh, x, idx, slot, kept, offsets, row_token, x_perm, out_dropped,
                                      reinterpret_cast<int32_t *>(w + L.disp_counts),
                                      reinterpret_cast<int32_t *>(w + L.disp_base),
                                      reinterpret_cast<unsigned int *>(w + L.status + 128),
                                      reinterpret_cast<DeviceStatus *>(w + L.status), stream, &rr);
}

}  // namespace moe
