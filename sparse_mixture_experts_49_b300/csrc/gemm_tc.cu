// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM, operands
// staged by TMA), for the expert FFNs of the MoE layer.
//
// The experts' token groups are the variable-size groups that compaction of
// the kept token-expert pairs produces ("LRMoE: Demand-Side Load
// Re-Calibration for Efficient MoE Training on Memory-Constrained Nodes",
// section この記事のポイント: physical compaction -> variable-size grouped
// GEMM). Group sizes stay on the device: a persistent kernel reads the expert
// offsets and walks its tiles itself, so no host synchronisation is needed.
//
// Two grouping modes:
//   grouped-M: C[rows of e, N] = A[rows of e, K] * B_e[N, K]^T
//              (forward GEMMs, and the dgrad GEMMs of the backward pass with
//              B_e read MN-major from the weight tensor);
//   grouped-K: C_e[M, N] = sum over rows r of e of A[r, M]^T B[r, N]
//              (weight gradients; K is the group size, which varies).
// Tile 128 x 256 x 64 (bf16, fp32 accumulator in TMEM), 4-stage TMA ring,
// warp roles: warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
// warps 2-9 epilogue (two per TMEM lane quarter, one per column half). Two
// TMEM accumulators let the epilogue of one tile run under the MMAs of the
// next. The plain-store and forward-activation epilogues stage each warp's
// 32 output rows in 128-byte-swizzled shared memory and write them with TMA
// tile stores; the backward-activation and combine epilogues store rows
// directly.
//
// Pair tiles (PAIR = 1): the two CTAs of a cluster share one tcgen05 MMA of
// M = 256 (cta_group::2). Each CTA stages its own 128 rows of A and its half
// of B's 256 columns (32 KB per K step instead of 48 KB, six stages), and
// keeps its 128 rows of the accumulator in its own TMEM. The even CTA issues
// the MMAs; both CTAs run the epilogue on their own rows. Grouped-M: the odd
// CTA's loads complete on the even CTA's stage barrier, which expects the
// bytes of both halves. Grouped-K (whose last K step of a group zeroes rows
// in each CTA's own half): each CTA's loads complete locally and the odd
// CTA's MMA warp forwards its stage to the even CTA.
#include <cstdlib>

#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {

namespace tc {

constexpr int BM = 128;                // accumulator rows per CTA
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int TMEM_COLS = 512;         // two 128 x 256 fp32 accumulators
constexpr int THREADS = 320;         // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int MAX_E = 256;
// TMA ring: four 48 KB stages (one CTA per tile), six 32 KB stages (pair
// tiles).
template <int PAIR, int EPI> constexpr int n_stages() { return PAIR ? 6 : 4; }
template <int PAIR> constexpr int b_bytes() { return (PAIR ? BN / 2 : BN) * BK * 2; }
template <int PAIR> constexpr int stage_bytes() { return A_BYTES + b_bytes<PAIR>(); }

// Grouped-K: every group has the same tiles, so no prefix array is kept.
// Tile queue of the dynamic scheduler: the producer warp takes tile indices
// from a global counter and passes each to the MMA warp and the eight
// epilogue warps through TQ slots.
constexpr int TQ = 8;
template <bool GK, int NST> struct __align__(8) SmemT {
  uint64_t full[NST];       // this CTA's TMA bytes of the stage have landed
  uint64_t empty[NST];      // the MMAs reading the stage have completed
  uint64_t peer_full[NST];  // pair tiles, even CTA: the odd CTA's half of the stage has landed
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t tq_full[TQ];     // dynamic tiles: slot written by the producer
  uint64_t tq_empty[TQ];    // dynamic tiles: slot read by the MMA warp and every epilogue warp
  uint32_t tmem_base;
  int abort_flag;
  int tile_q[TQ];           // dynamic tiles: the tile of each slot (-1: no more tiles)
  int tile_start[GK ? 1 : MAX_E + 1];  // grouped-M: tiles of the groups before e
};
// Plain-store epilogues (EPI_STORE, EPI_STORE_F32) stage each warp's 32-row
// slice in shared memory (128-byte swizzled rows, 4 KB per warp) and write it
// with a TMA tile store.
constexpr int STAGE_OUT_BYTES = 4096;
constexpr int EPI_WARPS = 8;
template <int EPI> constexpr bool tma_store_epi() { return EPI == EPI_STORE || EPI == EPI_STORE_F32; }
// Epilogues that stage output tiles in shared memory for TMA tile stores: the
// plain stores, and the forward activations (h, and SwiGLU's saved
// pre-activations).
template <int EPI> constexpr bool staged_epi() {
  return tma_store_epi<EPI>() || EPI == EPI_SWIGLU || EPI == EPI_RELU || EPI == EPI_SWIGLU_BWD;
}
// Staging bytes per epilogue warp: one 4 KB buffer (the SwiGLU backward
// splits it into two 2 KB halves: G and U in, dG and dU out).
template <int EPI> constexpr int staging_per_warp() { return staged_epi<EPI>() ? STAGE_OUT_BYTES : 0; }
template <int PAIR, int GROUP_K, int EPI> constexpr size_t smem_bytes() {
  return 1024 /*align slack*/ + (size_t)n_stages<PAIR, EPI>() * stage_bytes<PAIR>() +
         (size_t)EPI_WARPS * staging_per_warp<EPI>() + sizeof(SmemT<GROUP_K != 0, n_stages<PAIR, EPI>()>);
}
static_assert(smem_bytes<0, 0, EPI_STORE>() <= 232448 && smem_bytes<0, 1, EPI_STORE>() <= 232448 &&
                  smem_bytes<1, 0, EPI_STORE>() <= 232448 && smem_bytes<1, 1, EPI_STORE>() <= 232448 &&
                  smem_bytes<0, 0, EPI_SWIGLU>() <= 232448 && smem_bytes<1, 0, EPI_SWIGLU>() <= 232448 &&
                  smem_bytes<0, 0, EPI_SWIGLU_BWD>() <= 232448 && smem_bytes<1, 0, EPI_SWIGLU_BWD>() <= 232448,
              "shared memory budget");

struct Args {
  const int32_t *offsets;  // [E + 1] row offsets of the groups
  int E;
  int M, N, K;             // grouped-M: N (output columns), K; grouped-K: M, N
  int F;                   // SwiGLU: offset of the up half (rows of W1, columns of pre_act / dA)
  int b_once;              // grouped-M: each weight tile is read by one m-tile only (L2 evict-first)
  void *C;                 // bf16, or fp32 for EPI_STORE_F32
  int64_t ldc;
  int64_t sce;             // grouped-K: C_e = C + e * sce
  bf16 *C2;                // SwiGLU forward: pre-activations [rows, 2F]
  int64_t ldc2;
  const bf16 *aux;         // ReLU bwd: h; SwiGLU bwd: pre-activations; combine: x (residual)
  int64_t ldaux;
  const int32_t *a_rows;   // EPI_COMBINE: token of each packed row (row_token)
  const float *gate;       // EPI_COMBINE: gate of each token (top-1)
  int residual;            // EPI_COMBINE: out = x + g y (1) or g y (0)
  unsigned int *sched;     // {next tile, finished CTAs}, zero at launch: dynamic tile order (null: static)
  int m64;                 // grouped-M: M = 64 MMAs for m-tiles with at most 64 rows (1) or full tiles (0)
  int tail_split;          // grouped-M: cut the tiles of a small last wave into column windows (1) or not (0)
  DeviceStatus *st;
};

__device__ __forceinline__ int find_group(const int *tile_start, int E, int tile) {
  int lo = 0, hi = E - 1;  // largest e with tile_start[e] <= tile
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Bounded wait used only after an abort, to let copies already in flight land.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity))
    if (global_timer_ns() - t0 > 200000000ull) break;  // 0.2 s
}

template <int PAIR, int GROUP_K, int A_MN, int B_MN, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                        const __grid_constant__ CUtensorMap tmE, const Args p) {
  constexpr bool TMA_STORE = tma_store_epi<EPI>();
  constexpr bool STAGED = staged_epi<EPI>();
  constexpr int NST = n_stages<PAIR, EPI>();
  constexpr int SPW = staging_per_warp<EPI>();
  constexpr int SB = stage_bytes<PAIR>();
  constexpr int TM = PAIR ? 2 * BM : BM;  // rows of a tile (over both CTAs of a pair)
  using Smem = SmemT<GROUP_K != 0, NST>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *tiles = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t *stage_out = tiles + (size_t)NST * SB;  // STAGED only: [EPI_WARPS][SPW]
  Smem &s = *reinterpret_cast<Smem *>(stage_out + EPI_WARPS * SPW);
  volatile int *abort_flag = &s.abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  // Pair tiles: rank of this CTA in its pair (0 issues the MMAs), the pair's
  // index and count; one CTA per tile otherwise.
  const int crank = PAIR ? (int)cluster_ctarank() : 0;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int half_row = crank * BM;  // first row of this CTA inside the tile
  // grouped-M pair tiles: the odd CTA's loads complete on the even CTA's barriers
  constexpr bool DIRECT = PAIR && !GROUP_K;
  constexpr bool SWIGLU_FWD = (EPI == EPI_SWIGLU);
  // Output columns one tile covers (SwiGLU forward: 128 gate + 128 up accumulators -> 128 outputs).
  constexpr int TN_OUT = SWIGLU_FWD ? 128 : BN;
  const int n_tiles = (p.N + TN_OUT - 1) / TN_OUT;
  const int m_tiles_k = GROUP_K ? (p.M + TM - 1) / TM : 0;

  // ---------------------------------------------------------------- set-up
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (STAGED) prefetch_tmap(&tmC);
      if (SWIGLU_FWD || EPI == EPI_SWIGLU_BWD) prefetch_tmap(&tmD);
      if (SWIGLU_FWD) prefetch_tmap(&tmE);
      for (int i = 0; i < NST; ++i) {
        mbar_init(&s.full[i], 1);
        mbar_init(&s.empty[i], 1);
        mbar_init(&s.peer_full[i], 1);
      }
      // pair tiles: the even CTA's acc_empty collects the epilogue warps of both CTAs
      for (int i = 0; i < 2; ++i) { mbar_init(&s.acc_full[i], 1); mbar_init(&s.acc_empty[i], PAIR ? 16 : 8); }
      mbar_init(&s.drain, 1);
      for (int i = 0; i < TQ; ++i) { mbar_init(&s.tq_full[i], 1); mbar_init(&s.tq_empty[i], 1 + EPI_WARPS); }
      s.abort_flag = 0;
      fence_barrier_init();
    }
  } else if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&s.tmem_base, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&s.tmem_base, TMEM_COLS);
      tmem_relinquish();
    }
    tc_fence_before();
  }
  if (!GROUP_K && warp == 0) {
    // tile_start[e] = number of tiles of groups before e
    int carry = 0;
    if (lane == 0) s.tile_start[0] = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int t = 0;
      if (e < E) {
        const int lo = p.offsets[e], hi = p.offsets[e + 1];
        t = ((hi - lo + TM - 1) / TM) * n_tiles;
      }
      int incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) s.tile_start[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  if (PAIR) cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int tiles_per_group_k = m_tiles_k * n_tiles;  // grouped-K
  const int total_tiles = GROUP_K ? E * tiles_per_group_k : s.tile_start[E];

  // Group row offsets, written by the dispatch before this launch (read-only here).
  auto off = [&](int i) -> int { return __ldg(p.offsets + i); };
  // Tile order inside a group. Grouped-M: m-tiles fastest, so the m-tiles
  // that read the same weight tile run side by side and share it through L2.
  // Grouped-K: n-tiles fastest (the activation tiles are small and shared).
  auto decode = [&](int tile, int &e, int &mt, int &nt) {
    if (GROUP_K) {
      e = tile / tiles_per_group_k;
      const int local = tile - e * tiles_per_group_k;
      mt = local / n_tiles;
      nt = local - mt * n_tiles;
    } else {
      e = find_group(s.tile_start, E, tile);
      const int local = tile - s.tile_start[e];
      const int m_tiles = (s.tile_start[e + 1] - s.tile_start[e]) / n_tiles;
      nt = local / m_tiles;
      mt = local - nt * m_tiles;
    }
  };
  // Short tiles (grouped-M, one CTA per tile): an m-tile holding at most 64 of
  // its group's rows runs M = 64 MMAs, which write tile row 16 q + i to TMEM
  // lane 32 q + i (i < 16) of lane quarter q.
  auto short_tile = [&](int e, int mt) -> bool {
    if (GROUP_K || PAIR || !p.m64) return false;
    const int rem = off(e + 1) - off(e) - mt * BM;
    return rem > 0 && rem <= 64;
  };
  auto k_steps = [&](int e) -> int {
    return GROUP_K ? (off(e + 1) - off(e) + BK - 1) / BK : (p.K + BK - 1) / BK;
  };
  // Grouped-K: the last K step of a group may run past its rows. Only the
  // K16 slices holding group rows are issued (returned), and the rows past
  // the group inside the last of them are zeroed in this CTA's A and B blocks
  // (each row is one 128-byte line per 64-wide block) by the calling warp.
  auto trim_last_step = [&](uint8_t *a_s, int e, int ks, bool &zeroed) -> int {
    int nkk = BK / 16;
    zeroed = false;
    if (GROUP_K) {
      const int valid = off(e + 1) - (off(e) + ks * BK);
      if (valid < BK) {
        nkk = (valid + 15) >> 4;
        const int nrows = nkk * 16 - valid;
        zeroed = nrows > 0;
        if (nrows > 0) {
          constexpr int NBLK = SB / 8192;  // 64-wide blocks of A and B in the stage
          const int chunks = nrows * 8;    // 16-byte chunks per block (rows valid .. valid + nrows - 1)
          uint8_t *z0 = a_s + valid * 128;
#pragma unroll
          for (int blk = 0; blk < NBLK; ++blk)
            for (int i = lane; i < chunks; i += 32)
              *reinterpret_cast<uint4 *>(z0 + blk * 8192 + (i >> 3) * 128 + (i & 7) * 16) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
        }
        __syncwarp();
      }
    }
    return nkk;
  };

  // Tile order. Static: unit, unit + units, ... Dynamic (one CTA per tile,
  // p.sched given): the producer takes the next index from the global
  // counter as it starts each tile (one fetch ahead) and publishes it in the
  // tile queue; the MMA and epilogue warps read the same sequence from the
  // queue. A CTA whose producer has fetched past the end counts itself
  // finished; the last one resets both counters for the next launch.
  const bool dyn = !PAIR && p.sched != nullptr;
  // Tail split (grouped-M, one CTA per tile, fixed order; not the SwiGLU
  // forward, whose tile pairs gate and up columns): when a launch has fewer
  // than four waves of tiles and its last partial wave holds at most half as
  // many tiles as there are CTAs, each tile of that wave is cut along N into
  // 2 (or, at most a quarter, 4) column windows of 128 (64) columns, so that
  // more CTAs share the wave. A window's MMAs write its columns of the
  // accumulator (N = window width) and the epilogue stores only those; the
  // other work units are whole tiles. (With many waves the last one weighs
  // little, and a window re-reads its tile's whole A rows.)
  int tail = 0, split = 1;
  if (!GROUP_K && !PAIR && !SWIGLU_FWD && !dyn && p.tail_split && total_tiles < 4 * units) {
    tail = total_tiles % units;
    if (tail > 0 && 2 * tail <= units) split = 4 * tail <= units ? 4 : 2;
    else tail = 0;
  }
  const int total_units = total_tiles + (split - 1) * tail;
  // work unit -> (tile, first column of the window inside the tile, window width)
  auto unit_of = [&](int w, int &tile, int &c_off, int &width) {
    const int nfull = total_tiles - tail;
    if (w < nfull) {
      tile = w;
      c_off = 0;
      width = BN;
    } else {
      const int j = w - nfull;
      tile = nfull + j / split;
      width = BN / split;
      c_off = (j - (j / split) * split) * width;
    }
  };
  struct TileIter {
    int next, q;
    uint32_t ph;
  };
  // consumers (MMA warp, epilogue warps): the next tile, -1 when there are no more, -2 on abort
  auto consumer_next = [&](TileIter &it) -> int {
    if (!dyn) {
      const int t = it.next;
      it.next += units;
      return t < total_units ? t : -1;
    }
    if (!mbar_wait_bounded(&s.tq_full[it.q], it.ph, abort_flag, p.st)) return -2;
    const int t = *reinterpret_cast<volatile int *>(&s.tile_q[it.q]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.tq_empty[it.q]);
    if (++it.q == TQ) { it.q = 0; it.ph ^= 1; }
    return t;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Lane 0 waits for free stages and issues this CTA's tile loads.
    const uint64_t pol_a = policy_evict_last();
    // Weight tiles that no other m-tile will read are streamed (evict-first);
    // when groups span several m-tiles they are kept for the other m-tiles.
    const uint64_t pol_b = (!GROUP_K && p.b_once) ? policy_evict_first() : policy_evict_last();
    // DIRECT, odd CTA: the even CTA's stage barriers (cluster addresses)
    const uint32_t lead_full0 = DIRECT ? mapa_shared(smem_u32(&s.full[0]), 0) : 0u;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    TileIter it{unit0, 0, 0};
    int fetched = 0;   // dynamic: lane 0's prefetched index
    if (dyn && lane == 0) fetched = (int)atomicAdd(p.sched, 1u);
    while (ok) {
      int tile;
      if (dyn) {
        tile = __shfl_sync(0xffffffffu, fetched, 0);
        int pub = 1;
        if (lane == 0) {
          pub = mbar_wait_bounded(&s.tq_empty[it.q], it.ph ^ 1, abort_flag, p.st) ? 1 : 0;
          if (pub) {
            s.tile_q[it.q] = tile < total_tiles ? tile : -1;
            mbar_arrive(&s.tq_full[it.q]);
          }
        }
        if (!__shfl_sync(0xffffffffu, pub, 0)) { ok = false; break; }
        if (++it.q == TQ) { it.q = 0; it.ph ^= 1; }
        if (tile >= total_tiles) break;
        if (lane == 0) fetched = (int)atomicAdd(p.sched, 1u);   // the next tile, fetched ahead of its use
      } else {
        tile = it.next;
        it.next += units;
        if (tile >= total_units) break;
      }
      int e, mt, nt, c_off, width;
      unit_of(tile, tile, c_off, width);
      decode(tile, e, mt, nt);
      const int nk = k_steps(e);
      // bytes of one stage: A, and B for the window (K-major B: 128-row boxes; MN-major: 64-column boxes).
      // With K-major B, A comes in 64-row boxes and a short tile loads one; with MN-major B (already four
      // boxes a stage) in one 128-row box (measured: the extra box slowed dH by 5%).
      constexpr bool A64 = !GROUP_K && !B_MN;
      const bool a_half = A64 && short_tile(e, mt);
      const uint32_t stage_tx = (width == BN ? (uint32_t)(DIRECT ? 2 * SB : SB)
                                             : (uint32_t)(A_BYTES + (B_MN ? (width / 64) * 8192 : 16384))) -
                                (a_half ? (uint32_t)(A_BYTES / 2) : 0u);
      for (int ks = 0; ks < nk; ++ks) {
        int got = 1;
        if (lane == 0) got = mbar_wait_bounded(&s.empty[stage], phase ^ 1, abort_flag, p.st) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        uint8_t *a_s = tiles + (size_t)stage * SB;
        uint8_t *b_s = a_s + A_BYTES;
        // DIRECT: the even CTA expects both halves' bytes; the odd CTA only loads
        if (lane == 0 && !(DIRECT && crank)) mbar_arrive_expect_tx(&s.full[stage], stage_tx);
        __syncwarp();
        const int k0 = ks * BK;
        if (lane == 0) {
          if (!GROUP_K) {
            const uint32_t fb = lead_full0 + 8u * (uint32_t)stage;
            auto ld2 = [&](void *dst, const CUtensorMap *m, int c0, int c1, uint64_t pol) {
              if (DIRECT && crank) tma_load_2d_pair(dst, m, fb, c0, c1, pol);
              else tma_load_2d(dst, m, &s.full[stage], c0, c1, pol);
            };
            auto ld3 = [&](void *dst, const CUtensorMap *m, int c0, int c1, int c2, uint64_t pol) {
              if (DIRECT && crank) tma_load_3d_pair(dst, m, fb, c0, c1, c2, pol);
              else tma_load_3d(dst, m, &s.full[stage], c0, c1, c2, pol);
            };
            const int row0 = off(e) + mt * TM + half_row;
            ld2(a_s, &tmA, k0, row0, pol_a);
            if (A64 && !a_half) ld2(a_s + 8192, &tmA, k0, row0 + 64, pol_a);   // A64: the second 64-row box
            if (!B_MN) {
              // B rows of the tile: 128 per CTA of a pair, 256 (two boxes) otherwise
              int r0, r1;
              if (SWIGLU_FWD) { r0 = nt * 128; r1 = p.F + nt * 128; }
              else { r0 = nt * BN + c_off; r1 = nt * BN + 128; }
              if (PAIR) {
                ld3(b_s, &tmB, k0, crank ? r1 : r0, e, pol_b);
              } else {
                ld3(b_s, &tmB, k0, r0, e, pol_b);   // (a narrower window: its first rows of this box)
                if (width == BN) ld3(b_s + 16384, &tmB, k0, r1, e, pol_b);
              }
            } else {
              const int c0 = nt * BN + (PAIR ? crank * 128 : c_off);
              const int nb = PAIR ? 2 : width / 64;
              for (int j = 0; j < nb; ++j) ld3(b_s + j * 8192, &tmB, c0 + 64 * j, k0, e, pol_b);
            }
          } else {
            const int r0 = off(e) + k0;
            const int m0 = mt * TM + half_row;
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_2d(a_s + j * 8192, &tmA, &s.full[stage], m0 + 64 * j, r0, pol_a);
            const int c0 = nt * BN + (PAIR ? crank * 128 : 0);
#pragma unroll
            for (int j = 0; j < (PAIR ? 2 : 4); ++j)
              tma_load_2d(b_s + j * 8192, &tmB, &s.full[stage], c0 + 64 * j, r0, pol_b);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
    }
    // dynamic tiles: the last CTA whose producer is done resets the counters
    if (dyn && ok && lane == 0 && atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      p.sched[0] = 0u;
      p.sched[1] = 0u;
    }
    // (DIRECT, odd CTA: its bytes complete on the even CTA's barriers, which
    // that CTA drains)
    if (lane == 0 && *abort_flag && !(DIRECT && crank)) {
      for (int i = 0; i < NST; ++i)
        if (issued & (1u << i)) drain_wait(&s.full[i], (issued_parity >> i) & 1);
    }
    __syncwarp();
  } else if (warp == 1 && crank == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC = idesc_bf16_f32(TM, BN, A_MN, B_MN);
    constexpr uint32_t IDESC_128 = idesc_bf16_f32(TM, 128, A_MN, B_MN);   // tail windows
    constexpr uint32_t IDESC_64 = idesc_bf16_f32(TM, 64, A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    TileIter it{unit0, 0, 0};
    while (ok) {
      int tile = consumer_next(it);
      if (tile < 0) { ok = tile == -1; break; }
      int e, mt, nt, c_off, width;
      unit_of(tile, tile, c_off, width);
      decode(tile, e, mt, nt);
      const int nk = k_steps(e);
      const bool m64 = short_tile(e, mt);
      uint32_t idesc = width == BN ? IDESC : (width == 128 ? IDESC_128 : IDESC_64);
      if (m64) idesc = (idesc & ~(0x1Fu << 24)) | ((uint32_t)(64 >> 4) << 24);   // M = 64
      if (!mbar_wait_bounded<PAIR != 0>(&s.acc_empty[acc], acc_phase ^ 1, abort_flag, p.st)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * BN + c_off);   // a window: its columns of the accumulator
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait_bounded(&s.full[stage], phase, abort_flag, p.st)) { ok = false; break; }
        uint8_t *a_s = tiles + (size_t)stage * SB;
        uint8_t *b_s = a_s + A_BYTES;
        bool zeroed;
        const int nkk = trim_last_step(a_s, e, ks, zeroed);
        if (PAIR && !DIRECT && !mbar_wait_bounded<true>(&s.peer_full[stage], phase, abort_flag, p.st)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(a_s), b0 = smem_u32(b_s);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nkk) break;
            const uint64_t ad = A_MN ? smem_desc_sw128(a0 + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(b0 + kk * 32, 16, 1024);
            if (PAIR) tc_mma_bf16_pair(d_tmem, ad, bd, IDESC, (ks > 0 || kk > 0) ? 1u : 0u);
            else tc_mma_bf16(d_tmem, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          if (PAIR) tc_commit_pair_mc(&s.empty[stage], 0x3);
          else tc_commit(&s.empty[stage]);
        }
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) {
        if (PAIR) tc_commit_pair_mc(&s.acc_full[acc], 0x3);
        else tc_commit(&s.acc_full[acc]);
      }
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (*abort_flag) {
      if (lane == 0) {
        if (PAIR) tc_commit_pair(&s.drain);
        else tc_commit(&s.drain);
      }
      __syncwarp();
      drain_wait(&s.drain, 0);
    }
  } else if (warp == 1 && !DIRECT) {
    // ---------------------------------------------------------------- grouped-K pair tiles, odd CTA
    // Forwards each stage to the even CTA once this CTA's half has landed
    // (and, in the last K step of a group, its rows past the group are zeroed:
    // then with release ordering, for those generic writes).
    const uint32_t peer_full0 = mapa_shared(smem_u32(&s.peer_full[0]), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = unit0; ok && tile < total_tiles; tile += units) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int nk = k_steps(e);
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait_bounded(&s.full[stage], phase, abort_flag, p.st)) { ok = false; break; }
        bool zeroed;
        trim_last_step(tiles + (size_t)stage * SB, e, ks, zeroed);
        if (lane == 0) {
          if (zeroed) mbar_arrive_cluster(peer_full0 + 8u * (uint32_t)stage);
          else mbar_arrive_cluster_relaxed(peer_full0 + 8u * (uint32_t)stage);
        }
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    // Two warps per TMEM lane quarter: warp w reads lanes 32 (w % 4) .. + 31
    // (its rows) and the column half (w - 2) / 4 of the tile.
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;  // column half of the tile
    // the accumulator's release goes to the MMA issuer's CTA (rank 0 of a pair)
    const uint32_t acc_empty0 = PAIR ? mapa_shared(smem_u32(&s.acc_empty[0]), 0) : 0u;
    int acc = 0;
    uint32_t acc_phase = 0;
    TileIter it{unit0, 0, 0};
    while (true) {
      int tile = consumer_next(it);
      if (tile < 0) break;
      int e, mt, nt, c_off, width;
      unit_of(tile, tile, c_off, width);
      decode(tile, e, mt, nt);
      // output columns of this unit: [cs, ce) (the whole tile, or a tail window)
      const int cs = nt * BN + c_off, ce = cs + width;
      // this lane's row of the tile and the warp's slice (32 rows; a short tile: 16 rows in lanes 0-15)
      const bool m64 = short_tile(e, mt);
      const int r = m64 ? (lane < 16 ? 16 * q + lane : 1 << 20) : q * 32 + lane;
      const int slice0 = m64 ? 16 * q : 32 * q, slice_n = m64 ? 16 : 32;
      if (!mbar_wait_bounded<PAIR != 0>(&s.acc_full[acc], acc_phase, abort_flag, p.st)) break;
      tc_fence_after();
      const uint32_t t_row = tmem + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      const int mrow0 = mt * TM + half_row;  // this CTA's first row of the tile (group- or M-relative)
      float v[32], w[32];
      bool released = false;  // the accumulator handed back to the MMA warp
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR) mbar_arrive_cluster(acc_empty0 + 8u * (uint32_t)acc);
          else mbar_arrive(&s.acc_empty[acc]);
        }
        released = true;
      };
      if (TMA_STORE) {
        // This warp's 32-row slice: whole slices go through the staging buffer
        // and a TMA store; a slice cut by the end of its group (grouped-M) is
        // stored row by row, so the next group's rows are never touched.
        constexpr bool F32 = (EPI == EPI_STORE_F32);
        constexpr int CPB = F32 ? 1 : 2;  // 32-column chunks per 128-byte staging row
        uint8_t *stg = stage_out + (warp - 2) * SPW;
        int nvalid = 32;
        int r0;
        const bool zero = GROUP_K && off(e + 1) == off(e);
        if (!GROUP_K) {
          const int lo = mrow0 + slice0;
          nvalid = min(slice_n, max(0, off(e + 1) - off(e) - lo));
          r0 = off(e) + lo;
        } else {
          r0 = mrow0 + q * 32;
        }
        // the warp's four 32-column pieces in flight together, then the
        // accumulator goes back to the MMA warp before any store
        uint32_t xr[4][32];
        if (!zero && nvalid > 0) {
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_ld32_issue(t_row + (4 * half + u) * 32, xr[u]);
#pragma unroll
          for (int u = 0; u < 4; ++u) tmem_wait32(xr[u]);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < 32; ++i) xr[u][i] = 0u;
        }
        release_acc();
#pragma unroll
        for (int cu = 0; cu < 4; cu += CPB) {
          const int c = 4 * half + cu;
          const int col = nt * BN + c * 32;
          if (nvalid == 0 || col >= p.N || col < cs || col >= ce) continue;
          float x[32 * CPB];
#pragma unroll
          for (int u = 0; u < CPB; ++u)
#pragma unroll
            for (int i = 0; i < 32; ++i) x[32 * u + i] = __uint_as_float(xr[cu + u][i]);
          if (nvalid == 32) {
            if (lane == 0) bulk_wait_read_all();  // the previous store has left the buffer
            __syncwarp();
            uint8_t *rowp = stg + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint8_t *dst = rowp + ((j ^ (lane & 7)) << 4);
              if (F32) Vec16<float>::store(dst, x + 4 * j);
              else Vec16<bf16>::store(dst, x + 8 * j);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (GROUP_K) tma_store_3d(&tmC, stg, col, r0, e);
              else tma_store_2d(&tmC, stg, col, r0);
              bulk_commit();
            }
          } else if (lane < nvalid) {
            const int64_t row = (int64_t)r0 + lane;
            if (F32) {
              float *cp = static_cast<float *>(p.C) + row * p.ldc + col;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (col + 4 * i < p.N) Vec16<float>::store(cp + 4 * i, x + 4 * i);
            } else {
              bf16 *cp = static_cast<bf16 *>(p.C) + row * p.ldc + col;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (col + 8 * i < p.N) Vec16<bf16>::store(cp + 8 * i, x + 8 * i);
            }
          }
        }
      } else if (!GROUP_K) {
        const int rows_e = off(e + 1) - off(e);
        const bool valid = mrow0 + r < rows_e;
        const int64_t row = (int64_t)off(e) + mrow0 + r;
        if (EPI == EPI_SWIGLU) {
          // This warp's 32-row slice and 64 output columns [col0, col0 + 64):
          // h = silu(G) U and, when saved, the pre-activations G and U. A whole
          // slice goes through the staging buffer (128-byte swizzled rows,
          // reused for h, G and U in turn) and one TMA tile store each; a
          // slice cut by the end of its group is stored row by row, so the
          // next group's rows are never touched. Accumulator columns: G at
          // [c 32, + 32), U at 128 + [c 32, + 32) for the warp's chunks c.
          const int col0 = nt * 128 + half * 64;
          const int lo = mrow0 + slice0;
          const int nvalid = min(slice_n, max(0, rows_e - lo));
          if (nvalid == 32 && col0 < p.N) {
            uint8_t *stg = stage_out + (warp - 2) * SPW;
            uint8_t *rowp = stg + lane * 128;
            const int r0 = off(e) + lo;
            const int nout = p.C2 ? 3 : 1;
#pragma unroll 1
            for (int o = 0; o < nout; ++o) {  // 0: h, 1: G, 2: U
              if (lane == 0) bulk_wait_read_all();  // the previous store has left the buffer
              __syncwarp();
#pragma unroll 1
              for (int c = 0; c < 2; ++c) {
                const int cc = 2 * half + c;
                if (o == 0) {
                  tmem_ld32(t_row + cc * 32, v);
                  tmem_ld32(t_row + 128 + cc * 32, w);
#pragma unroll
                  for (int i = 0; i < 32; ++i) v[i] = silu_f(v[i]) * w[i];
                } else {
                  tmem_ld32(t_row + (o - 1) * 128 + cc * 32, v);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  Vec16<bf16>::store(rowp + (((c * 4 + j) ^ (lane & 7)) << 4), v + 8 * j);
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (o == 0) tma_store_2d(&tmC, stg, col0, r0);
                else tma_store_2d(o == 1 ? &tmD : &tmE, stg, col0, r0);
                bulk_commit();
              }
            }
          } else if (nvalid > 0) {
#pragma unroll 1
            for (int c = 2 * half; c < 2 * half + 2; ++c) {
              const int col = nt * 128 + c * 32;
              tmem_ld32(t_row + c * 32, v);
              tmem_ld32(t_row + 128 + c * 32, w);
              if (valid && col < p.N) {
                float hv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) hv[i] = silu_f(v[i]) * w[i];
                bf16 *hp = static_cast<bf16 *>(p.C) + row * p.ldc + col;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (col + 8 * i < p.N) Vec16<bf16>::store(hp + 8 * i, hv + 8 * i);
                if (p.C2) {
                  bf16 *gp = p.C2 + row * p.ldc2 + col;
                  bf16 *up = gp + p.F;
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    if (col + 8 * i >= p.N) continue;
                    Vec16<bf16>::store(gp + 8 * i, v + 8 * i);
                    Vec16<bf16>::store(up + 8 * i, w + 8 * i);
                  }
                }
              }
            }
          }
        } else if (EPI == EPI_RELU && !m64 && mrow0 + q * 32 + 32 <= rows_e) {
          // ReLU forward, whole 32-row slice: per 64-column group, h =
          // relu(acc) staged in 128-byte swizzled rows and written with one
          // TMA tile store.
          uint8_t *stg = stage_out + (warp - 2) * SPW;
          uint8_t *rowp = stg + lane * 128;
          const int r0 = off(e) + mrow0 + q * 32;
#pragma unroll 1
          for (int gi = 0; gi < 2; ++gi) {
            const int col0 = nt * BN + half * 128 + gi * 64;
            if (col0 >= p.N) break;
            if (col0 < cs || col0 >= ce) continue;
            if (lane == 0) bulk_wait_read_all();  // the previous store has left the buffer
            __syncwarp();
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
              tmem_ld32(t_row + (half * 4 + gi * 2 + c) * 32, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.0f);
#pragma unroll
              for (int j = 0; j < 4; ++j) Vec16<bf16>::store(rowp + (((c * 4 + j) ^ (lane & 7)) << 4), v + 8 * j);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, stg, col0, r0);
              bulk_commit();
            }
          }
        } else if (EPI == EPI_SWIGLU_BWD && !m64 && mrow0 + q * 32 + 32 <= rows_e) {
          // SwiGLU backward, whole 32-row slice, per 32-column group: the
          // slice's saved G and U are read with coalesced 16-byte loads (4
          // lanes per 64-byte row piece, all 8 loads of a lane in flight
          // together: 4 of G, 4 of U) into this warp's two 2 KB halves (64-byte rows, 16-byte
          // units permuted by bits 7-8 of the address, as the 64-byte-swizzle
          // maps write them). Each lane then takes its row's G and U from
          // them, forms dG = dH U silu'(G) and dU = dH silu(G) in place, and
          // the two halves go out as TMA tile stores into dA = [dG | dU].
          uint8_t *bg = stage_out + (warp - 2) * SPW;  // G, then dG
          uint8_t *bu = bg + STAGE_OUT_BYTES / 2;      // U, then dU
          const int64_t rbase = (int64_t)off(e) + mrow0 + q * 32;
          const int piece = lane & 3;
#pragma unroll 1
          for (int gi = 0; gi < 4; ++gi) {
            const int col0 = nt * BN + half * 128 + gi * 32;
            if (col0 >= p.N) break;
            if (col0 < cs || col0 >= ce) continue;
            if (lane == 0) bulk_wait_read_all();  // the previous group's stores have left the halves
            __syncwarp();
            {
              uint4 lg[4], lu[4];
              const bool in_f = col0 + piece * 8 < p.F;   // columns past F: zeros (stores clip there)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rr = 8 * i + (lane >> 2);      // rows 0..31 of the slice
                const bf16 *src = p.aux + (rbase + rr) * p.ldaux + col0 + piece * 8;
                lg[i] = in_f ? *reinterpret_cast<const uint4 *>(src) : make_uint4(0u, 0u, 0u, 0u);
                lu[i] = in_f ? *reinterpret_cast<const uint4 *>(src + p.F) : make_uint4(0u, 0u, 0u, 0u);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int rr = 8 * i + (lane >> 2);
                const int o = rr * 64 + ((piece ^ ((rr >> 1) & 3)) << 4);
                *reinterpret_cast<uint4 *>(bg + o) = lg[i];
                *reinterpret_cast<uint4 *>(bu + o) = lu[i];
              }
            }
            __syncwarp();
            tmem_ld32(t_row + (half * 4 + gi) * 32, v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int o = lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4);
              float gg[8], uu[8], dgv[8], duv[8];
              Vec16<bf16>::load(bg + o, gg);
              Vec16<bf16>::load(bu + o, uu);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float sg = 1.0f / (1.0f + expf(-gg[j]));
                const float dh = v[8 * i + j];
                duv[j] = dh * gg[j] * sg;                                      // dU = dH * silu(G)
                dgv[j] = dh * uu[j] * (sg * (1.0f + gg[j] * (1.0f - sg)));     // dG = dH * U * silu'(G)
              }
              Vec16<bf16>::store(bg + o, dgv);
              Vec16<bf16>::store(bu + o, duv);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, bg, col0, (int)rbase);   // dG half of dA
              tma_store_2d(&tmD, bu, col0, (int)rbase);   // dU half of dA
              bulk_commit();
            }
          }
        } else {
          // The backward epilogues read saved activations; the loads of G
          // chunks are issued together before any of them is used.
          constexpr int NAUX = (EPI == EPI_SWIGLU_BWD) ? 8 : ((EPI == EPI_RELU_BWD || EPI == EPI_COMBINE) ? 4 : 0);
          constexpr int G = (EPI == EPI_SWIGLU_BWD) ? 1 : 4;  // (SwiGLU: only slices cut by a group end come here)
          // combine (top-1): the output and residual rows are the token's own
          int64_t orow = row;
          float gt = 0.0f;
          if (EPI == EPI_COMBINE && valid) {
            orow = __ldg(p.a_rows + row);
            gt = __ldg(p.gate + orow);
          }
#pragma unroll 1
          for (int c0 = 4 * half; c0 < 4 * half + 4; c0 += G) {
            uint4 aux[NAUX > 0 ? G * NAUX : 1];
            if (NAUX > 0) {
#pragma unroll
              for (int g = 0; g < G; ++g) {
                const int col = nt * BN + (c0 + g) * 32;
                if (valid && col < p.N) {
                  const bf16 *ap = p.aux + orow * p.ldaux + col;
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    aux[g * NAUX + i] = col + 8 * i < p.N ? *reinterpret_cast<const uint4 *>(ap + 8 * i)
                                                          : make_uint4(0u, 0u, 0u, 0u);
                  if (EPI == EPI_SWIGLU_BWD) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                      aux[g * NAUX + 4 + i] = col + 8 * i < p.N ? *reinterpret_cast<const uint4 *>(ap + p.F + 8 * i)
                                                                : make_uint4(0u, 0u, 0u, 0u);
                  }
                }
              }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const int col = nt * BN + (c0 + g) * 32;
              tmem_ld32(t_row + (c0 + g) * 32, v);
              if (!valid || col >= p.N || col < cs || col >= ce) continue;
              if (EPI == EPI_RELU) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.0f);
              } else if (EPI == EPI_COMBINE) {
#pragma unroll
                for (int i = 0; i < 4; ++i) Vec16<bf16>::unpack(aux[g * NAUX + i], w + 8 * i);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = p.residual ? fmaf(gt, v[i], w[i]) : gt * v[i];   // out = x + g y
              } else if (EPI == EPI_RELU_BWD) {
#pragma unroll
                for (int i = 0; i < 4; ++i) Vec16<bf16>::unpack(aux[g * NAUX + i], w + 8 * i);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = (w[i] > 0.0f) ? v[i] : 0.0f;
              } else if (EPI == EPI_SWIGLU_BWD) {
                bf16 *dp2 = static_cast<bf16 *>(p.C) + row * p.ldc + p.F + col;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  float gg[8], uu[8], du[8];
                  Vec16<bf16>::unpack(aux[g * NAUX + i], gg);
                  Vec16<bf16>::unpack(aux[g * NAUX + 4 + i], uu);
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    const float sg = 1.0f / (1.0f + expf(-gg[j]));
                    const float dh = v[8 * i + j];
                    du[j] = dh * gg[j] * sg;                                      // dU = dH * silu(G)
                    v[8 * i + j] = dh * uu[j] * (sg * (1.0f + gg[j] * (1.0f - sg)));  // dG = dH * U * silu'(G)
                  }
                  if (col + 8 * i < p.N) Vec16<bf16>::store(dp2 + 8 * i, du);
                }
              }
              if (EPI == EPI_STORE_F32) {
                float *cp = static_cast<float *>(p.C) + row * p.ldc + col;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  if (col + 4 * i < p.N) Vec16<float>::store(cp + 4 * i, v + 4 * i);
              } else {
                bf16 *cp = static_cast<bf16 *>(p.C) + orow * p.ldc + col;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (col + 8 * i < p.N) Vec16<bf16>::store(cp + 8 * i, v + 8 * i);
              }
            }
          }
        }
      } else {
        const bool empty_group = off(e + 1) == off(e);
        const int m = mrow0 + r;
        const int64_t cofs = (int64_t)e * p.sce + (int64_t)m * p.ldc;
#pragma unroll 1
        for (int c = 4 * half; c < 4 * half + 4; ++c) {
          const int col = nt * BN + c * 32;
          if (!empty_group) tmem_ld32(t_row + c * 32, v);
          else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
          if (m < p.M && col < p.N) {
            if (EPI == EPI_STORE_F32) {
              float *cp = static_cast<float *>(p.C) + cofs + col;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (col + 4 * i < p.N) Vec16<float>::store(cp + 4 * i, v + 4 * i);
            } else {
              bf16 *cp = static_cast<bf16 *>(p.C) + cofs + col;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (col + 8 * i < p.N) Vec16<bf16>::store(cp + 8 * i, v + 8 * i);
            }
          }
        }
      }
      if (!released) release_acc();
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (STAGED && lane == 0) bulk_wait_all();  // stores complete before the CTA exits
  }

  __syncthreads();
  // Pair tiles: neither CTA leaves while the other may still reach its shared
  // memory or TMEM (remote arrivals, the even CTA's MMAs).
  if (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
    else tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
// Persistent grid: one CTA per SM, or as many CTA pairs as can be resident
// at once (0 when no cluster of two fits).
template <int PAIR, int GROUP_K, int A_MN, int B_MN, int EPI>
static int grid_size() {
  static int grid = -1;
  if (grid >= 0) return grid;
  auto kern = grouped_gemm_kernel<PAIR, GROUP_K, A_MN, B_MN, EPI>;
  constexpr size_t smem = smem_bytes<PAIR, GROUP_K, EPI>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
  if (!PAIR) return grid = sm_count();
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count() & ~1);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, (const void *)kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    clusters = 0;
  }
  if (clusters > sm_count() / 2) clusters = sm_count() / 2;
  return grid = 2 * clusters;
}

// mc is the output's tile map for the plain-store epilogues (ignored otherwise).
// pair: CTA-pair tiles when a cluster of two fits, one CTA per tile otherwise.
// md: the second output map (SwiGLU forward: the pre-activations).
// Tile order of one-CTA-per-tile launches: the fixed stride (CTA u takes
// tiles u, u + grid, ...), or, with MOE_GEMM_SCHED=dynamic in the
// environment (read at every call), tiles handed out by a counter in the
// workspace as CTAs free up. Measured on the B300 (bench.py, static and
// dynamic back to back): no faster on any workload (the skewed GShard-style
// layer's GEMMs are held back by their last partial wave of tiles, not by
// uneven tile costs), and the short weight-gradient tiles of the large layer
// slower by the queue handshake, so the fixed stride is the default.
// Tail windows of the last partial wave (grouped-M, fixed order): on unless
// MOE_GEMM_TAIL=0 in the environment (read at every call).
static int tail_split_enabled() {
  const char *v = getenv("MOE_GEMM_TAIL");
  return (v && v[0] == '0') ? 0 : 1;
}
// M = 64 MMAs for grouped-M m-tiles with at most 64 rows: on unless
// MOE_GEMM_M64=0 in the environment (read at every call).
static int m64_enabled() {
  const char *v = getenv("MOE_GEMM_M64");
  return (v && v[0] == '0') ? 0 : 1;
}
static unsigned int *tile_counters(DeviceStatus *st) {
  const char *v = getenv("MOE_GEMM_SCHED");
  if (!(v && v[0] == 'd')) return nullptr;
  return reinterpret_cast<unsigned int *>(reinterpret_cast<uint8_t *>(st) + kGemmSchedOffset);
}

template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch(bool pair, const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                          const CUtensorMap &md, const CUtensorMap &me, const Args &a, cudaStream_t stream) {
  Args args = a;
  if (pair) {
    const int g = grid_size<1, GROUP_K, A_MN, B_MN, EPI>();
    args.sched = nullptr;   // pair tiles keep the fixed order
    if (g > 0)
      return launch_kernel_cluster(grouped_gemm_kernel<1, GROUP_K, A_MN, B_MN, EPI>, 2, dim3(g), dim3(THREADS),
                                   smem_bytes<1, GROUP_K, EPI>(), stream, ma, mb, mc, md, me, args);
  }
  const int g = grid_size<0, GROUP_K, A_MN, B_MN, EPI>();
  if (g <= 0) return cudaErrorInvalidConfiguration;
  args.sched = tile_counters(a.st);
  args.tail_split = tail_split_enabled();
  args.m64 = m64_enabled();
  return launch_kernel(grouped_gemm_kernel<0, GROUP_K, A_MN, B_MN, EPI>, dim3(g), dim3(THREADS),
                       smem_bytes<0, GROUP_K, EPI>(), stream, ma, mb, mc, md, me, args);
}
template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch(bool pair, const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                          const CUtensorMap &md, const Args &a, cudaStream_t stream) {
  static_assert(EPI != EPI_SWIGLU, "the SwiGLU forward epilogue needs the G and U maps");
  return launch<GROUP_K, A_MN, B_MN, EPI>(pair, ma, mb, mc, md, md, a, stream);
}
template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch(bool pair, const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                          const Args &a, cudaStream_t stream) {
  static_assert(EPI != EPI_SWIGLU && EPI != EPI_SWIGLU_BWD, "the SwiGLU epilogues need their second map");
  return launch<GROUP_K, A_MN, B_MN, EPI>(pair, ma, mb, mc, mc, mc, a, stream);
}
template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch(bool pair, const CUtensorMap &ma, const CUtensorMap &mb, const Args &a,
                          cudaStream_t stream) {
  static_assert(!staged_epi<EPI>(), "staged epilogues need the output map");
  return launch<GROUP_K, A_MN, B_MN, EPI>(pair, ma, mb, ma, ma, ma, a, stream);
}
// One CTA per tile only (shapes whose M is not a multiple of a pair tile).
template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch_single(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                                 const Args &a, cudaStream_t stream) {
  const int g = grid_size<0, GROUP_K, A_MN, B_MN, EPI>();
  if (g <= 0) return cudaErrorInvalidConfiguration;
  Args args = a;
  args.sched = tile_counters(a.st);
  args.tail_split = tail_split_enabled();
  args.m64 = m64_enabled();
  return launch_kernel(grouped_gemm_kernel<0, GROUP_K, A_MN, B_MN, EPI>, dim3(g), dim3(THREADS),
                       smem_bytes<0, GROUP_K, EPI>(), stream, ma, mb, mc, mc, mc, args);
}

}  // namespace tc

// ---------------------------------------------------------------- launchers used by the C ABI
// CTA-pair tiles (256 rows) or one CTA per tile (128 rows). Pair tiles are
// opt-in: MOE_GEMM_PAIR=1 in the environment selects them for every expert
// GEMM (grouped-M and grouped-K), anything else or unset keeps one CTA per
// tile. Measured on the B300: equal speed on the tensor-bound grouped-M
// GEMMs (the per-SM operand bytes per MMA do not change, half of B arrives
// from the peer's shared memory), slower on the HBM-bound layers and on
// grouped-K, whose odd CTA forwards every stage.
static bool pair_tiles() {
  const char *v = getenv("MOE_GEMM_PAIR");
  return v && v[0] == '1';
}
static bool pair_grouped_m(const Shape &) { return pair_tiles(); }
static bool pair_grouped_k(int) { return pair_tiles(); }

// True when the capacity keeps every group within one m-tile (128 rows, 256
// for pair tiles), so that each weight tile is read by a single m-tile.
static int weights_read_once(const Shape &sh, bool pair) {
  return (sh.C >= 0 && sh.C <= (pair ? 2 : 1) * tc::BM) ? 1 : 0;
}

// GEMM 1 with its activation epilogue (a.C = h, a.C2 = SwiGLU pre-activations
// or null). The epilogues write h (and the pre-activations) through TMA tile
// stores: output maps with 64-column x 32-row boxes.
static cudaError_t gemm1_act(const Shape &sh, bool pair, const CUtensorMap &ma, const CUtensorMap &mb,
                             const tc::Args &a, uint64_t rows, cudaStream_t stream) {
  using namespace tc;
  CUtensorMap mc, md, me;
  if (!make_map_2d(&mc, a.C, sh.F, rows, 64, 32)) return cudaErrorInvalidValue;
  if (sh.act != MOE_ACT_SWIGLU) return launch<0, 0, 0, EPI_RELU>(pair, ma, mb, mc, a, stream);
  if (a.C2 != nullptr) {
    // G and U, each F wide, in the two halves of each 2F-wide pre-activation row
    const uint64_t stride = 2 * (uint64_t)sh.F * 2;
    if (!make_map_2d_strided(&md, a.C2, sh.F, rows, stride, 64, 32) ||
        !make_map_2d_strided(&me, a.C2 + sh.F, sh.F, rows, stride, 64, 32))
      return cudaErrorInvalidValue;
  } else {
    md = me = mc;
  }
  return launch<0, 0, 0, EPI_SWIGLU>(pair, ma, mb, mc, md, me, a, stream);
}

cudaError_t tc_expert_forward(const Shape &sh, const void *x_perm, const int32_t *offsets, const void *w1,
                              const void *w2, void *pre_act, void *h, void *y_perm, DeviceStatus *st,
                              cudaStream_t stream) {
  using namespace tc;
  CUtensorMap ma, mb;
  const uint64_t rows = sh.rows > 0 ? (uint64_t)sh.rows : 1;  // a map needs at least one row
  const bool pair = pair_grouped_m(sh);
  const int b_once = weights_read_once(sh, pair);
  Args a{};
  a.offsets = offsets;
  a.E = sh.E;
  a.F = sh.F;
  a.st = st;
  a.b_once = b_once;
  // GEMM 1 (+ activation): A = x_perm [rows, d], B = W1 [E, R1, d]
  if (!make_map_2d(&ma, x_perm, sh.d, rows, 64, 64) || !make_map_3d(&mb, w1, sh.d, sh.R1, sh.E, 64, 128))
    return cudaErrorInvalidValue;
  a.N = sh.F;
  a.K = sh.d;
  a.C = h;
  a.ldc = sh.F;
  a.C2 = (bf16 *)pre_act;
  a.ldc2 = 2 * (int64_t)sh.F;
  cudaError_t err = gemm1_act(sh, pair, ma, mb, a, rows, stream);
  if (err != cudaSuccess) return err;
  // GEMM 2: A = h [rows, F], B = W2 [E, d, F]
  if (!make_map_2d(&ma, h, sh.F, rows, 64, 64) || !make_map_3d(&mb, w2, sh.F, sh.d, sh.E, 64, 128))
    return cudaErrorInvalidValue;
  Args b{};
  b.offsets = offsets;
  b.E = sh.E;
  b.F = sh.F;
  b.st = st;
  b.b_once = b_once;
  b.N = sh.d;
  b.K = sh.F;
  b.C = y_perm;
  b.ldc = sh.d;
  CUtensorMap mc;
  if (!make_map_2d(&mc, y_perm, sh.d, rows, 64, 32)) return cudaErrorInvalidValue;
  return launch<0, 0, 0, EPI_STORE>(pair, ma, mb, mc, b, stream);
}

int router_grad_splits(const Shape &sh) {
  const int ep = sh.E <= 32 ? 32 : sh.E <= 64 ? 64 : sh.E <= 128 ? 128 : 256;
  const int tiles = ((3 * ep + tc::BM - 1) / tc::BM) * ((sh.d + tc::BN - 1) / tc::BN);
  int g = (sm_count() + tiles - 1) / tiles;
  const int most = sh.T / 512 > 1 ? sh.T / 512 : 1;  // at least 512 tokens per range
  if (g > most) g = most;
  if (g > 64) g = 64;
  return g < 1 ? 1 : g;
}

// Forward expert FFNs whose second GEMM, for top-1 layers, combines in its
// epilogue: out[t] = x[t] + g[t] * y for the row's token t (no y_perm). For
// k > 1 the second GEMM writes y_perm and the caller combines.
cudaError_t tc_expert_forward_combine(const Shape &sh, const void *x, const void *x_perm, const int32_t *row_token,
                                      const int32_t *offsets, const void *w1, const void *w2, void *h,
                                      const float *gate, void *out, void *y_perm, DeviceStatus *st,
                                      cudaStream_t stream) {
  using namespace tc;
  if (sh.k != 1) return tc_expert_forward(sh, x_perm, offsets, w1, w2, nullptr, h, y_perm, st, stream);
  CUtensorMap ma, mb;
  const uint64_t rows = sh.rows > 0 ? (uint64_t)sh.rows : 1;
  const bool pair = pair_grouped_m(sh);
  const int b_once = weights_read_once(sh, pair);
  Args a{};
  a.offsets = offsets;
  a.E = sh.E;
  a.F = sh.F;
  a.st = st;
  a.b_once = b_once;
  // GEMM 1 (+ activation): A = x_perm [rows, d], B = W1 [E, R1, d]
  if (!make_map_2d(&ma, x_perm, sh.d, rows, 64, 64) || !make_map_3d(&mb, w1, sh.d, sh.R1, sh.E, 64, 128))
    return cudaErrorInvalidValue;
  a.N = sh.F;
  a.K = sh.d;
  a.C = h;
  a.ldc = sh.F;
  cudaError_t err = gemm1_act(sh, pair, ma, mb, a, rows, stream);
  if (err != cudaSuccess) return err;
  // GEMM 2 + combine: A = h [rows, F], B = W2 [E, d, F]
  if (!make_map_2d(&ma, h, sh.F, rows, 64, 64) || !make_map_3d(&mb, w2, sh.F, sh.d, sh.E, 64, 128))
    return cudaErrorInvalidValue;
  Args b{};
  b.offsets = offsets;
  b.E = sh.E;
  b.F = sh.F;
  b.st = st;
  b.b_once = b_once;
  b.N = sh.d;
  b.K = sh.F;
  b.ldc = sh.d;
  b.C = out;
  b.aux = (const bf16 *)x;
  b.ldaux = sh.d;
  b.a_rows = row_token;
  b.gate = gate;
  b.residual = sh.residual;
  return launch<0, 0, 0, EPI_COMBINE>(pair, ma, mb, b, stream);
}

cudaError_t tc_expert_backward(const Shape &sh, const int32_t *offsets, const void *x_perm, const void *w1,
                               const void *w2, const void *pre_act, const void *h, const void *dyp, void *da,
                               void *dxp, void *dw1, void *dw2, DeviceStatus *st, cudaStream_t stream) {
  using namespace tc;
  CUtensorMap ma, mb;
  const uint64_t rows = sh.rows > 0 ? (uint64_t)sh.rows : 1;
  cudaError_t err;
  const bool swiglu = sh.act == MOE_ACT_SWIGLU;
  const bool pair = pair_grouped_m(sh);
  const int b_once = weights_read_once(sh, pair);
  // dH = dYp W2_e (B MN-major from W2 [E, d, F]), fused activation backward -> dA [rows, R1]
  {
    Args a{};
    a.offsets = offsets; a.E = sh.E; a.F = sh.F; a.st = st;
    a.N = sh.F; a.K = sh.d;
    a.C = da; a.ldc = sh.R1;
    a.b_once = b_once;
    if (!make_map_2d(&ma, dyp, sh.d, rows, 64, 128) || !make_map_3d(&mb, w2, sh.F, sh.d, sh.E, 64, 64))
      return cudaErrorInvalidValue;
    if (swiglu) {
      a.aux = (const bf16 *)pre_act; a.ldaux = 2 * (int64_t)sh.F;
      // dA [rows, 2F] = [dG | dU]: one map per F-wide half, 32-column x 32-row store boxes (64-byte swizzle)
      CUtensorMap mc, md;
      const uint64_t stride = 2 * (uint64_t)sh.F * 2;
      if (!make_map_2d_strided_sw64(&mc, da, sh.F, rows, stride, 32, 32) ||
          !make_map_2d_strided_sw64(&md, static_cast<bf16 *>(da) + sh.F, sh.F, rows, stride, 32, 32))
        return cudaErrorInvalidValue;
      err = launch<0, 0, 1, EPI_SWIGLU_BWD>(pair, ma, mb, mc, md, a, stream);
    } else {
      a.aux = (const bf16 *)h; a.ldaux = sh.F;
      err = launch<0, 0, 1, EPI_RELU_BWD>(pair, ma, mb, a, stream);
    }
    if (err != cudaSuccess) return err;
  }
  // Weight gradients: the unit-resident kernel when the capacity bounds the rows per expert (one CTA per
  // tile only; MOE_WGRAD=gemm in the environment selects the grouped GEMM below for them as well).
  const char *wv = getenv("MOE_WGRAD");
  const bool resident = wgrad_fits(sh) && !pair_grouped_k(sh.d) && !(wv && wv[0] == 'g');
  // dW2_e = dYp_e^T H_e   (grouped over K = rows of e): M = d, N = F
  if (resident) {
    err = launch_wgrad(sh, offsets, dyp, sh.d, h, sh.F, dw2, st, stream);
    if (err != cudaSuccess) return err;
  } else {
    Args a{};
    a.offsets = offsets; a.E = sh.E; a.F = sh.F; a.st = st;
    a.M = sh.d; a.N = sh.F;
    a.C = dw2; a.ldc = sh.F; a.sce = (int64_t)sh.d * sh.F;
    CUtensorMap mc;
    if (!make_map_2d(&ma, dyp, sh.d, rows, 64, 64) || !make_map_2d(&mb, h, sh.F, rows, 64, 64) ||
        !make_map_3d(&mc, dw2, sh.F, sh.d, sh.E, 64, 32))
      return cudaErrorInvalidValue;
    err = launch<1, 1, 1, EPI_STORE>(pair_grouped_k(a.M), ma, mb, mc, a, stream);
    if (err != cudaSuccess) return err;
  }
  // dXp = dA W1_e (B MN-major from W1 [E, R1, d]): N = d, K = R1
  {
    Args a{};
    a.offsets = offsets; a.E = sh.E; a.F = sh.F; a.st = st;
    a.N = sh.d; a.K = sh.R1;
    a.C = dxp; a.ldc = sh.d;
    a.b_once = b_once;
    CUtensorMap mc;
    if (!make_map_2d(&ma, da, sh.R1, rows, 64, 128) || !make_map_3d(&mb, w1, sh.d, sh.R1, sh.E, 64, 64) ||
        !make_map_2d(&mc, dxp, sh.d, rows, 64, 32))
      return cudaErrorInvalidValue;
    err = launch<0, 0, 1, EPI_STORE>(pair, ma, mb, mc, a, stream);
    if (err != cudaSuccess) return err;
  }
  // dW1_e = dA_e^T X_e: M = R1, N = d
  if (resident) {
    err = launch_wgrad(sh, offsets, da, sh.R1, x_perm, sh.d, dw1, st, stream);
  } else {
    Args a{};
    a.offsets = offsets; a.E = sh.E; a.F = sh.F; a.st = st;
    a.M = sh.R1; a.N = sh.d;
    a.C = dw1; a.ldc = sh.d; a.sce = (int64_t)sh.R1 * sh.d;
    CUtensorMap mc;
    if (!make_map_2d(&ma, da, sh.R1, rows, 64, 64) || !make_map_2d(&mb, x_perm, sh.d, rows, 64, 64) ||
        !make_map_3d(&mc, dw1, sh.d, sh.R1, sh.E, 64, 32))
      return cudaErrorInvalidValue;
    err = launch<1, 1, 1, EPI_STORE>(pair_grouped_k(a.M), ma, mb, mc, a, stream);
  }
  return err;
}

// Router gradient GEMMs of a bf16 layer on the tensor cores, from exact bf16
// parts (dh = h1 + h2 + h3, W_r = w1 + w2 + w3):
//   dXr [T, d] fp32 = A6 [T, 6EP] * B6 [6EP, d], where the six EP-wide blocks
//     pair (h1,w1) (h1,w2) (h2,w1) (h1,w3) (h2,w2) (h3,w1); the pairs left out
//     are below 2^-24 of the result;
//   C3 [3EP, d] fp32 = A6[:, 3EP:6EP]^T x, i.e. h1^T x, h2^T x and h3^T x
//     (x is bf16, so every product is exact), summed into dW_r afterwards.
// offs2 = {0, T}: dX_r runs as one group of T rows. dW_r is split over
// `splits` token ranges (offs_split, multiples of 64 rows) so that enough
// tiles run; range g writes its three part products to c3 + g [3EP, d].
cudaError_t tc_router_grads(const Shape &sh, int ep, const void *a6, const void *b6, const void *x,
                            const int32_t *offs2, const int32_t *offs_split, int splits, float *dxr, float *c3,
                            DeviceStatus *st, cudaStream_t stream) {
  using namespace tc;
  CUtensorMap ma, mb;
  cudaError_t err;
  {
    Args a{};
    a.offsets = offs2; a.E = 1; a.F = 0; a.st = st;
    a.N = sh.d; a.K = 6 * ep;
    a.C = dxr; a.ldc = sh.d;
    CUtensorMap mc;
    if (!make_map_2d(&ma, a6, 6 * (uint64_t)ep, sh.T, 64, 128) ||
        !make_map_3d(&mb, b6, sh.d, 6 * (uint64_t)ep, 1, 64, 64) || !make_map_2d_f32(&mc, dxr, sh.d, sh.T, 32, 32))
      return cudaErrorInvalidValue;
    err = launch_single<0, 0, 1, EPI_STORE_F32>(ma, mb, mc, a, stream);
    if (err != cudaSuccess) return err;
  }
  {
    Args a{};
    a.offsets = offs_split; a.E = splits; a.F = 0; a.st = st;
    a.M = 3 * ep; a.N = sh.d;
    a.C = c3; a.ldc = sh.d; a.sce = (int64_t)3 * ep * sh.d;
    CUtensorMap mc;
    if (!make_map_2d_strided(&ma, static_cast<const bf16 *>(a6) + 3 * ep, 3 * (uint64_t)ep, sh.T,
                             6 * (uint64_t)ep * 2, 64, 64) ||
        !make_map_2d(&mb, x, sh.d, sh.T, 64, 64) ||
        !make_map_3d_f32(&mc, c3, sh.d, 3 * (uint64_t)ep, (uint64_t)splits, 32, 32))
      return cudaErrorInvalidValue;
    err = launch_single<1, 1, 1, EPI_STORE_F32>(ma, mb, mc, a, stream);
  }
  return err;
}

}  // namespace moe
