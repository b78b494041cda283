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
// next.
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {

namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;             // TMA ring depth
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;         // two 128 x 256 fp32 accumulators
constexpr int THREADS = 320;         // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr int MAX_E = 256;

// Grouped-K: every group has the same tiles, so no prefix array is kept.
template <bool GK> struct __align__(8) SmemT {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int tile_start[GK ? 1 : MAX_E + 1];  // grouped-M: tiles of the groups before e
};
// Plain-store epilogues (EPI_STORE, EPI_STORE_F32) stage each warp's 32-row
// slice in shared memory (128-byte swizzled rows, 4 KB per warp) and write it
// with a TMA tile store.
constexpr int STAGE_OUT_BYTES = 4096;
constexpr int EPI_WARPS = 8;
template <int EPI> constexpr bool tma_store_epi() { return EPI == EPI_STORE || EPI == EPI_STORE_F32; }
template <int GROUP_K, int EPI> constexpr size_t smem_bytes() {
  return 1024 /*align slack*/ + (size_t)STAGES * STAGE_BYTES +
         (tma_store_epi<EPI>() ? (size_t)EPI_WARPS * STAGE_OUT_BYTES : 0) + sizeof(SmemT<GROUP_K != 0>);
}
static_assert(smem_bytes<0, EPI_STORE>() <= 232448 && smem_bytes<1, EPI_STORE>() <= 232448, "shared memory budget");

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

template <int GROUP_K, int A_MN, int B_MN, int EPI>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const Args p) {
  constexpr bool TMA_STORE = tma_store_epi<EPI>();
  constexpr int NST = STAGES;
  using Smem = SmemT<GROUP_K != 0>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *tiles = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t *stage_out = tiles + (size_t)NST * STAGE_BYTES;  // TMA_STORE only: [EPI_WARPS][4 KB]
  Smem &s = *reinterpret_cast<Smem *>(stage_out + (TMA_STORE ? EPI_WARPS * STAGE_OUT_BYTES : 0));
  volatile int *abort_flag = &s.abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  constexpr bool SWIGLU_FWD = (EPI == EPI_SWIGLU);
  // Output columns one tile covers (SwiGLU forward: 128 gate + 128 up accumulators -> 128 outputs).
  constexpr int TN_OUT = SWIGLU_FWD ? 128 : BN;
  const int n_tiles = (p.N + TN_OUT - 1) / TN_OUT;
  const int m_tiles_k = GROUP_K ? (p.M + BM - 1) / BM : 0;

  // ---------------------------------------------------------------- set-up
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (TMA_STORE) prefetch_tmap(&tmC);
      for (int i = 0; i < NST; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
      for (int i = 0; i < 2; ++i) { mbar_init(&s.acc_full[i], 1); mbar_init(&s.acc_empty[i], 8); }
      mbar_init(&s.drain, 1);
      s.abort_flag = 0;
      fence_barrier_init();
    }
  } else if (warp == 1) {
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
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
        t = GROUP_K ? m_tiles_k * n_tiles : ((hi - lo + BM - 1) / BM) * n_tiles;
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
  auto k_steps = [&](int e) -> int {
    return GROUP_K ? (off(e + 1) - off(e) + BK - 1) / BK : (p.K + BK - 1) / BK;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    // Lane 0 waits for free stages and issues the tile loads.
    const uint64_t pol_a = policy_evict_last();
    // Weight tiles that no other m-tile will read are streamed (evict-first);
    // when groups span several m-tiles they are kept for the other m-tiles.
    const uint64_t pol_b = (!GROUP_K && p.b_once) ? policy_evict_first() : policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int nk = k_steps(e);
      for (int ks = 0; ks < nk; ++ks) {
        int got = 1;
        if (lane == 0) got = mbar_wait_bounded(&s.empty[stage], phase ^ 1, abort_flag, p.st) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        uint8_t *a_s = tiles + (size_t)stage * STAGE_BYTES;
        uint8_t *b_s = a_s + A_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(&s.full[stage], STAGE_BYTES);
        __syncwarp();
        const int k0 = ks * BK;
        if (lane == 0) {
          if (!GROUP_K) {
            const int row0 = off(e) + mt * BM;
            tma_load_2d(a_s, &tmA, &s.full[stage], k0, row0, pol_a);
            if (!B_MN) {
              int r0, r1;
              if (SWIGLU_FWD) { r0 = nt * 128; r1 = p.F + nt * 128; }
              else { r0 = nt * BN; r1 = nt * BN + 128; }
              tma_load_3d(b_s, &tmB, &s.full[stage], k0, r0, e, pol_b);
              tma_load_3d(b_s + 16384, &tmB, &s.full[stage], k0, r1, e, pol_b);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_3d(b_s + j * 8192, &tmB, &s.full[stage], nt * BN + 64 * j, k0, e, pol_b);
            }
          } else {
            const int r0 = off(e) + k0;
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_2d(a_s + j * 8192, &tmA, &s.full[stage], mt * BM + 64 * j, r0, pol_a);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(b_s + j * 8192, &tmB, &s.full[stage], nt * BN + 64 * j, r0, pol_b);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
    }
    if (lane == 0 && *abort_flag) {
      for (int i = 0; i < NST; ++i)
        if (issued & (1u << i)) drain_wait(&s.full[i], (issued_parity >> i) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, A_MN, B_MN);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      const int nk = k_steps(e);
      if (!mbar_wait_bounded(&s.acc_empty[acc], acc_phase ^ 1, abort_flag, p.st)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
      for (int ks = 0; ks < nk; ++ks) {
        if (!mbar_wait_bounded(&s.full[stage], phase, abort_flag, p.st)) { ok = false; break; }
        tc_fence_after();
        uint8_t *a_s = tiles + (size_t)stage * STAGE_BYTES;
        uint8_t *b_s = a_s + A_BYTES;
        int nkk = BK / 16;  // K16 slices of this step that hold rows of the group
        if (GROUP_K) {
          // The last K step of a group may run past its rows: only the slices
          // holding group rows are issued, and the rows past the group inside
          // the last of them are zeroed in both operands (each row is one
          // 128-byte line per 64-wide block).
          const int valid = off(e + 1) - (off(e) + ks * BK);
          if (valid < BK) {
            nkk = (valid + 15) >> 4;
            const int nrows = nkk * 16 - valid;
            if (nrows > 0) {
              const int chunks = nrows * 8;  // 16-byte chunks per block
              for (int i = lane; i < 6 * chunks; i += 32) {
                const int blk = i / chunks, rem = i - blk * chunks;
                const int row = valid + (rem >> 3), c = rem & 7;
                uint8_t *base = (blk < 2) ? (a_s + blk * 8192) : (b_s + (blk - 2) * 8192);
                *reinterpret_cast<uint4 *>(base + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
            }
            __syncwarp();
          }
        }
        if (lane == 0) {
          const uint32_t a0 = smem_u32(a_s), b0 = smem_u32(b_s);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nkk) break;
            const uint64_t ad = A_MN ? smem_desc_sw128(a0 + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(a0 + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024)
                                     : smem_desc_sw128(b0 + kk * 32, 16, 1024);
            tc_mma_bf16(d_tmem, ad, bd, IDESC, (ks > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&s.empty[stage]);
        }
        __syncwarp();
        if (++stage == NST) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&s.acc_full[acc]);
      __syncwarp();
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (*abort_flag) {
      if (lane == 0) tc_commit(&s.drain);
      __syncwarp();
      drain_wait(&s.drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    // Two warps per TMEM lane quarter: warp w reads lanes 32 (w % 4) .. + 31
    // (its rows) and the column half (w - 2) / 4 of the tile.
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;       // row inside the 128-row tile
    const int half = (warp - 2) >> 2;  // column half of the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int e, mt, nt;
      decode(tile, e, mt, nt);
      if (!mbar_wait_bounded(&s.acc_full[acc], acc_phase, abort_flag, p.st)) break;
      tc_fence_after();
      const uint32_t t_row = tmem + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      float v[32], w[32];
      if (TMA_STORE) {
        // This warp's 32-row slice: whole slices go through the staging buffer
        // and a TMA store; a slice cut by the end of its group (grouped-M) is
        // stored row by row, so the next group's rows are never touched.
        constexpr bool F32 = (EPI == EPI_STORE_F32);
        constexpr int CPB = F32 ? 1 : 2;  // 32-column chunks per 128-byte staging row
        uint8_t *stg = stage_out + (warp - 2) * STAGE_OUT_BYTES;
        int nvalid = 32;
        int r0;
        const bool zero = GROUP_K && off(e + 1) == off(e);
        if (!GROUP_K) {
          const int lo = mt * BM + q * 32;
          nvalid = min(32, max(0, off(e + 1) - off(e) - lo));
          r0 = off(e) + lo;
        } else {
          r0 = mt * BM + q * 32;
        }
#pragma unroll 1
        for (int c = 4 * half; c < 4 * half + 4; c += CPB) {
          const int col = nt * BN + c * 32;
          if (nvalid == 0 || col >= p.N) continue;
          float x[32 * CPB];
#pragma unroll
          for (int u = 0; u < CPB; ++u) {
            if (!zero) tmem_ld32(t_row + (c + u) * 32, x + 32 * u);
            else {
#pragma unroll
              for (int i = 0; i < 32; ++i) x[32 * u + i] = 0.0f;
            }
          }
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
              for (int i = 0; i < 8; ++i) Vec16<float>::store(cp + 4 * i, x + 4 * i);
            } else {
              bf16 *cp = static_cast<bf16 *>(p.C) + row * p.ldc + col;
#pragma unroll
              for (int i = 0; i < 8; ++i) Vec16<bf16>::store(cp + 8 * i, x + 8 * i);
            }
          }
        }
      } else if (!GROUP_K) {
        const int rows_e = off(e + 1) - off(e);
        const bool valid = mt * BM + r < rows_e;
        const int64_t row = (int64_t)off(e) + mt * BM + r;
        if (EPI == EPI_SWIGLU) {
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
              for (int i = 0; i < 4; ++i) Vec16<bf16>::store(hp + 8 * i, hv + 8 * i);
              if (p.C2) {
                bf16 *gp = p.C2 + row * p.ldc2 + col;
                bf16 *up = gp + p.F;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  Vec16<bf16>::store(gp + 8 * i, v + 8 * i);
                  Vec16<bf16>::store(up + 8 * i, w + 8 * i);
                }
              }
            }
          }
        } else {
          // The backward epilogues read saved activations; the loads of G
          // chunks are issued together before any of them is used.
          constexpr int NAUX = (EPI == EPI_SWIGLU_BWD) ? 8 : ((EPI == EPI_RELU_BWD || EPI == EPI_COMBINE) ? 4 : 0);
          constexpr int G = (EPI == EPI_SWIGLU_BWD) ? 2 : 4;
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
                  for (int i = 0; i < 4; ++i) aux[g * NAUX + i] = *reinterpret_cast<const uint4 *>(ap + 8 * i);
                  if (EPI == EPI_SWIGLU_BWD) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                      aux[g * NAUX + 4 + i] = *reinterpret_cast<const uint4 *>(ap + p.F + 8 * i);
                  }
                }
              }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const int col = nt * BN + (c0 + g) * 32;
              tmem_ld32(t_row + (c0 + g) * 32, v);
              if (!valid || col >= p.N) continue;
              if (EPI == EPI_RELU) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.0f);
              } else if (EPI == EPI_COMBINE) {
#pragma unroll
                for (int i = 0; i < 4; ++i) Vec16<bf16>::unpack(aux[g * NAUX + i], w + 8 * i);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = fmaf(gt, v[i], w[i]);   // out = x + g * y, rounded once
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
                  Vec16<bf16>::store(dp2 + 8 * i, du);
                }
              }
              if (EPI == EPI_STORE_F32) {
                float *cp = static_cast<float *>(p.C) + row * p.ldc + col;
#pragma unroll
                for (int i = 0; i < 8; ++i) Vec16<float>::store(cp + 4 * i, v + 4 * i);
              } else {
                bf16 *cp = static_cast<bf16 *>(p.C) + orow * p.ldc + col;
#pragma unroll
                for (int i = 0; i < 4; ++i) Vec16<bf16>::store(cp + 8 * i, v + 8 * i);
              }
            }
          }
        }
      } else {
        const bool empty_group = off(e + 1) == off(e);
        const int m = mt * BM + r;
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
              for (int i = 0; i < 8; ++i) Vec16<float>::store(cp + 4 * i, v + 4 * i);
            } else {
              bf16 *cp = static_cast<bf16 *>(p.C) + cofs + col;
#pragma unroll
              for (int i = 0; i < 4; ++i) Vec16<bf16>::store(cp + 8 * i, v + 8 * i);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.acc_empty[acc]);
      if (++acc == 2) { acc = 0; acc_phase ^= 1; }
    }
    if (TMA_STORE && lane == 0) bulk_wait_all();  // stores complete before the CTA exits
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
// mc is the output's tile map for the plain-store epilogues (ignored otherwise).
template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc, const Args &a,
                          cudaStream_t stream) {
  auto kern = grouped_gemm_kernel<GROUP_K, A_MN, B_MN, EPI>;
  constexpr size_t smem = smem_bytes<GROUP_K, EPI>();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_kernel(kern, dim3(sm_count()), dim3(THREADS), smem, stream, ma, mb, mc, a);
}
template <int GROUP_K, int A_MN, int B_MN, int EPI>
static cudaError_t launch(const CUtensorMap &ma, const CUtensorMap &mb, const Args &a, cudaStream_t stream) {
  static_assert(!tma_store_epi<EPI>(), "plain-store epilogues need the output map");
  return launch<GROUP_K, A_MN, B_MN, EPI>(ma, mb, ma, a, stream);
}

}  // namespace tc

// ---------------------------------------------------------------- launchers used by the C ABI
// True when the capacity keeps every group within one 128-row tile, so that
// each weight tile is read by a single m-tile.
static int weights_read_once(const Shape &sh) { return (sh.C >= 0 && sh.C <= tc::BM) ? 1 : 0; }

cudaError_t tc_expert_forward(const Shape &sh, const void *x_perm, const int32_t *offsets, const void *w1,
                              const void *w2, void *pre_act, void *h, void *y_perm, DeviceStatus *st,
                              cudaStream_t stream) {
  using namespace tc;
  CUtensorMap ma, mb;
  const uint64_t rows = sh.rows > 0 ? (uint64_t)sh.rows : 1;  // a map needs at least one row
  const int b_once = weights_read_once(sh);
  Args a{};
  a.offsets = offsets;
  a.E = sh.E;
  a.F = sh.F;
  a.st = st;
  a.b_once = b_once;
  // GEMM 1 (+ activation): A = x_perm [rows, d], B = W1 [E, R1, d]
  if (!make_map_2d(&ma, x_perm, sh.d, rows, 64, 128) || !make_map_3d(&mb, w1, sh.d, sh.R1, sh.E, 64, 128))
    return cudaErrorInvalidValue;
  a.N = sh.F;
  a.K = sh.d;
  a.C = h;
  a.ldc = sh.F;
  cudaError_t err;
  if (sh.act == MOE_ACT_SWIGLU) {
    a.C2 = (bf16 *)pre_act;
    a.ldc2 = 2 * (int64_t)sh.F;
    err = launch<0, 0, 0, EPI_SWIGLU>(ma, mb, a, stream);
  } else {
    err = launch<0, 0, 0, EPI_RELU>(ma, mb, a, stream);
  }
  if (err != cudaSuccess) return err;
  // GEMM 2: A = h [rows, F], B = W2 [E, d, F]
  if (!make_map_2d(&ma, h, sh.F, rows, 64, 128) || !make_map_3d(&mb, w2, sh.F, sh.d, sh.E, 64, 128))
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
  return launch<0, 0, 0, EPI_STORE>(ma, mb, mc, b, stream);
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
  const int b_once = weights_read_once(sh);
  Args a{};
  a.offsets = offsets;
  a.E = sh.E;
  a.F = sh.F;
  a.st = st;
  a.b_once = b_once;
  // GEMM 1 (+ activation): A = x_perm [rows, d], B = W1 [E, R1, d]
  if (!make_map_2d(&ma, x_perm, sh.d, rows, 64, 128) || !make_map_3d(&mb, w1, sh.d, sh.R1, sh.E, 64, 128))
    return cudaErrorInvalidValue;
  a.N = sh.F;
  a.K = sh.d;
  a.C = h;
  a.ldc = sh.F;
  cudaError_t err = sh.act == MOE_ACT_SWIGLU ? launch<0, 0, 0, EPI_SWIGLU>(ma, mb, a, stream)
                                             : launch<0, 0, 0, EPI_RELU>(ma, mb, a, stream);
  if (err != cudaSuccess) return err;
  // GEMM 2 + combine: A = h [rows, F], B = W2 [E, d, F]
  if (!make_map_2d(&ma, h, sh.F, rows, 64, 128) || !make_map_3d(&mb, w2, sh.F, sh.d, sh.E, 64, 128))
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
  return launch<0, 0, 0, EPI_COMBINE>(ma, mb, b, stream);
}

cudaError_t tc_expert_backward(const Shape &sh, const int32_t *offsets, const void *x_perm, const void *w1,
                               const void *w2, const void *pre_act, const void *h, const void *dyp, void *da,
                               void *dxp, void *dw1, void *dw2, DeviceStatus *st, cudaStream_t stream) {
  using namespace tc;
  CUtensorMap ma, mb;
  const uint64_t rows = sh.rows > 0 ? (uint64_t)sh.rows : 1;
  cudaError_t err;
  const bool swiglu = sh.act == MOE_ACT_SWIGLU;
  const int b_once = weights_read_once(sh);
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
      err = launch<0, 0, 1, EPI_SWIGLU_BWD>(ma, mb, a, stream);
    } else {
      a.aux = (const bf16 *)h; a.ldaux = sh.F;
      err = launch<0, 0, 1, EPI_RELU_BWD>(ma, mb, a, stream);
    }
    if (err != cudaSuccess) return err;
  }
  // dW2_e = dYp_e^T H_e   (grouped over K = rows of e): M = d, N = F
  {
    Args a{};
    a.offsets = offsets; a.E = sh.E; a.F = sh.F; a.st = st;
    a.M = sh.d; a.N = sh.F;
    a.C = dw2; a.ldc = sh.F; a.sce = (int64_t)sh.d * sh.F;
    CUtensorMap mc;
    if (!make_map_2d(&ma, dyp, sh.d, rows, 64, 64) || !make_map_2d(&mb, h, sh.F, rows, 64, 64) ||
        !make_map_3d(&mc, dw2, sh.F, sh.d, sh.E, 64, 32))
      return cudaErrorInvalidValue;
    err = launch<1, 1, 1, EPI_STORE>(ma, mb, mc, a, stream);
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
    err = launch<0, 0, 1, EPI_STORE>(ma, mb, mc, a, stream);
    if (err != cudaSuccess) return err;
  }
  // dW1_e = dA_e^T X_e: M = R1, N = d
  {
    Args a{};
    a.offsets = offsets; a.E = sh.E; a.F = sh.F; a.st = st;
    a.M = sh.R1; a.N = sh.d;
    a.C = dw1; a.ldc = sh.d; a.sce = (int64_t)sh.R1 * sh.d;
    CUtensorMap mc;
    if (!make_map_2d(&ma, da, sh.R1, rows, 64, 64) || !make_map_2d(&mb, x_perm, sh.d, rows, 64, 64) ||
        !make_map_3d(&mc, dw1, sh.d, sh.R1, sh.E, 64, 32))
      return cudaErrorInvalidValue;
    err = launch<1, 1, 1, EPI_STORE>(ma, mb, mc, a, stream);
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
    err = launch<0, 0, 1, EPI_STORE_F32>(ma, mb, mc, a, stream);
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
    err = launch<1, 1, 1, EPI_STORE_F32>(ma, mb, mc, a, stream);
  }
  return err;
}

}  // namespace moe
