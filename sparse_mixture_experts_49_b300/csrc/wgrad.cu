// Expert weight gradients of the MoE layer for layers whose capacity bounds
// the rows per expert: dW_e = A_e^T B_e over the K = rows of group e, with
// A and B the packed rows of the group (dW2: A = dYp [rows, d], B = h
// [rows, F]; dW1: A = dA [rows, R1], B = x_perm [rows, d]).
//
// The chain rule through eq. (2) of "Mixture of Experts (MoE) を1から解説 —
// Switch Transformerのルーティングと負荷分散" gives these products; the
// compaction of kept rows into variable-size groups is the one of "LRMoE"
// (section この記事のポイント).
//
// With at most 192 rows per group (three 64-deep K steps) the A rows of one
// (expert, two 128-row m-tiles) unit fit in shared memory (96 KB). Each CTA
// takes whole units (unit u, u + grid, ...): it loads the unit's A rows once,
// keeps them while its MMAs run over every 128-column n-tile of the unit, and
// streams only B through the ring; each 16 KB K step of B feeds the MMAs of
// both m-tiles (four 128 x 128 fp32 accumulators: two per m-tile, double-
// buffered), so 256 x 128 of output loads 16 KB of B per K step instead of
// the grouped GEMM's 96 KB of A and B per 128 x 256. The rows past the group's end in its last K step
// are zeroed once per unit in A (a zero row of A makes every product over that
// K index zero), and in B as well after the last rows of all groups, where the
// packed buffers hold whatever an earlier call left.
//
//   warp 0: TMA loads (A of a unit once its buffer is free, B per K step);
//   warp 1: TMEM (512 columns of fp32 accumulators) and the tcgen05 MMAs;
//   warps 2-9: drain the accumulators (per TMEM lane quarter, one warp per
//           m-tile), round to bf16, stage 32 rows x 64 columns in 128-byte
//           swizzled shared memory and write them by TMA tile store.
// Every wait is bounded (the same limit and abort handling as the grouped
// GEMM).
#include "common.cuh"
#include "kernels.h"
#include "tma_host.h"

namespace moe {
namespace wg {

// Two m-tiles per unit: the large layer's backward pass 9.71-9.86 ms against
// 10.17-10.20 ms with one (one box, CUDA events, same bits).
#ifndef MOE_WG_MH
#define MOE_WG_MH 2
#endif
constexpr int BM = 128, BK = 64;
constexpr int MH = MOE_WG_MH;                  // m-tiles of 128 rows per unit, each with its accumulators
constexpr int TN = 256 / MH;                   // output columns per n-tile (TMEM: 2 buffers x MH x TN = 512)
constexpr int NBB = TN / 64;                   // 64-column B boxes per K step
constexpr int KSTEPS = 3;                      // K steps a resident unit may have
constexpr int MAX_ROWS = KSTEPS * BK;          // rows per group this kernel takes
constexpr int A_STEP = BM * BK * 2;            // 16 KB per m-tile: two 64-column boxes
constexpr int A_BUF = MH * KSTEPS * A_STEP;    // a unit's A rows
constexpr int B_STEP = TN * BK * 2;            // one K step of an n-tile's B
// Buffer counts (measured on the large layer's backward pass, one box, CUDA
// events: 1 A buffer + 4 B stages 10.02-10.04 ms; 2 + 3: 10.20-10.37 ms;
// 1 + 3 with two staging buffers per warp: 10.48-10.51 ms; 2 + 2 with two:
// 11.30 ms; the grouped GEMM: 11.03-11.06 ms).
#ifndef MOE_WG_A_BUFS
#define MOE_WG_A_BUFS 1
#endif
#ifndef MOE_WG_B_STAGES
#define MOE_WG_B_STAGES (MH == 1 ? 4 : 6)
#endif
#ifndef MOE_WG_STG_BUFS
#define MOE_WG_STG_BUFS 1
#endif
constexpr int A_BUFS = MOE_WG_A_BUFS;           // units' A buffers (two: the next unit's A loads under this one's MMAs)
constexpr int NSTB = MOE_WG_B_STAGES;          // B ring stages
constexpr int STG_BUFS = MOE_WG_STG_BUFS;      // staging buffers per epilogue warp
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int STG = 4096;                      // staging bytes per epilogue warp
constexpr int TMEM_COLS = 512;

struct __align__(8) Smem {
  uint64_t a_full[A_BUFS], a_empty[A_BUFS];
  uint64_t full[NSTB], empty[NSTB];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + A_BUFS * A_BUF + NSTB * B_STEP + EPI_WARPS * STG_BUFS * STG + sizeof(Smem);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Args {
  const int32_t *offsets;  // [E + 1] group row offsets
  int E, M, N;             // dW_e is M x N
  bf16 *C;                 // [E, M, N]
  DeviceStatus *st;
};

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity))
    if (global_timer_ns() - t0 > 200000000ull) break;  // 0.2 s
}

// Zeroes rows [valid, valid + nrows) of `blocks` 64-column blocks (one 128-byte line per row).
__device__ __forceinline__ void zero_rows(uint8_t *base, int blocks, int valid, int nrows, int lane) {
  const int chunks = nrows * 8;
  uint8_t *z0 = base + valid * 128;
  for (int blk = 0; blk < blocks; ++blk)
    for (int i = lane; i < chunks; i += 32)
      *reinterpret_cast<uint4 *>(z0 + blk * 8192 + (i >> 3) * 128 + (i & 7) * 16) = make_uint4(0, 0, 0, 0);
}

// K steps of group e, at most KSTEPS: more rows than the capacity allows are
// recorded as an error and only the first KSTEPS steps are used (identically
// in every role, so no buffer is overrun).
__device__ __forceinline__ int unit_steps(int rows) {
  const int nk = (rows + BK - 1) / BK;
  return nk < KSTEPS ? nk : KSTEPS;
}

__global__ void __launch_bounds__(THREADS, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const Args p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *base = smem_raw + ((1024 - (raw & 1023)) & 1023);
  uint8_t *abuf = base;                                   // [A_BUFS][KSTEPS][A_STEP]
  uint8_t *bring = abuf + A_BUFS * A_BUF;                 // [NSTB][B_STEP]
  uint8_t *stage_out = bring + NSTB * B_STEP;             // [EPI_WARPS][STG_BUFS][STG]
  Smem &s = *reinterpret_cast<Smem *>(stage_out + EPI_WARPS * STG_BUFS * STG);
  volatile int *abort_flag = &s.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (p.M + BM - 1) / BM, n_tiles = (p.N + TN - 1) / TN;
  const int m_units = (m_tiles + MH - 1) / MH;    // units per expert (MH m-tiles each)
  const int n_units = p.E * m_units;
  auto off = [&](int i) -> int { return __ldg(p.offsets + i); };
  auto nt0_error = [](int mt) { return mt == 0; };   // one report per group

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmC);
    for (int i = 0; i < A_BUFS; ++i) { mbar_init(&s.a_full[i], 1); mbar_init(&s.a_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s.acc_full[i], 1); mbar_init(&s.acc_empty[i], EPI_WARPS); }
    for (int i = 0; i < NSTB; ++i) { mbar_init(&s.full[i], 1); mbar_init(&s.empty[i], 1); }
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_barrier_init();
  } else if (warp == 1) {
    tmem_alloc(&s.tmem_base, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int last_row = off(p.E);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();   // a unit's B tiles are read again by the unit's other m-tiles
      int ab = 0, stage = 0;
      uint32_t aph = 0, ph = 0;
      uint32_t a_issued = 0, a_par = 0, issued = 0, par = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const int e = u / m_units, mp = u - e * m_units;
        const int r0 = off(e), rows = off(e + 1) - r0;
        const int nk = unit_steps(rows);
        if (rows > MAX_ROWS && nt0_error(mp)) record_error(p.st, MOE_DEVERR_GROUP_ROWS, e);
        if (!mbar_wait_bounded(&s.a_empty[ab], aph ^ 1, abort_flag, p.st)) break;
        mbar_arrive_expect_tx(&s.a_full[ab], (uint32_t)(MH * nk * A_STEP));
        uint8_t *a_s = abuf + ab * A_BUF;
        for (int h = 0; h < MH; ++h)   // (an m-tile past M reads the tensor map's zero fill)
          for (int ks = 0; ks < nk; ++ks)
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_2d(a_s + (h * KSTEPS + ks) * A_STEP + j * 8192, &tmA, &s.a_full[ab],
                          (mp * MH + h) * BM + 64 * j, r0 + ks * BK, pol);
        a_issued |= 1u << ab;
        a_par = (a_par & ~(1u << ab)) | (aph << ab);
        for (int nt = 0; ok && nt < n_tiles; ++nt) {
          for (int ks = 0; ks < nk; ++ks) {
            if (!mbar_wait_bounded(&s.empty[stage], ph ^ 1, abort_flag, p.st)) { ok = false; break; }
            mbar_arrive_expect_tx(&s.full[stage], B_STEP);
            uint8_t *b_s = bring + stage * B_STEP;
#pragma unroll
            for (int j = 0; j < NBB; ++j)
              tma_load_2d(b_s + j * 8192, &tmB, &s.full[stage], nt * TN + 64 * j, r0 + ks * BK, pol);
            issued |= 1u << stage;
            par = (par & ~(1u << stage)) | (ph << stage);
            if (++stage == NSTB) { stage = 0; ph ^= 1; }
          }
        }
        if (++ab == A_BUFS) { ab = 0; aph ^= 1; }
      }
      if (*abort_flag) {   // let every copy in flight land before the CTA can leave
        for (int i = 0; i < NSTB; ++i)
          if (issued & (1u << i)) drain_wait(&s.full[i], (par >> i) & 1);
        for (int i = 0; i < A_BUFS; ++i)
          if (a_issued & (1u << i)) drain_wait(&s.a_full[i], (a_par >> i) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC = idesc_bf16_f32(BM, TN, 1, 1);
    int ab = 0, stage = 0, acc = 0;
    uint32_t aph = 0, ph = 0, acc_ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const int e = u / m_units;
      const int r0 = off(e), rows = off(e + 1) - r0;
      const int nk = unit_steps(rows);
      const int valid = rows - (nk - 1) * BK;          // rows in the last K step (more if clamped: no padding)
      const int nkk_last = (valid + 15) >> 4;          // its K16 slices holding rows
      const int pad = nk > 0 ? nkk_last * 16 - valid : 0;
      const bool tail = r0 + rows == last_row;         // B's rows past the group: not another group's
      if (!mbar_wait_bounded(&s.a_full[ab], aph, abort_flag, p.st)) break;
      uint8_t *a_s = abuf + ab * A_BUF;
      if (pad > 0) {
        for (int h = 0; h < MH; ++h) zero_rows(a_s + (h * KSTEPS + nk - 1) * A_STEP, 2, valid, pad, lane);
        fence_proxy_async_smem();
      }
      __syncwarp();
      tc_fence_after();
      for (int nt = 0; nt < n_tiles; ++nt) {
        if (!mbar_wait_bounded(&s.acc_empty[acc], acc_ph ^ 1, abort_flag, p.st)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * MH * TN);   // m-half h: + h TN
        for (int ks = 0; ks < nk; ++ks) {
          if (!mbar_wait_bounded(&s.full[stage], ph, abort_flag, p.st)) { ok = false; break; }
          uint8_t *b_s = bring + stage * B_STEP;
          const bool last = ks == nk - 1;
          if (last && tail && pad > 0) {
            zero_rows(b_s, NBB, valid, pad, lane);
            fence_proxy_async_smem();
          }
          __syncwarp();
          tc_fence_after();
          if (lane == 0) {
            const uint32_t b0 = smem_u32(b_s);
            const int nkk = last ? nkk_last : BK / 16;
#pragma unroll
            for (int h = 0; h < MH; ++h) {
              const uint32_t a0 = smem_u32(a_s + (h * KSTEPS + ks) * A_STEP);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                if (kk >= nkk) break;
                tc_mma_bf16(d_tmem + (uint32_t)(h * TN), smem_desc_sw128(a0 + kk * 2048, 8192, 1024),
                            smem_desc_sw128(b0 + kk * 2048, 8192, 1024), IDESC, (ks > 0 || kk > 0) ? 1u : 0u);
              }
            }
            tc_commit(&s.empty[stage]);
          }
          __syncwarp();
          if (++stage == NSTB) { stage = 0; ph ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) tc_commit(&s.acc_full[acc]);   // (no MMAs for an empty group: the epilogue writes zeros)
        __syncwarp();
        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&s.a_empty[ab]);        // A is free once this unit's MMAs have completed
      __syncwarp();
      if (++ab == A_BUFS) { ab = 0; aph ^= 1; }
    }
    if (*abort_flag) {
      if (lane == 0) tc_commit(&s.drain);
      __syncwarp();
      drain_wait(&s.drain, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..9)
    const int q = warp & 3;            // TMEM lane quarter: rows 32 q .. 32 q + 31
    const int half = (warp - 2) >> 2;  // one m-tile: the tile's column half; two: the m-half (all TN columns)
    const int hm = MH == 2 ? half : 0, hc = MH == 2 ? 0 : half;
    uint8_t *stg = stage_out + (warp - 2) * STG_BUFS * STG;
    int sbuf = 0;   // the staging buffer of this warp's next store
    int acc = 0;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const int e = u / m_units, mt = (u - e * m_units) * MH + hm;
      const bool zero = off(e + 1) == off(e);
      const int r0 = mt * BM + q * 32;   // first output row of this warp's slice
      const bool out_rows = r0 < p.M;    // (the second m-tile of the last unit may lie past M)
      for (int nt = 0; nt < n_tiles; ++nt) {
        if (!mbar_wait_bounded(&s.acc_full[acc], acc_ph, abort_flag, p.st)) { ok = false; break; }
        tc_fence_after();
        const uint32_t t_row = tmem + (uint32_t)((acc * MH + hm) * TN) + ((uint32_t)(q * 32) << 16);
        uint32_t xr[4][32];
        if (!zero) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_issue(t_row + (4 * hc + c) * 32, xr[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_wait32(xr[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) xr[c][i] = 0u;
        }
        // the accumulator goes back to the MMA warp before any store
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.acc_empty[acc]);
        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
#pragma unroll
        for (int cu = 0; cu < 4; cu += 2) {
          const int col = nt * TN + (4 * hc + cu) * 32;
          if (col >= p.N || !out_rows) continue;
          float x[64];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            x[i] = __uint_as_float(xr[cu][i]);
            x[32 + i] = __uint_as_float(xr[cu + 1][i]);
          }
          // the store that last read this buffer has left it (with two buffers: the one before the previous)
          if (lane == 0) {
            if (STG_BUFS == 2) bulk_wait_read_1();
            else bulk_wait_read_all();
          }
          __syncwarp();
          uint8_t *sb = stg + sbuf * STG;
          uint8_t *rowp = sb + lane * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) Vec16<bf16>::store(rowp + ((j ^ (lane & 7)) << 4), x + 8 * j);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmC, sb, col, r0, e);   // rows past M and columns past N are clipped
            bulk_commit();
          }
          if (++sbuf == STG_BUFS) sbuf = 0;
        }
      }
    }
    if (lane == 0) bulk_wait_all();  // stores complete before the CTA exits
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace wg

bool wgrad_fits(const Shape &sh) { return sh.C > 0 && sh.C <= wg::MAX_ROWS; }

// dW_e [M, N] = A_e^T B_e for every expert e: A [rows, M], B [rows, N] packed
// rows (bf16, row-major), C [E, M, N] bf16.
cudaError_t launch_wgrad(const Shape &sh, const int32_t *offsets, const void *a, int M, const void *b, int N,
                         void *c, DeviceStatus *st, cudaStream_t stream) {
  static cudaError_t attr = cudaFuncSetAttribute(wg::wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)wg::SMEM_BYTES);
  if (attr != cudaSuccess) return attr;
  const uint64_t rows = sh.rows > 0 ? (uint64_t)sh.rows : 1;
  CUtensorMap ma, mb, mc;
  if (!make_map_2d(&ma, a, (uint64_t)M, rows, 64, 64) || !make_map_2d(&mb, b, (uint64_t)N, rows, 64, 64) ||
      !make_map_3d(&mc, c, (uint64_t)N, (uint64_t)M, (uint64_t)sh.E, 64, 32))
    return cudaErrorInvalidValue;
  wg::Args p;
  p.offsets = offsets;
  p.E = sh.E;
  p.M = M;
  p.N = N;
  p.C = static_cast<bf16 *>(c);
  p.st = st;
  const int units = sh.E * ((M + wg::MH * wg::BM - 1) / (wg::MH * wg::BM));
  int g = sm_count();
  if (g > units) g = units;
  return launch_kernel(wg::wgrad_kernel, dim3(g > 0 ? g : 1), dim3(wg::THREADS), wg::SMEM_BYTES, stream, ma, mb,
                       mc, p);
}

}  // namespace moe
