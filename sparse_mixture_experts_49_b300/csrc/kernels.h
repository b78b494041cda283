// Internal launchers behind the C ABI (C++ linkage, not exported).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

struct DeviceStatus;

// moe_config after validation, with derived sizes.
struct Shape {
  int T, d, E, k, F, R1, act, dtype, renorm;
  int residual;   // add_residual
  int score;      // MOE_SCORE_*
  int reroute;    // No-Token-Left-Behind: k = 2 columns (first choice, second candidate)
  int ec;         // expert-choice routing: rows = E * min(C, T), groups of min(C, T) rows
  int k_route;    // top_k of the config: the columns load and f count (1 with reroute)
  int64_t C;      // capacity, < 0 = none
  float alpha;
  int64_t rows;   // rows of the packed buffers
  int elt;        // bytes per element of the x dtype
};

enum { EPI_STORE = 0, EPI_RELU = 1, EPI_SWIGLU = 2, EPI_RELU_BWD = 3, EPI_SWIGLU_BWD = 4, EPI_STORE_F32 = 5,
       EPI_COMBINE = 6 };

// Workspace carve-up (byte offsets from the workspace base). The first 256
// bytes hold the error word (offset 0), the router's completion counter (64),
// the dispatch's completion counters (128; 160 for rerouting's second round)
// and the grouped GEMM's tile counters (192: next tile, 196: CTAs done); the
// router's statistics accumulators follow. All of [0, zeroed) starts at zero (moe_workspace_init)
// and every call leaves it at zero again.
constexpr size_t kGemmSchedOffset = 192;
struct WsLayout {
  size_t status;                 // DeviceStatus
  size_t router_acc;               // [E] u64 importance (units of 2^-32), then [E] int32 load
  size_t zeroed;                   // end of the region that must start at zero
  size_t router_parts;             // [3, EP, d] bf16: hi/mid/lo split of W_r (tensor-core router)
  size_t disp_counts, disp_base;   // [dispatch blocks, E]
  size_t disp_counts2, disp_base2, disp_kept1;  // rerouting's second round: [blocks, E], [blocks, E], [E]
  size_t ec_bm, ec_prefix;         // expert choice: membership bitmap [E, W] u32 and word prefixes [E, W]
  size_t ec_idx, ec_gate, ec_load, ec_aux, ec_dg;  // expert choice: the router's top-1 outputs (unused), dg per row
  size_t dyp, da, dxp;             // backward: [rows, d], [rows, R1], [rows, d]
  size_t dg, dh, dxr;              // backward: [T, k], [T, E], [T, d] fp32
  size_t rg_a6, rg_b6, rg_c3, rg_offs;  // bf16 router gradient: [T, 6EP], [6EP, d] bf16; [G, 3EP, d] fp32;
                                       // {0, T} then the G + 1 token-range bounds of the dW_r split
  size_t total;
};
WsLayout ws_layout(const Shape &sh);

constexpr int ROUTER_TOKENS = 64;     // tokens per router block
constexpr int DISPATCH_TOKENS = 256;  // tokens per dispatch block

int router_blocks(const Shape &sh);

// How the router runs for a shape: tensor cores for bf16 x (one fused kernel
// per 128-token tile over all ep padded expert columns, d split over a
// cluster of `cluster` CTAs), CUDA cores for fp32 x.
struct RouterPlan {
  bool tensor_cores;
  int ep, m_tiles, cluster;
};
RouterPlan router_plan(const Shape &sh);
int dispatch_blocks(const Shape &sh);

// sel_bias: the selection-only correction bias (bf16 layers), or null.
cudaError_t launch_router(const Shape &sh, const void *x, const float *w_r, const float *bias, const float *sel_bias,
                          float *probs, int32_t *idx, float *gate, float *importance, int32_t *load, float *aux,
                          void *ws, cudaStream_t stream);
cudaError_t launch_select_bias_update(const Shape &sh, const int32_t *load, float gamma, float *sel_bias,
                                      cudaStream_t stream);

// x_perm may be null (rows are not copied); out_dropped, when given, gets
// x[t] for every token with no kept assignment. With sh.reroute the second
// round runs too (scratch in the workspace's rerouting regions).
cudaError_t launch_dispatch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot, int32_t *kept,
                            int32_t *offsets, int32_t *row_token, void *x_perm, void *out_dropped, void *ws,
                            cudaStream_t stream);

// Scratch of rerouting's second round: per-block counts and bases [blocks, E],
// the first round's kept counts [E], a zero-initialised completion counter.
struct RerouteScratch {
  int32_t *counts2, *base2, *kept1;
  unsigned int *counter2;
};
cudaError_t launch_dispatch_with_scratch(const Shape &sh, const void *x, const int32_t *idx, int32_t *slot,
                                         int32_t *kept, int32_t *offsets, int32_t *row_token, void *x_perm,
                                         void *out_dropped, int32_t *counts, int32_t *base, unsigned int *counter,
                                         DeviceStatus *st, cudaStream_t stream, const RerouteScratch *rr = nullptr);
moe_status dispatch_shape(const moe_config *cfg, Shape *sh);
moe_status report_cuda(cudaError_t e);

// Expert-choice routing (expert_choice.cu); T <= kExpertChoiceMaxTokens.
constexpr int kExpertChoiceMaxTokens = 32768;
cudaError_t launch_ec_select(const Shape &sh, const float *probs, int32_t *row_token, float *row_gate,
                             int32_t *expert_offsets, uint32_t *bm, int32_t *prefix, cudaStream_t stream);
cudaError_t launch_ec_membership(const Shape &sh, const int32_t *row_token, uint32_t *bm, int32_t *prefix,
                                 cudaStream_t stream);
cudaError_t launch_ec_gather(const Shape &sh, const void *x, const int32_t *row_token, void *x_perm,
                             cudaStream_t stream);
cudaError_t launch_ec_combine(const Shape &sh, const void *x, const void *y_perm, const float *row_gate,
                              const uint32_t *bm, const int32_t *prefix, void *out, cudaStream_t stream);
cudaError_t launch_ec_combine_backward(const Shape &sh, const void *dy, const void *y_perm, const int32_t *row_token,
                                       const float *row_gate, void *dyp, float *dg_row, cudaStream_t stream);
cudaError_t launch_ec_unpermute(const Shape &sh, const void *dy, const void *dxp, const float *dxr, const uint32_t *bm,
                                const int32_t *prefix, void *dx, cudaStream_t stream);
cudaError_t launch_router_backward_ec(const Shape &sh, const void *x, const float *w_r, const float *probs,
                                      const uint32_t *bm, const int32_t *bm_prefix, const float *dg_row, float *dh,
                                      float *dw_r, float *dxr, void *ws, cudaStream_t stream);

cudaError_t launch_combine(const Shape &sh, const void *x, const void *y_perm, const int32_t *idx,
                           const float *gate, const int32_t *slot, const int32_t *offsets, void *out,
                           cudaStream_t stream);

// Expert FFN forward on tensor cores (bf16) / CUDA cores (fp32).
cudaError_t tc_expert_forward(const Shape &sh, const void *x_perm, const int32_t *offsets, const void *w1,
                              const void *w2, void *pre_act, void *h, void *y_perm, DeviceStatus *st,
                              cudaStream_t stream);
cudaError_t simt_expert_forward(const Shape &sh, const void *x_perm, const int32_t *offsets, const void *w1,
                                const void *w2, void *pre_act, void *h, void *y_perm, cudaStream_t stream);

// Forward whose second GEMM combines in its epilogue for top-1 layers (out);
// k > 1 layers write y_perm.
cudaError_t tc_expert_forward_combine(const Shape &sh, const void *x, const void *x_perm, const int32_t *row_token,
                                      const int32_t *offsets, const void *w1, const void *w2, void *h,
                                      const float *gate, void *out, void *y_perm, DeviceStatus *st,
                                      cudaStream_t stream);
// Expert weight gradients with each (expert, m-tile)'s A rows resident (wgrad.cu), for layers whose
// capacity bounds the rows per expert (wgrad_fits): dW_e [M, N] = A_e^T B_e, C [E, M, N] bf16.
bool wgrad_fits(const Shape &sh);
cudaError_t launch_wgrad(const Shape &sh, const int32_t *offsets, const void *a, int M, const void *b, int N,
                         void *c, DeviceStatus *st, cudaStream_t stream);
cudaError_t tc_expert_backward(const Shape &sh, const int32_t *offsets, const void *x_perm, const void *w1,
                               const void *w2, const void *pre_act, const void *h, const void *dyp, void *da,
                               void *dxp, void *dw1, void *dw2, DeviceStatus *st, cudaStream_t stream);
cudaError_t simt_expert_backward(const Shape &sh, const int32_t *offsets, const void *x_perm, const void *w1,
                                 const void *w2, const void *pre_act, const void *h, const void *dyp, void *da,
                                 void *dxp, void *dw1, void *dw2, cudaStream_t stream);

// Router gradient GEMMs of a bf16 layer on the tensor cores (exact bf16 parts
// of dh and W_r; see gemm_tc.cu).
cudaError_t tc_router_grads(const Shape &sh, int ep, const void *a6, const void *b6, const void *x,
                            const int32_t *offs2, const int32_t *offs_split, int splits, float *dxr, float *c3,
                            DeviceStatus *st, cudaStream_t stream);
// Token ranges the dW_r = dh^T x GEMM is split into, so that about one tile per SM runs.
int router_grad_splits(const Shape &sh);

// Backward pieces outside the grouped GEMMs.
cudaError_t launch_combine_backward(const Shape &sh, const void *dy, const void *y_perm, const int32_t *idx,
                                    const float *gate, const int32_t *slot, const int32_t *offsets, void *dyp,
                                    float *dg, cudaStream_t stream);
cudaError_t launch_router_backward(const Shape &sh, const void *x, const float *w_r, const float *probs,
                                   const int32_t *idx, const float *gate, const int32_t *load, const float *dg,
                                   float *dh, float *dw_r, float *dxr, void *ws, cudaStream_t stream);
cudaError_t launch_unpermute(const Shape &sh, const void *dy, const void *dxp, const float *dxr,
                             const int32_t *idx, const int32_t *slot, const int32_t *offsets, void *dx,
                             cudaStream_t stream);

}  // namespace moe
