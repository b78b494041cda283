// The C ABI of the MoE layer (declared in include/moe.h): argument
// validation on the host, workspace carve-up, and the launch sequence of each
// call. No call allocates device memory or synchronises the host, except
// moe_get_device_error, which is documented to synchronise.
#include <cmath>
#include <cstdio>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

static thread_local char g_cuda_error[256] = "";

static moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  snprintf(g_cuda_error, sizeof(g_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static moe_status make_shape(const moe_config *c, Shape *sh) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 1 || c->d_model < 1 || c->n_experts < 1 || c->top_k < 1 || c->d_ff < 1) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (c->add_residual != 0 && c->add_residual != 1) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID && c->score != MOE_SCORE_SQRT_SOFTPLUS)
    return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if ((c->reroute != 0 && c->reroute != 1) || !std::isfinite(c->aux_alpha)) return MOE_ERR_INVALID_ARG;
  if ((c->expert_choice != 0 && c->expert_choice != 1) || c->reserved != 0) return MOE_ERR_INVALID_ARG;
  if (c->expert_choice && (c->top_k != 1 || c->reroute || c->renormalize || c->score != MOE_SCORE_SOFTMAX ||
                           c->capacity < 1 || c->T > kExpertChoiceMaxTokens))
    return MOE_ERR_UNSUPPORTED;
  if (c->reroute && (c->top_k != 1 || c->n_experts < 2 || c->renormalize)) return MOE_ERR_UNSUPPORTED;
  if (c->top_k > c->n_experts) return MOE_ERR_INVALID_ARG;
  if (c->n_experts > 256 || c->top_k > 8) return MOE_ERR_UNSUPPORTED;
  const int mult = c->dtype == MOE_BF16 ? 8 : 4;   // 16-byte rows for TMA and the vector accesses
  if (c->d_model % mult != 0 || c->d_ff % mult != 0) return MOE_ERR_ALIGNMENT;
  const int64_t Tk = (int64_t)c->T * c->top_k;
  if (Tk > (int64_t)1 << 30 || (int64_t)c->d_model * c->d_ff * 2 > ((int64_t)1 << 31) || c->d_model > (1 << 22))
    return MOE_ERR_UNSUPPORTED;
  sh->T = c->T;
  sh->d = c->d_model;
  sh->E = c->n_experts;
  sh->k = c->top_k;
  sh->F = c->d_ff;
  sh->R1 = c->act == MOE_ACT_SWIGLU ? 2 * c->d_ff : c->d_ff;
  sh->act = c->act;
  sh->dtype = c->dtype;
  sh->renorm = c->renormalize;
  sh->residual = c->add_residual;
  sh->score = c->score;
  sh->reroute = c->reroute;
  sh->ec = c->expert_choice;
  sh->k_route = c->top_k;
  if (c->reroute) sh->k = 2;   // columns: first choice, second candidate
  sh->C = c->capacity < 0 ? -1 : c->capacity;
  sh->alpha = c->aux_alpha;
  int64_t rows = c->reroute ? (int64_t)c->T : Tk;   // rerouting keeps at most one assignment per token
  if (sh->C >= 0 && sh->C * sh->E < rows) rows = sh->C * sh->E;
  if (c->expert_choice) rows = (int64_t)c->n_experts * (c->capacity < c->T ? c->capacity : c->T);
  sh->rows = rows;
  sh->elt = c->dtype == MOE_BF16 ? 2 : 4;
  return MOE_OK;
}

WsLayout ws_layout(const Shape &sh) {
  WsLayout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = round_up(o + bytes, 256);
    return at;
  };
  L.status = take(256);
  const size_t db = (size_t)dispatch_blocks(sh);
  L.router_acc = take((size_t)sh.E * 12);
  L.zeroed = o;
  const RouterPlan rp = router_plan(sh);
  L.router_parts = take(rp.tensor_cores ? (size_t)3 * rp.ep * sh.d * 2 : 0);
  L.disp_counts = take(db * sh.E * 4);
  L.disp_base = take(db * sh.E * 4);
  L.disp_counts2 = take(sh.reroute ? db * sh.E * 4 : 0);
  L.disp_base2 = take(sh.reroute ? db * sh.E * 4 : 0);
  L.disp_kept1 = take(sh.reroute ? (size_t)sh.E * 4 : 0);
  const size_t ecw = sh.ec ? (size_t)sh.E * ((sh.T + 31) / 32) * 4 : 0;
  L.ec_bm = take(ecw);
  L.ec_prefix = take(ecw);
  L.ec_idx = take(sh.ec ? (size_t)sh.T * 4 : 0);
  L.ec_gate = take(sh.ec ? (size_t)sh.T * 4 : 0);
  L.ec_load = take(sh.ec ? (size_t)sh.E * 4 : 0);
  L.ec_aux = take(sh.ec ? 4 : 0);
  L.ec_dg = take(sh.ec ? (size_t)sh.rows * 4 : 0);
  const size_t rows = (size_t)(sh.rows > 0 ? sh.rows : 1);
  L.dyp = take(rows * sh.d * sh.elt);
  L.da = take(rows * sh.R1 * sh.elt);
  L.dxp = take(rows * sh.d * sh.elt);
  L.dg = take((size_t)sh.T * sh.k * 4);
  L.dh = take((size_t)sh.T * sh.E * 4);
  L.dxr = take((size_t)sh.T * sh.d * 4);
  const bool tc = sh.dtype == MOE_BF16;
  L.rg_a6 = take(tc ? (size_t)sh.T * 6 * rp.ep * 2 : 0);
  L.rg_b6 = take(tc ? (size_t)6 * rp.ep * sh.d * 2 : 0);
  const int G = tc ? router_grad_splits(sh) : 0;
  L.rg_c3 = take(tc ? (size_t)G * 3 * rp.ep * sh.d * 4 : 0);
  L.rg_offs = take(tc ? (size_t)(2 + G + 1) * 4 : 0);
  L.total = o;
  return L;
}

static DeviceStatus *status_of(void *ws) { return reinterpret_cast<DeviceStatus *>(ws); }

// Validation and error text shared with the workspace-free entry point.
moe_status dispatch_shape(const moe_config *cfg, Shape *sh) { return make_shape(cfg, sh); }
moe_status report_cuda(cudaError_t e) { return cuda_status(e); }

}  // namespace moe

using namespace moe;

// NVTX range over one ABI call, named after it (shown on Nsight timelines;
// without a tool attached the push and pop do nothing).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};
#define MOE_NVTX(name) NvtxRange moe_nvtx_range_(name)

#define MOE_CHECK(expr)                 \
  do {                                  \
    moe_status _s = (expr);             \
    if (_s != MOE_OK) return _s;        \
  } while (0)
#define MOE_REQUIRE(cond, code) \
  do {                          \
    if (!(cond)) return (code); \
  } while (0)
#define MOE_PTR(p) \
  do {                                               \
    if ((p) == nullptr) return MOE_ERR_INVALID_ARG;  \
    if (!aligned16(p)) return MOE_ERR_ALIGNMENT;     \
  } while (0)
#define MOE_OPT_PTR(p) \
  do {                                                    \
    if ((p) != nullptr && !aligned16(p)) return MOE_ERR_ALIGNMENT; \
  } while (0)

extern "C" {

int64_t moe_capacity(int64_t T, int32_t E, int32_t k, int32_t cf_num, int32_t cf_den, int32_t count_assignments) {
  if (T < 0 || E <= 0 || k <= 0 || cf_num < 0 || cf_den <= 0) return -1;
  const int64_t n = count_assignments ? T * (int64_t)k : T;
  return (n * (int64_t)cf_num) / ((int64_t)E * (int64_t)cf_den);
}

int64_t moe_max_rows(const moe_config *cfg) {
  Shape sh;
  if (make_shape(cfg, &sh) != MOE_OK) return -1;
  return sh.rows;
}

moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes) {
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(bytes != nullptr, MOE_ERR_INVALID_ARG);
  *bytes = ws_layout(sh).total;
  return MOE_OK;
}

moe_status moe_workspace_init(const moe_config *cfg, void *ws, moe_stream_t stream) {
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_PTR(ws);
  return cuda_status(cudaMemsetAsync(ws, 0, ws_layout(sh).zeroed, (cudaStream_t)stream));
}

moe_status moe_router(const moe_config *cfg, const void *x, const float *w_r, const float *logit_bias,
                      float *probs, int32_t *topk_idx, float *topk_gate, float *importance, int32_t *load,
                      float *aux_loss, void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_router");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(!sh.ec, MOE_ERR_INVALID_ARG);   // expert-choice layers route with moe_router_expert_choice
  MOE_PTR(x); MOE_PTR(w_r); MOE_PTR(topk_idx); MOE_PTR(topk_gate); MOE_PTR(importance); MOE_PTR(load);
  MOE_PTR(ws);
  MOE_OPT_PTR(logit_bias); MOE_OPT_PTR(probs); MOE_OPT_PTR(aux_loss);
  return cuda_status(launch_router(sh, x, w_r, logit_bias, nullptr, probs, topk_idx, topk_gate, importance, load,
                                   aux_loss, ws, (cudaStream_t)stream));
}

moe_status moe_router_biased(const moe_config *cfg, const void *x, const float *w_r, const float *logit_bias,
                             const float *select_bias, float *probs, int32_t *topk_idx, float *topk_gate,
                             float *importance, int32_t *load, float *aux_loss, void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_router_biased");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sh.dtype == MOE_BF16, MOE_ERR_UNSUPPORTED);
  MOE_PTR(x); MOE_PTR(w_r); MOE_PTR(select_bias); MOE_PTR(topk_idx); MOE_PTR(topk_gate); MOE_PTR(importance);
  MOE_PTR(load); MOE_PTR(ws);
  MOE_OPT_PTR(logit_bias); MOE_OPT_PTR(probs); MOE_OPT_PTR(aux_loss);
  return cuda_status(launch_router(sh, x, w_r, logit_bias, select_bias, probs, topk_idx, topk_gate, importance, load,
                                   aux_loss, ws, (cudaStream_t)stream));
}

moe_status moe_select_bias_update(const moe_config *cfg, const int32_t *load, float *select_bias, float gamma,
                                  moe_stream_t stream) {
  MOE_NVTX("moe_select_bias_update");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_PTR(load); MOE_PTR(select_bias);
  MOE_REQUIRE(std::isfinite(gamma), MOE_ERR_INVALID_ARG);
  return cuda_status(launch_select_bias_update(sh, load, gamma, select_bias, (cudaStream_t)stream));
}

moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *topk_idx, int32_t *slot,
                        int32_t *kept, int32_t *expert_offsets, int32_t *row_token, void *x_perm, void *ws,
                        moe_stream_t stream) {
  MOE_NVTX("moe_dispatch");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_PTR(x); MOE_PTR(topk_idx); MOE_PTR(slot); MOE_PTR(kept); MOE_PTR(expert_offsets); MOE_PTR(row_token);
  MOE_PTR(x_perm); MOE_PTR(ws);
  return cuda_status(launch_dispatch(sh, x, topk_idx, slot, kept, expert_offsets, row_token, x_perm, nullptr, ws,
                                     (cudaStream_t)stream));
}

moe_status moe_expert_gemm(const moe_config *cfg, const void *x_perm, const int32_t *expert_offsets,
                           const void *w1, const void *w2, void *pre_act, void *h, void *y_perm, void *ws,
                           moe_stream_t stream) {
  MOE_NVTX("moe_expert_gemm");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_PTR(x_perm); MOE_PTR(expert_offsets); MOE_PTR(w1); MOE_PTR(w2); MOE_PTR(h); MOE_PTR(y_perm); MOE_PTR(ws);
  MOE_OPT_PTR(pre_act);
  MOE_REQUIRE(!(sh.act == MOE_ACT_RELU && pre_act != nullptr), MOE_ERR_INVALID_ARG);
  DeviceStatus *st = status_of(ws);
  cudaError_t e = sh.dtype == MOE_BF16
                      ? tc_expert_forward(sh, x_perm, expert_offsets, w1, w2, pre_act, h, y_perm, st,
                                          (cudaStream_t)stream)
                      : simt_expert_forward(sh, x_perm, expert_offsets, w1, w2, pre_act, h, y_perm,
                                            (cudaStream_t)stream);
  return cuda_status(e);
}

moe_status moe_combine(const moe_config *cfg, const void *x, const void *y_perm, const int32_t *topk_idx,
                       const float *topk_gate, const int32_t *slot, const int32_t *expert_offsets, void *out,
                       moe_stream_t stream) {
  MOE_NVTX("moe_combine");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_PTR(x); MOE_PTR(y_perm); MOE_PTR(topk_idx); MOE_PTR(topk_gate); MOE_PTR(slot); MOE_PTR(expert_offsets);
  MOE_PTR(out);
  MOE_REQUIRE(out != x && out != y_perm, MOE_ERR_INVALID_ARG);
  return cuda_status(
      launch_combine(sh, x, y_perm, topk_idx, topk_gate, slot, expert_offsets, out, (cudaStream_t)stream));
}

moe_status moe_forward(const moe_config *cfg, const void *x, const float *w_r, const float *logit_bias,
                       const void *w1, const void *w2, float *probs, int32_t *topk_idx, float *topk_gate,
                       float *importance, int32_t *load, float *aux_loss, int32_t *slot, int32_t *kept,
                       int32_t *expert_offsets, int32_t *row_token, void *x_perm, void *h, void *y_perm, void *out,
                       void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_forward");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sh.dtype == MOE_BF16, MOE_ERR_UNSUPPORTED);
  MOE_PTR(x); MOE_PTR(w_r); MOE_PTR(w1); MOE_PTR(w2); MOE_PTR(topk_idx); MOE_PTR(topk_gate); MOE_PTR(importance);
  MOE_PTR(load); MOE_PTR(slot); MOE_PTR(kept); MOE_PTR(expert_offsets); MOE_PTR(row_token); MOE_PTR(x_perm);
  MOE_PTR(h); MOE_PTR(out); MOE_PTR(ws);
  MOE_OPT_PTR(logit_bias); MOE_OPT_PTR(probs); MOE_OPT_PTR(aux_loss); MOE_OPT_PTR(y_perm);
  if (sh.k > 1) MOE_PTR(y_perm);
  MOE_REQUIRE(out != x, MOE_ERR_INVALID_ARG);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e =
      launch_router(sh, x, w_r, logit_bias, nullptr, probs, topk_idx, topk_gate, importance, load, aux_loss, ws, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_dispatch(sh, x, topk_idx, slot, kept, expert_offsets, row_token, x_perm, sh.k == 1 ? out : nullptr, ws,
                      s);
  if (e != cudaSuccess) return cuda_status(e);
  e = tc_expert_forward_combine(sh, x, x_perm, row_token, expert_offsets, w1, w2, h, topk_gate, out, y_perm,
                                status_of(ws), s);
  if (e != cudaSuccess) return cuda_status(e);
  if (sh.k == 1) return MOE_OK;
  return cuda_status(launch_combine(sh, x, y_perm, topk_idx, topk_gate, slot, expert_offsets, out, s));
}

moe_status moe_backward(const moe_config *cfg, const moe_saved *sv, const void *dy, void *dx, float *dw_r,
                        void *dw1, void *dw2, void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_backward");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sv != nullptr, MOE_ERR_INVALID_ARG);
  MOE_PTR(sv->x); MOE_PTR(sv->w_r); MOE_PTR(sv->w1); MOE_PTR(sv->w2); MOE_PTR(sv->probs); MOE_PTR(sv->topk_idx);
  MOE_PTR(sv->topk_gate); MOE_PTR(sv->slot); MOE_PTR(sv->expert_offsets); MOE_PTR(sv->load);
  MOE_PTR(sv->x_perm); MOE_PTR(sv->h); MOE_PTR(sv->y_perm);
  if (sh.act == MOE_ACT_SWIGLU) MOE_PTR(sv->pre_act);
  MOE_PTR(dy); MOE_PTR(dx); MOE_PTR(dw_r); MOE_PTR(dw1); MOE_PTR(dw2); MOE_PTR(ws);
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  void *dyp = w + L.dyp, *da = w + L.da, *dxp = w + L.dxp;
  float *dg = reinterpret_cast<float *>(w + L.dg);
  float *dh = reinterpret_cast<float *>(w + L.dh);
  float *dxr = reinterpret_cast<float *>(w + L.dxr);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_combine_backward(sh, dy, sv->y_perm, sv->topk_idx, sv->topk_gate, sv->slot,
                                          sv->expert_offsets, dyp, dg, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = sh.dtype == MOE_BF16 ? tc_expert_backward(sh, sv->expert_offsets, sv->x_perm, sv->w1, sv->w2, sv->pre_act,
                                                sv->h, dyp, da, dxp, dw1, dw2, status_of(ws), s)
                           : simt_expert_backward(sh, sv->expert_offsets, sv->x_perm, sv->w1, sv->w2,
                                                  sv->pre_act, sv->h, dyp, da, dxp, dw1, dw2, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_router_backward(sh, sv->x, sv->w_r, sv->probs, sv->topk_idx, sv->topk_gate, sv->load, dg, dh, dw_r,
                             dxr, ws, s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_unpermute(sh, dy, dxp, dxr, sv->topk_idx, sv->slot, sv->expert_offsets, dx, s));
}

moe_status moe_router_expert_choice(const moe_config *cfg, const void *x, const float *w_r, const float *logit_bias,
                                    float *probs, int32_t *row_token, float *row_gate, int32_t *expert_offsets,
                                    float *importance, void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_router_expert_choice");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sh.ec, MOE_ERR_INVALID_ARG);
  MOE_PTR(x); MOE_PTR(w_r); MOE_PTR(probs); MOE_PTR(row_token); MOE_PTR(row_gate); MOE_PTR(expert_offsets);
  MOE_PTR(importance); MOE_PTR(ws);
  MOE_OPT_PTR(logit_bias);
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  cudaStream_t s = (cudaStream_t)stream;
  // the softmax scores and their column sums; the top-1 choice the router also makes is not used
  cudaError_t e = launch_router(sh, x, w_r, logit_bias, nullptr, probs, reinterpret_cast<int32_t *>(w + L.ec_idx),
                                reinterpret_cast<float *>(w + L.ec_gate), importance,
                                reinterpret_cast<int32_t *>(w + L.ec_load), reinterpret_cast<float *>(w + L.ec_aux), ws,
                                s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_ec_select(sh, probs, row_token, row_gate, expert_offsets,
                                      reinterpret_cast<uint32_t *>(w + L.ec_bm),
                                      reinterpret_cast<int32_t *>(w + L.ec_prefix), s));
}

moe_status moe_dispatch_expert_choice(const moe_config *cfg, const void *x, const int32_t *row_token, void *x_perm,
                                      moe_stream_t stream) {
  MOE_NVTX("moe_dispatch_expert_choice");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sh.ec, MOE_ERR_INVALID_ARG);
  MOE_PTR(x); MOE_PTR(row_token); MOE_PTR(x_perm);
  return cuda_status(launch_ec_gather(sh, x, row_token, x_perm, (cudaStream_t)stream));
}

moe_status moe_combine_expert_choice(const moe_config *cfg, const void *x, const void *y_perm, const int32_t *row_token,
                                     const float *row_gate, void *out, void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_combine_expert_choice");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sh.ec, MOE_ERR_INVALID_ARG);
  MOE_PTR(x); MOE_PTR(y_perm); MOE_PTR(row_token); MOE_PTR(row_gate); MOE_PTR(out); MOE_PTR(ws);
  MOE_REQUIRE(out != x && out != y_perm, MOE_ERR_INVALID_ARG);
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  uint32_t *bm = reinterpret_cast<uint32_t *>(w + L.ec_bm);
  int32_t *prefix = reinterpret_cast<int32_t *>(w + L.ec_prefix);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_ec_membership(sh, row_token, bm, prefix, s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_ec_combine(sh, x, y_perm, row_gate, bm, prefix, out, s));
}

moe_status moe_backward_expert_choice(const moe_config *cfg, const moe_saved_expert_choice *sv, const void *dy,
                                      void *dx, float *dw_r, void *dw1, void *dw2, void *ws, moe_stream_t stream) {
  MOE_NVTX("moe_backward_expert_choice");
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(sh.ec && sv != nullptr, MOE_ERR_INVALID_ARG);
  MOE_PTR(sv->x); MOE_PTR(sv->w_r); MOE_PTR(sv->w1); MOE_PTR(sv->w2); MOE_PTR(sv->probs); MOE_PTR(sv->row_token);
  MOE_PTR(sv->row_gate); MOE_PTR(sv->expert_offsets); MOE_PTR(sv->x_perm); MOE_PTR(sv->h); MOE_PTR(sv->y_perm);
  if (sh.act == MOE_ACT_SWIGLU) MOE_PTR(sv->pre_act);
  MOE_PTR(dy); MOE_PTR(dx); MOE_PTR(dw_r); MOE_PTR(dw1); MOE_PTR(dw2); MOE_PTR(ws);
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  void *dyp = w + L.dyp, *da = w + L.da, *dxp = w + L.dxp;
  float *dh = reinterpret_cast<float *>(w + L.dh);
  float *dxr = reinterpret_cast<float *>(w + L.dxr);
  float *dg_row = reinterpret_cast<float *>(w + L.ec_dg);
  uint32_t *bm = reinterpret_cast<uint32_t *>(w + L.ec_bm);
  int32_t *prefix = reinterpret_cast<int32_t *>(w + L.ec_prefix);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_ec_membership(sh, sv->row_token, bm, prefix, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_ec_combine_backward(sh, dy, sv->y_perm, sv->row_token, sv->row_gate, dyp, dg_row, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = sh.dtype == MOE_BF16 ? tc_expert_backward(sh, sv->expert_offsets, sv->x_perm, sv->w1, sv->w2, sv->pre_act,
                                                sv->h, dyp, da, dxp, dw1, dw2, status_of(ws), s)
                           : simt_expert_backward(sh, sv->expert_offsets, sv->x_perm, sv->w1, sv->w2, sv->pre_act,
                                                  sv->h, dyp, da, dxp, dw1, dw2, s);
  if (e != cudaSuccess) return cuda_status(e);
  e = launch_router_backward_ec(sh, sv->x, sv->w_r, sv->probs, bm, prefix, dg_row, dh, dw_r, dxr, ws, s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_ec_unpermute(sh, dy, dxp, dxr, bm, prefix, dx, s));
}

moe_status moe_backward_intermediates(const moe_config *cfg, void *ws, void **dyp, void **da, void **dxp,
                                      float **dg, float **dh) {
  Shape sh;
  MOE_CHECK(make_shape(cfg, &sh));
  MOE_REQUIRE(ws != nullptr, MOE_ERR_INVALID_ARG);
  const WsLayout L = ws_layout(sh);
  uint8_t *w = static_cast<uint8_t *>(ws);
  if (dyp) *dyp = w + L.dyp;
  if (da) *da = w + L.da;
  if (dxp) *dxp = w + L.dxp;
  if (dg) *dg = reinterpret_cast<float *>(w + L.dg);
  if (dh) *dh = reinterpret_cast<float *>(w + L.dh);
  return MOE_OK;
}

moe_status moe_get_device_error(void *ws, moe_stream_t stream, int32_t *code) {
  MOE_REQUIRE(ws != nullptr && code != nullptr, MOE_ERR_INVALID_ARG);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e);
  DeviceStatus st;
  e = cudaMemcpy(&st, ws, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  e = cudaMemset(ws, 0, sizeof(st));
  if (e != cudaSuccess) return cuda_status(e);
  *code = st.code;
  return MOE_OK;
}

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer or size";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device-side error recorded";
  }
  return "unknown status";
}

const char *moe_last_cuda_error(void) { return g_cuda_error; }

}  // extern "C"
