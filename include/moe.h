/*
 * moe.h — C ABI of the sparsely-gated Mixture-of-Experts FFN layer on one
 * NVIDIA B300 (sm_103a): router -> top-k -> capacity/dispatch -> expert FFNs
 * as a grouped GEMM -> combine, and the matching backward pass.
 *
 * Pages the operations follow (cited by title and section/equation):
 *   [Switch] "Mixture of Experts (MoE) を1から解説 — Switch Transformerの
 *            ルーティングと負荷分散": eq. (1) softmax router, eq. (2) gated sum,
 *            eq. (3) expert capacity and dropped tokens, eq. (4) load-balancing
 *            loss, the fp32 router of section 学習を安定させる3つの工夫, and the
 *            parameter vocabulary of section 現場ではこう使う
 *            (num_experts, capacity_factor, expert_capacity, alpha).
 *   [LRMoE]  "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE
 *            Training on Memory-Constrained Nodes", section この記事のポイント:
 *            kept token-expert pairs compacted into variable-size groups that
 *            feed a grouped GEMM.
 *   [Wiki]   "Mixture-of-Experts" (notes.yuuk.io): top-k routing with k > 1,
 *            SwiGLU experts, importance/load statistics, replay of recorded
 *            routing.
 *
 * Conventions for every call:
 *   - All array pointers are caller-owned DEVICE memory, row-major, at least
 *     16-byte aligned (MOE_ERR_ALIGNMENT otherwise). The library never
 *     allocates device memory: scratch lives in the caller's workspace.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream). Nothing on the path synchronises the host;
 *     moe_get_device_error is the one call that does.
 *   - Arguments are validated on the host before any launch. On an error
 *     status nothing was launched and no output was touched.
 *   - Outputs are overwritten, never accumulated into.
 *   - "x dtype" below is cfg->dtype: MOE_BF16 (bf16 x, expert weights,
 *     activations; fp32 accumulation) or MOE_F32 (fp32 throughout, no TF32).
 *     Router weights, probabilities and gates are always fp32 ([Switch]
 *     section 学習を安定させる3つの工夫: the router stays in float32).
 *   - Sizes: T tokens, d = d_model, E experts, k = top_k, F = d_ff,
 *     R1 = F (ReLU) or 2F (SwiGLU: gate rows then up rows),
 *     rows = moe_max_rows(cfg) = min(T*k, E*C) (T*k without a capacity;
 *     min(T, E*C) with cfg->reroute). "k columns" below are 2 with
 *     cfg->reroute (see moe_config), else k.
 *   - Limits: 1 <= E <= 256, 1 <= k <= min(E, 8), T >= 1, d <= 2^22; d and F are
 *     multiples of 8 for MOE_BF16 and of 4 for MOE_F32, so that every row is
 *     a whole number of 16-byte vectors (MOE_ERR_ALIGNMENT otherwise).
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2, /* outside the limits above */
  MOE_ERR_ALIGNMENT = 3,   /* pointer not 16-byte aligned, or d/F not a multiple of 8 (bf16) or 4 (fp32) */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call failed (see moe_last_cuda_error) */
  MOE_ERR_DEVICE = 5       /* a kernel recorded an error (see moe_get_device_error) */
} moe_status;

enum { MOE_ACT_RELU = 0, MOE_ACT_SWIGLU = 1 };
enum { MOE_F32 = 0, MOE_BF16 = 1 };
/* Router score functions. MOE_SCORE_SOFTMAX is [Switch] eq. (1); the two
 * elementwise scores are the variants [Wiki] section 横断的知見 names (sigmoid
 * gating without the softmax's zero-sum coupling, and sqrt(Softplus(h))):
 *   sigmoid:       s_e = 1 / (1 + exp(-h_e))
 *   sqrt_softplus: s_e = sqrt(log(1 + exp(h_e))) */
enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1, MOE_SCORE_SQRT_SOFTPLUS = 2 };

/* Codes a kernel can record in the workspace's error word. */
enum {
  MOE_DEVERR_NONE = 0,
  MOE_DEVERR_BAD_EXPERT = 1, /* a top-k index outside [0, E) */
  MOE_DEVERR_DUP_EXPERT = 2, /* the same expert twice in one token's top-k */
  MOE_DEVERR_TIMEOUT = 3,    /* a bounded on-chip wait gave up; outputs are invalid */
  MOE_DEVERR_GROUP_ROWS = 4  /* moe_backward: an expert's packed rows exceed cfg->capacity (offsets not
                                from this layer's dispatch); that expert's weight gradients are invalid */
};

/* Problem description ([Switch] section 現場ではこう使う: num_experts,
 * expert_capacity, the aux-loss coefficient alpha). */
typedef struct moe_config {
  int32_t T;           /* tokens in this call ("tokens per batch" of eq. (3)) */
  int32_t d_model;     /* d */
  int32_t n_experts;   /* E, the N of eqs. (1)-(4) */
  int32_t top_k;       /* k (Switch: 1) */
  int32_t d_ff;        /* F, hidden width of one expert */
  int32_t act;         /* MOE_ACT_RELU: W2 relu(W1 z); MOE_ACT_SWIGLU: W2 (silu(Wg z) * Wu z) */
  int32_t dtype;       /* MOE_BF16 or MOE_F32 */
  int32_t renormalize; /* 1: gates renormalised over the k selected experts */
  int32_t add_residual; /* 1: out = x + MoE(x) and a fully dropped token returns x ([Switch]
                           section エキスパートには「定員」がある: overflow passes through the
                           residual); 0: out = MoE(x), zeros for a fully dropped token (the
                           caller adds the residual), and dX carries no dY term */
  int32_t score;       /* MOE_SCORE_*: the router's score function (softmax by default) */
  int64_t capacity;    /* expert capacity C per expert; < 0: no limit (dropless) */
  float aux_alpha;     /* alpha of eq. (4) */
  int32_t reroute;     /* 1: No-Token-Left-Behind ([Switch] section 論文の限界と、まだ分かって
                          いないこと: overflow goes to the token's second candidate). Top-1 layers
                          with E >= 2 and no renormalisation only. topk_idx, topk_gate and slot
                          then have 2 columns: the first choice, and the second-best expert that a
                          token dropped by its first choice's capacity is offered to in a second
                          round (token order, into the room each expert has left; slot -1 where
                          not kept). Load and f count first choices. 0: plain top-k. */
  int32_t expert_choice; /* 1: expert-choice routing (see moe_router_expert_choice): each expert
                            takes the min(C, T) tokens with the largest scores; top_k must be 1
                            (unused), capacity C >= 1, softmax scores, T <= 32768, no rerouting
                            or renormalisation. 0: token-choice top-k. */
  int32_t reserved;    /* must be 0 */
} moe_config;

/* Expert capacity, [Switch] eq. (3): floor(n * cf_num / (E * cf_den)) with
 * n = k*T assignments (count_assignments != 0) or n = T tokens. Integer
 * arithmetic only. Returns -1 on invalid arguments (E, cf_den <= 0, ...). */
int64_t moe_capacity(int64_t T, int32_t E, int32_t k, int32_t cf_num, int32_t cf_den,
                     int32_t count_assignments);

/* Rows of the permuted buffers x_perm / h / y_perm / pre_act: min(T*k, E*C),
 * or T*k without a capacity. -1 if cfg is invalid. */
int64_t moe_max_rows(const moe_config *cfg);

/* Bytes of the workspace every call below takes (forward and backward
 * scratch, and the device error word). */
moe_status moe_workspace_size(const moe_config *cfg, size_t *bytes);

/* Clears the workspace's error word, completion counters and statistics
 * accumulators (its first few KB). Call once after allocating it; every
 * call below leaves that region cleared again. */
moe_status moe_workspace_init(const moe_config *cfg, void *ws, moe_stream_t stream);

/*
 * Router: h = W_r x (+ b), p = softmax(h) over all E experts ([Switch]
 * eq. (1)), the k largest logits per token (descending, ties to the lower
 * index), gates g = p of the chosen experts ([Switch] eq. (2); divided by
 * their sum when cfg->renormalize), and the balance statistics of eq. (4).
 *
 *   x          [T, d]  x dtype
 *   w_r        [E, d]  fp32 (h = W_r x)
 *   logit_bias [E]     fp32 constant added to h before the softmax, or NULL
 *   probs      [T, E]  fp32 out, or NULL (the backward pass needs it)
 *   topk_idx   [T, k]  int32 out
 *   topk_gate  [T, k]  fp32 out
 *   importance [E]     fp32 out: sum_t p[t, e]
 *   load       [E]     int32 out: number of tokens with e in their top-k
 *   aux_loss   [1]     fp32 out or NULL: alpha * E * sum_e f_e P_e with
 *                      f_e = load_e / (T k), P_e = importance_e / T
 * Statistics are summed per block in a fixed order, then across blocks in
 * integers (load) and 64-bit fixed point (importance, units of 2^-32): the
 * results are bitwise reproducible whatever the order the blocks run in.
 */
moe_status moe_router(const moe_config *cfg, const void *x, const float *w_r,
                      const float *logit_bias, float *probs, int32_t *topk_idx,
                      float *topk_gate, float *importance, int32_t *load, float *aux_loss,
                      void *ws, moe_stream_t stream);

/*
 * Router with a selection-only correction bias: the auxiliary-loss-free load
 * balancing that [Wiki] "Mixture-of-Experts", section 横断的知見, describes
 * (each expert's bias is added to the routing scores when the experts are
 * chosen; the gates stay the scores). Everything as in moe_router, with
 * cfg->score choosing the score s (softmax, sigmoid or sqrt(softplus)):
 *   probs       [T, E] fp32 out (or NULL): the scores s
 *   select_bias [E]    fp32: the k largest s + b per token are chosen
 *                      (descending, ties to the lower index)
 *   topk_gate   [T, k] fp32 out: s of the chosen experts (divided by their
 *                      sum when cfg->renormalize); the bias is not in them
 *   importance  [E]    fp32 out: sum_t s[t, e]
 * Without a bias (moe_router, any cfg->score) the choice is the top-k of h,
 * which is the order of every score function here. MOE_BF16 layers only
 * (MOE_ERR_UNSUPPORTED otherwise). moe_backward differentiates the gates
 * through cfg->score; the bias and the choice carry no gradient.
 */
moe_status moe_router_biased(const moe_config *cfg, const void *x, const float *w_r,
                             const float *logit_bias, const float *select_bias, float *probs,
                             int32_t *topk_idx, float *topk_gate, float *importance, int32_t *load,
                             float *aux_loss, void *ws, moe_stream_t stream);

/*
 * The correction bias's update after a batch, the sign rule of the
 * auxiliary-loss-free method [Wiki] section 横断的知見 cites:
 *   select_bias[e] += gamma * sign(mean_e'(load) - load[e])
 * so overloaded experts move down and underloaded ones up (no change at the
 * mean). The sign is decided in integers, as sign(sum(load) - E load[e]).
 *   load        [E] int32 (moe_router_biased's output)
 *   select_bias [E] fp32, updated in place
 */
moe_status moe_select_bias_update(const moe_config *cfg, const int32_t *load, float *select_bias,
                                  float gamma, moe_stream_t stream);

/*
 * Dispatch ([Switch] eq. (3) and its dropped-token rule; [LRMoE] compaction
 * into variable-size groups). Every expert takes the tokens that chose it in
 * ascending token order and keeps the first C: slot = rank, or -1 when the
 * assignment is dropped. Kept pairs are packed expert by expert:
 * row(t, j) = expert_offsets[e] + slot[t, j], and x_perm[row] = x[t].
 * topk_idx may come from moe_router or from the caller (replay of a recorded
 * routing). An index outside [0, E) or a repeated expert within one token
 * records MOE_DEVERR_BAD_EXPERT / MOE_DEVERR_DUP_EXPERT and the pair is
 * treated as dropped.
 *
 *   x              [T, d]    x dtype
 *   topk_idx       [T, k]    int32
 *   slot           [T, k]    int32 out
 *   kept           [E]       int32 out: min(load_e, C)
 *   expert_offsets [E + 1]   int32 out: exclusive prefix sum of kept
 *   row_token      [rows]    int32 out: token of each packed row (rows past
 *                            expert_offsets[E] are left untouched)
 *   x_perm         [rows, d] x dtype out
 */
moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                        int32_t *slot, int32_t *kept, int32_t *expert_offsets,
                        int32_t *row_token, void *x_perm, void *ws, moe_stream_t stream);

/*
 * Workspace-free dispatch. The pages have no counterpart: this is an
 * interface convenience, not a step of the method.
 *
 * Same computation and outputs as moe_dispatch, for callers that cannot give
 * the library any scratch memory because they cannot allocate device memory
 * at all (a plugin inside a host framework that owns every device
 * allocation, or a latency-critical path that cannot pay for cudaMalloc's
 * device-wide synchronisation). The dispatch's scratch lives in one fixed
 * array inside the library instead, about 256 KB, held by every GPU that
 * loads the library until the process exits. The call allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine).
 *   - T <= MOE_NOALLOC_MAX_TOKENS, else MOE_ERR_UNSUPPORTED before any launch.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call shares the array, which keeps the last call's contents:
 *     calls whose work can overlap on the GPU (unordered streams) race and
 *     give wrong results. Order them on one stream, or use moe_dispatch with
 *     one workspace per stream.
 *   - Bad or repeated expert indices are treated as dropped, as in
 *     moe_dispatch, but are not reported (the error word is private).
 */
#define MOE_NOALLOC_MAX_TOKENS 32768
moe_status moe_dispatch_noalloc(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                                int32_t *slot, int32_t *kept, int32_t *expert_offsets,
                                int32_t *row_token, void *x_perm, moe_stream_t stream);

/*
 * Expert FFNs over the packed groups ([Switch] section 直感: each expert is a
 * copy of the FFN; [LRMoE] variable-size grouped GEMM). For the rows of
 * expert e (expert_offsets[e] .. expert_offsets[e+1]):
 *   ReLU:   h = relu(x_perm W1_e^T),                 y_perm = h W2_e^T
 *   SwiGLU: h = silu(x_perm Wg_e^T) * (x_perm Wu_e^T), y_perm = h W2_e^T
 * fp32 accumulation; h and y_perm rounded to the x dtype.
 *
 *   x_perm  [rows, d]      x dtype
 *   w1      [E, R1, d]     x dtype (SwiGLU: rows 0..F-1 gate, F..2F-1 up)
 *   w2      [E, d, F]      x dtype
 *   pre_act [rows, 2F]     x dtype out (SwiGLU only: gate | up pre-activations,
 *                          kept for the backward pass); NULL = not stored
 *                          (must be NULL for ReLU: h itself carries the mask)
 *   h       [rows, F]      x dtype out
 *   y_perm  [rows, d]      x dtype out
 * Rows past expert_offsets[E] are not written.
 *
 * bf16 layers run on tcgen05 tiles of 128 rows, one CTA each, in a fixed
 * order (CTA u takes tiles u, u + grid, ...). An m-tile that holds at most
 * 64 of its expert's rows runs 64-row MMAs, and when a launch has fewer
 * than four waves of tiles, the tiles of a last wave that fills at most half
 * of the CTAs are cut into 128- or 64-column windows; both give the same
 * bits as whole tiles. Environment variables, read at every call, change
 * this for this call and for moe_forward / moe_backward: MOE_GEMM_PAIR=1
 * runs CTA-pair tiles (two CTAs of a cluster share an MMA of 256 rows);
 * MOE_GEMM_SCHED=dynamic hands the one-CTA tiles out from a counter in the
 * workspace as CTAs free up; MOE_GEMM_M64=0 keeps short m-tiles at 128 rows;
 * MOE_GEMM_TAIL=0 keeps last-wave tiles whole. Results agree to fp32
 * accumulation order.
 */
moe_status moe_expert_gemm(const moe_config *cfg, const void *x_perm,
                           const int32_t *expert_offsets, const void *w1, const void *w2,
                           void *pre_act, void *h, void *y_perm, void *ws,
                           moe_stream_t stream);

/*
 * Combine ([Switch] eq. (2) plus the residual passthrough of dropped tokens):
 *   out[t] = x[t] + sum over j with slot[t, j] >= 0 of
 *            topk_gate[t, j] * y_perm[expert_offsets[e] + slot[t, j]]
 * summed in fp32 and rounded once. A token with every assignment dropped
 * gets x[t] bit for bit. With cfg->add_residual == 0 the x[t] term is left
 * out (a fully dropped token gets zeros).
 *
 *   out [T, d] x dtype out (may not alias x or y_perm)
 */
moe_status moe_combine(const moe_config *cfg, const void *x, const void *y_perm,
                       const int32_t *topk_idx, const float *topk_gate, const int32_t *slot,
                       const int32_t *expert_offsets, void *out, moe_stream_t stream);

/*
 * The whole forward layer in one call, for inference: router, dispatch,
 * expert FFNs and combine ([Switch] eqs. (1)-(4) and the dropped-token rule;
 * [LRMoE] compaction into variable-size groups). For top-1 layers the
 * second expert GEMM writes out[t] = x[t] + g[t] * E_e(x[t]) in its
 * epilogue (no y_perm and no combine launch; the dispatch copies x to out
 * for dropped tokens); k > 1 layers combine as moe_combine does. Results match
 * the separate calls except that, for top-1 layers, y is not rounded to the
 * x dtype before the gated residual sum (one rounding instead of two).
 * Nothing only the backward pass needs is stored (no pre-activations; no
 * y_perm for top-1): train with the separate calls.
 *
 * Arguments as in moe_router, moe_dispatch and moe_combine, plus
 *   w1, w2   expert weights as in moe_expert_gemm
 *   x_perm   [rows, d]  x dtype out (packed token rows)
 *   h        [rows, F]  x dtype out (hidden activations, packed rows)
 *   y_perm   [rows, d]  x dtype scratch, required when top_k > 1, ignored
 *                       (may be NULL) when top_k == 1
 *   out      [T, d]     x dtype out (may not alias x)
 * MOE_BF16 only (MOE_ERR_UNSUPPORTED for MOE_F32).
 */
moe_status moe_forward(const moe_config *cfg, const void *x, const float *w_r,
                       const float *logit_bias, const void *w1, const void *w2, float *probs,
                       int32_t *topk_idx, float *topk_gate, float *importance, int32_t *load,
                       float *aux_loss, int32_t *slot, int32_t *kept, int32_t *expert_offsets,
                       int32_t *row_token, void *x_perm, void *h, void *y_perm, void *out, void *ws,
                       moe_stream_t stream);

/*
 * Expert-choice routing ([Wiki] "Mixture-of-Experts", section 横断的知見: the
 * experts pick their top-k tokens instead of the tokens picking experts), for
 * layers with cfg->expert_choice = 1. Read with the rest of the layer: the
 * scores are eq. (1)'s softmax over the experts, p [T, E]; expert e takes the
 * Ce = min(C, T) tokens with the largest p[:, e] (descending, ties to the
 * lower token index) and keeps them in ascending token order as its group of
 * rows e Ce .. e Ce + Ce - 1; a chosen (t, e)'s gate is p[t, e]; a token can
 * be chosen by any number of experts, or none. rows = moe_max_rows(cfg) =
 * E * Ce. The balance is built in: no auxiliary loss is formed.
 *
 * Router: probs [T, E] fp32 out (required), row_token [rows] int32 out (the
 * token of each row), row_gate [rows] fp32 out (its gate), expert_offsets
 * [E + 1] int32 out (e Ce), importance [E] fp32 out (sum_t p[t, e]).
 * The expert FFNs are moe_expert_gemm with these offsets.
 */
moe_status moe_router_expert_choice(const moe_config *cfg, const void *x, const float *w_r,
                                    const float *logit_bias, float *probs, int32_t *row_token,
                                    float *row_gate, int32_t *expert_offsets, float *importance,
                                    void *ws, moe_stream_t stream);
/* x_perm [rows, d] out: x_perm[row] = x[row_token[row]]. */
moe_status moe_dispatch_expert_choice(const moe_config *cfg, const void *x, const int32_t *row_token,
                                      void *x_perm, moe_stream_t stream);
/* out[t] = x[t] (only with cfg->add_residual) + sum over the rows whose token
 * is t of row_gate[row] * y_perm[row], in expert order, summed in fp32 and
 * rounded once. out [T, d] may not alias x or y_perm. */
moe_status moe_combine_expert_choice(const moe_config *cfg, const void *x, const void *y_perm,
                                     const int32_t *row_token, const float *row_gate, void *out,
                                     void *ws, moe_stream_t stream);

/* Everything the forward pass produced that the backward pass reads. */
typedef struct moe_saved {
  const void *x;                  /* [T, d] */
  const float *w_r;               /* [E, d] */
  const void *w1;                 /* [E, R1, d] */
  const void *w2;                 /* [E, d, F] */
  const float *probs;             /* [T, E] */
  const int32_t *topk_idx;        /* [T, k] */
  const float *topk_gate;         /* [T, k] */
  const int32_t *slot;            /* [T, k] */
  const int32_t *expert_offsets;  /* [E + 1] */
  const int32_t *load;            /* [E] */
  const void *x_perm;             /* [rows, d] */
  const void *pre_act;            /* [rows, 2F] (SwiGLU) or NULL (ReLU) */
  const void *h;                  /* [rows, F] */
  const void *y_perm;             /* [rows, d] */
} moe_saved;

/* The expert-choice forward pass's saved tensors. */
typedef struct moe_saved_expert_choice {
  const void *x;                  /* [T, d] */
  const float *w_r;               /* [E, d] */
  const void *w1;                 /* [E, R1, d] */
  const void *w2;                 /* [E, d, F] */
  const float *probs;             /* [T, E] */
  const int32_t *row_token;       /* [rows] */
  const float *row_gate;          /* [rows] */
  const int32_t *expert_offsets;  /* [E + 1] */
  const void *x_perm;             /* [rows, d] */
  const void *pre_act;            /* [rows, 2F] (SwiGLU) or NULL (ReLU) */
  const void *h;                  /* [rows, F] */
  const void *y_perm;             /* [rows, d] */
} moe_saved_expert_choice;

/* Backward of an expert-choice layer's L = <dY, out> (the choices held
 * constant): dx, dw_r, dw1, dw2 as in moe_backward. */
moe_status moe_backward_expert_choice(const moe_config *cfg, const moe_saved_expert_choice *saved,
                                      const void *dy, void *dx, float *dw_r, void *dw1, void *dw2,
                                      void *ws, moe_stream_t stream);

/*
 * Backward of L = <dY, out> + aux, with the top-k sets, capacity masks and
 * f_e held constant ([Switch] section 負荷分散損失: f comes from an argmax and
 * carries no gradient; P does, through eq. (1)).
 *
 *   dy   [T, d]      x dtype
 *   dx   [T, d]      x dtype out: dY (residual; only when cfg->add_residual) +
 *                    expert path + router path
 *   dw_r [E, d]      fp32 out
 *   dw1  [E, R1, d]  x dtype out
 *   dw2  [E, d, F]   x dtype out
 * The fixed logit bias gets no gradient.
 *
 * bf16 layers with 0 < cfg->capacity <= 192 take the expert weight gradients
 * from a kernel that keeps each (expert, 128-row tile) unit's rows of dYp /
 * dA in shared memory across the unit's output tiles; it relies on every
 * expert's packed rows being at most cfg->capacity (true for offsets from
 * this layer's dispatch) and records MOE_DEVERR_GROUP_ROWS otherwise.
 * MOE_WGRAD=gemm in the environment (read at every call) sends them to the
 * grouped GEMM instead, as do CTA-pair tiles; results agree to fp32
 * accumulation order.
 */
moe_status moe_backward(const moe_config *cfg, const moe_saved *saved, const void *dy, void *dx,
                        float *dw_r, void *dw1, void *dw2, void *ws, moe_stream_t stream);

/* Device pointers, inside `ws`, of the backward pass's intermediates, valid
 * after moe_backward: dyp [rows, d] (g * dY per packed row), da [rows, R1]
 * (gradient at the expert's pre-activations), dxp [rows, d] (gradient at
 * x_perm), dg [T, k] fp32 (gradient at the gates), dh [T, E] fp32 (gradient
 * at the router logits). Any output pointer may be NULL. */
moe_status moe_backward_intermediates(const moe_config *cfg, void *ws, void **dyp, void **da,
                                      void **dxp, float **dg, float **dh);

/* Synchronises `stream`, returns the first error code a kernel recorded in
 * `ws` since the last call (MOE_DEVERR_*) in *code, and clears it. */
moe_status moe_get_device_error(void *ws, moe_stream_t stream, int32_t *code);

/* Self-test of the bounded on-chip waits the kernels use (every mbarrier wait
 * gives up after 4 s without progress, records MOE_DEVERR_TIMEOUT in the
 * workspace's error word and lets its kernel return). Launches one block that
 * runs that wait on a barrier nothing completes: after about 4 s the wait gives
 * up and the block exits. Afterwards moe_get_device_error reports
 * MOE_DEVERR_TIMEOUT. `ws` is any workspace (only its error word is used). */
moe_status moe_selftest_bounded_wait(void *ws, moe_stream_t stream);

const char *moe_status_string(moe_status s);
/* Text of the last CUDA error seen by a call that returned MOE_ERR_CUDA. */
const char *moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
