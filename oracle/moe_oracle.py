"""CPU oracle for the sparsely-gated Mixture-of-Experts FFN layer (test infrastructure).

This is a plain, slow, fp64 restatement of what the layer computes. Only the
tests, the package's smoke check and the benchmark's CPU-baseline leg may use
it; the CUDA library never calls it and shares no code with it.

Pages followed (cited by title and section/equation):

* [Switch] "Mixture of Experts (MoE) を1から解説 — Switch Transformerのルーティング
  と負荷分散": eq. (1) softmax router, eq. (2) gated sum over the selected
  experts, eq. (3) expert capacity and the dropped-token rule (section
  エキスパートには「定員」がある), eq. (4) load-balancing loss and its numpy
  sketch (section 負荷分散損失), fp32 router (section 学習を安定させる3つの工夫).
* [LRMoE] "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE Training on
  Memory-Constrained Nodes" (section この記事のポイント): kept token-expert
  pairs are physically compacted into variable-size groups per expert.
* [Wiki] "Mixture-of-Experts" (notes.yuuk.io): top-k lineage beyond k = 1,
  SwiGLU experts, importance/load statistics.

Readings taken where the pages are silent (the same list is kept in the
project's design notes):

* W_r is stored [E, d]; h = W_r x (+ a fixed logit bias b when given).
* Top-k is chosen on h: descending value, ties to the lower expert index.
* Gates are the raw p_i of the selected experts (eq. (2)); with
  renormalisation g_i = p_i / sum_{j in T} p_j over all k selected experts
  (dropped ones stay in the denominator and contribute nothing).
* Capacity C = floor(n * cf / E), n = k*T assignments by default (keeps the
  "cf = 1.0 fits a perfectly balanced batch" meaning for k > 1), n = T when
  count_assignments is off; no limit when cf is None.
* Within an expert, assignments are ranked in ascending token order; rank < C
  is kept (slot = rank), the rest are dropped (slot = -1).
* out = x + sum over kept selected experts of g * E_i(x); a token whose
  assignments are all dropped returns x unchanged. With add_residual off the
  layer returns the gated sum alone (zeros for such a token): the residual
  connection is the caller's.
* f_e = load_e / (T*k) counted before capacity, P_e = importance_e / T,
  aux = alpha * E * sum_e f_e P_e.
* Experts have no biases. ReLU: W2 relu(W1 z). SwiGLU: W2 (silu(Wg z) * (Wu z)),
  W1 = [Wg; Wu] stacked by rows, silu(u) = u / (1 + exp(-u)).
* Backward of L = <dY, out> + aux with top-k sets, capacity masks and f held
  constant.
* Router variants (score = sigmoid or sqrt_softplus, a selection-only
  correction bias): p is the score, importance sums it, the gates are p of
  the chosen experts, the choice is on p + b (on h without a bias); see
  router_variants.py.

Parity status: every function here is pinned by the oracle tests (invariants,
closed forms, brute force on tiny inputs, finite differences); none is
"parity unpinned".
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence, Tuple, Union

import numpy as np

from . import router_variants as RV

ExpertSource = Union[Tuple[np.ndarray, np.ndarray], Callable[[int], Tuple[np.ndarray, np.ndarray]]]


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _expert(experts: ExpertSource, e: int) -> Tuple[np.ndarray, np.ndarray]:
    if callable(experts):
        w1, w2 = experts(e)
    else:
        w1, w2 = experts[0][e], experts[1][e]
    return _f64(w1), _f64(w2)


# ------------------------------------------------------------------ router
def router_logits(x, w_r, bias=None) -> np.ndarray:
    """h = W_r . x per token ([Switch] section 仕組み(1)), plus the fixed bias."""
    h = _f64(x) @ _f64(w_r).T
    if bias is not None:
        h = h + _f64(bias)[None, :]
    return h


def softmax(h: np.ndarray) -> np.ndarray:
    """p_i = exp(h_i) / sum_j exp(h_j) over all N experts ([Switch] eq. (1)).

    The row maximum is subtracted first; the quotient is unchanged by it.
    """
    z = np.exp(h - h.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def score_grad(h: np.ndarray, p: np.ndarray, dp: np.ndarray, score: str) -> np.ndarray:
    """dL/dh from dL/dp through the score function: the softmax Jacobian of eq. (1),
    p (dp - <p, dp>); elementwise scores multiply by their derivative,
    sigmoid' = p (1 - p) and sqrt(softplus)'(h) = sigmoid(h) / (2 sqrt(softplus(h)))."""
    if score == "softmax":
        return p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    if score == "sigmoid":
        return p * (1.0 - p) * dp
    if score == "sqrt_softplus":
        return (1.0 / (1.0 + np.exp(-h))) / (2.0 * p) * dp
    raise ValueError(score)


def top_k(h: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, largest first, ties to the
    lower index ([Switch] section 仕組み(1): "上位k個を選び"; k = 1 is the
    argmax of the numpy sketch in section 負荷分散損失)."""
    order = np.argsort(-h, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def route(x, w_r, bias, k: int, renormalize: bool, alpha: float, score: str = "softmax",
          sel_bias=None, reroute: bool = False) -> dict:
    """Router, gates and balance statistics for one batch of T tokens.

    [Switch] eqs. (1), (2), (4) and the numpy sketch of section 負荷分散損失:
    probs -> expert choice -> gate -> f (fraction of assignments per expert)
    -> P (mean probability) -> aux = alpha * N * sum f_i P_i.

    `score` and `sel_bias` are the router variants of [Wiki] section 横断的知見
    (router_variants.py states them): p is then the elementwise score, and
    with a correction bias the experts are chosen on p + b while the gates
    stay p. Without a bias the choice is the top-k of h, which is the order
    of p for the softmax and for every strictly increasing score.

    With `reroute` (No-Token-Left-Behind, top-1 layers only) the two best
    experts of each token are kept, idx [T, 2] and gates [T, 2] (the second
    the token's candidate when its first choice overflows); the load and f
    still count the first choices, the layer's routing decision.
    """
    h = router_logits(x, w_r, bias)
    T, E = h.shape
    p = softmax(h) if score == "softmax" else RV.scores(h, score)
    if reroute and (k != 1 or renormalize or E < 2):
        raise ValueError("No-Token-Left-Behind rerouting is defined for top-1 layers of two or more experts")
    kk = 2 if reroute else k
    idx = top_k(h, kk) if sel_bias is None else RV.select(p, kk, sel_bias)
    gate = np.take_along_axis(p, idx, axis=1)
    if renormalize:
        gate = gate / gate.sum(axis=1, keepdims=True)
    load = np.bincount((idx[:, 0] if reroute else idx).ravel(), minlength=E).astype(np.int64)
    importance = p.sum(axis=0)
    f = load / float(T * k)
    P = importance / float(T)
    aux = alpha * E * float(np.sum(f * P))
    return dict(h=h, p=p, idx=idx, gate=gate, load=load, importance=importance,
                f=f, P=P, aux=aux)


# ------------------------------------------------------------------ capacity
def capacity(T: int, E: int, k: int, cf: Optional[Tuple[int, int]],
             count_assignments: bool = True) -> Optional[int]:
    """expert capacity = tokens per batch / number of experts * capacity factor
    ([Switch] eq. (3)), floored, in integer arithmetic. None = no limit."""
    if cf is None:
        return None
    num, den = cf
    n = (k * T) if count_assignments else T
    return (n * num) // (E * den)


def assign_slots(idx: np.ndarray, E: int, C: Optional[int]) -> dict:
    """Token-order capacity slots ([Switch] eq. (3) and the dropped-token rule).

    Each expert takes the tokens that chose it in ascending token order; the
    first C are kept (slot = their rank), later ones are dropped (slot = -1)
    and skip the expert. Kept pairs are compacted per expert into contiguous
    row groups ([LRMoE] physical compaction -> variable-size groups):
    row(t, j) = offsets[e] + slot.
    """
    T, k = idx.shape
    count = np.zeros(E, dtype=np.int64)
    slot = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            r = count[e]
            count[e] += 1
            if C is None or r < C:
                slot[t, j] = r
    kept = count.copy() if C is None else np.minimum(count, C)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    row_token = np.full(int(offsets[-1]), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            if slot[t, j] >= 0:
                row_token[offsets[idx[t, j]] + slot[t, j]] = t
    return dict(slot=slot, kept=kept, offsets=offsets, row_token=row_token)


def assign_slots_reroute(idx2: np.ndarray, E: int, C: Optional[int]) -> dict:
    """No-Token-Left-Behind ([Switch] section 論文の限界と、まだ分かっていないこと:
    overflow goes to the token's second candidate), read for top-1 layers.

    Round 1 is the dropped-token rule on the first choices: each expert takes
    its tokens in ascending token order and keeps the first C. Round 2: every
    token dropped in round 1 offers its second-choice expert, in ascending
    token order, the room that expert has left; slots continue after the
    round-1 ones. slot[t, 0] is the round-1 slot, slot[t, 1] the round-2 one
    (-1 where the assignment is not kept); a token keeps at most one.
    """
    T = idx2.shape[0]
    slot = np.full((T, 2), -1, dtype=np.int64)
    count = np.zeros(E, dtype=np.int64)
    for t in range(T):
        e = int(idx2[t, 0])
        if C is None or count[e] < C:
            slot[t, 0] = count[e]
        count[e] += 1
    fill = count.copy() if C is None else np.minimum(count, C)
    for t in range(T):
        if slot[t, 0] >= 0:
            continue
        e = int(idx2[t, 1])
        if C is None or fill[e] < C:
            slot[t, 1] = fill[e]
            fill[e] += 1
    kept = fill
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(kept)
    row_token = np.full(int(offsets[-1]), -1, dtype=np.int64)
    for t in range(T):
        for j in range(2):
            if slot[t, j] >= 0:
                row_token[offsets[idx2[t, j]] + slot[t, j]] = t
    return dict(slot=slot, kept=kept, offsets=offsets, row_token=row_token)


def _routing(x64, w_r, bias, k, renormalize, alpha, score, sel_bias, reroute, cf, count_assignments):
    """Route, capacity and slots of one batch, as forward and backward share them."""
    r = route(x64, w_r, bias, k, renormalize, alpha, score, sel_bias, reroute)
    T = x64.shape[0]
    E = r["p"].shape[1]
    C = capacity(T, E, k, cf, count_assignments)
    s = assign_slots_reroute(r["idx"], E, C) if reroute else assign_slots(r["idx"], E, C)
    return r, C, s


# ------------------------------------------------------------------ experts
def silu(u):
    return u / (1.0 + np.exp(-u))


def expert_ffn(z: np.ndarray, w1: np.ndarray, w2: np.ndarray, act: str) -> dict:
    """One expert FFN on rows z [n, d] ([Switch] section 直感: the experts are
    copies of the Transformer FFN; SwiGLU from [Wiki])."""
    if act == "relu":
        a = z @ w1.T
        hid = np.maximum(a, 0.0)
        return dict(a=a, hid=hid, y=hid @ w2.T)
    F = w2.shape[1]
    g = z @ w1[:F].T
    u = z @ w1[F:].T
    hid = silu(g) * u
    return dict(g=g, u=u, hid=hid, y=hid @ w2.T)


# ------------------------------------------------------------------ layer
def forward(x, w_r, bias, experts: ExpertSource, *, k: int, act: str,
            cf: Optional[Tuple[int, int]], count_assignments: bool = True,
            renormalize: bool = False, alpha: float = 0.01,
            tokens: Optional[Sequence[int]] = None, add_residual: bool = True, score: str = "softmax",
            sel_bias=None, reroute: bool = False) -> dict:
    """out = x + sum_{i in T, kept} g_i E_i(x) ([Switch] eq. (2) with the
    residual passthrough of dropped tokens); without the residual
    (add_residual=False) out is the gated sum alone, and a token whose
    assignments are all dropped gets zeros.

    `tokens` restricts the expert evaluation (and `out`) to a subset of
    tokens; routing, slots and statistics always cover the whole batch,
    because capacity depends on every token before a given one.
    """
    x64 = _f64(x)
    T, d = x64.shape
    E = np.asarray(w_r).shape[0]
    r, C, s = _routing(x64, w_r, bias, k, renormalize, alpha, score, sel_bias, reroute, cf, count_assignments)
    sel = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = x64[sel].copy() if add_residual else np.zeros((len(sel), d))
    where = {int(t): i for i, t in enumerate(sel)}
    for e in range(E):
        tt, jj = np.nonzero((r["idx"] == e) & (s["slot"] >= 0))
        keep = [n for n, t in enumerate(tt) if int(t) in where]
        if not keep:
            continue
        tt, jj = tt[keep], jj[keep]
        w1, w2 = _expert(experts, e)
        y = expert_ffn(x64[tt], w1, w2, act)["y"]
        for n in range(len(tt)):
            out[where[int(tt[n])]] += r["gate"][tt[n], jj[n]] * y[n]
    res = dict(r)
    res.update(s)
    res.update(C=C, out=out, tokens=sel)
    return res


def backward(x, w_r, bias, experts: ExpertSource, dy, *, k: int, act: str,
             cf: Optional[Tuple[int, int]], count_assignments: bool = True,
             renormalize: bool = False, alpha: float = 0.01,
             experts_needed: Optional[Sequence[int]] = None, add_residual: bool = True,
             score: str = "softmax", sel_bias=None, reroute: bool = False) -> dict:
    """Gradients of L = <dY, out> + aux (chain rule through eqs. (1), (2), (4)).

    Top-k sets, capacity masks and f are constants ([Switch] section
    負荷分散損失: f comes from an argmax and has no gradient; P does).
    Returns dx [T, d], dw_r [E, d], dg [T, k] and, for every expert in
    `experts_needed` (all by default), dw1[e] and dw2[e].
    """
    x64, dy64 = _f64(x), _f64(dy)
    T, d = x64.shape
    wr64 = _f64(w_r)
    E = wr64.shape[0]
    r, C, s = _routing(x64, wr64, bias, k, renormalize, alpha, score, sel_bias, reroute, cf, count_assignments)
    dx = dy64.copy() if add_residual else np.zeros_like(dy64)   # residual path
    dg = np.zeros(r["idx"].shape)         # [T, k] ([T, 2] with rerouting)
    dw1, dw2 = {}, {}
    need = set(range(E)) if experts_needed is None else set(int(e) for e in experts_needed)
    for e in range(E):
        tt, jj = np.nonzero((r["idx"] == e) & (s["slot"] >= 0))
        w1, w2 = _expert(experts, e)
        if len(tt) == 0:
            if e in need:
                dw1[e], dw2[e] = np.zeros_like(w1), np.zeros_like(w2)
            continue
        z = x64[tt]
        fw = expert_ffn(z, w1, w2, act)
        g = r["gate"][tt, jj][:, None]
        dg[tt, jj] = np.sum(dy64[tt] * fw["y"], axis=1)
        dyp = g * dy64[tt]                 # d(out)/d(y_e) = g
        dhid = dyp @ w2
        if e in need:
            dw2[e] = dyp.T @ fw["hid"]
        if act == "relu":
            da = dhid * (fw["a"] > 0)
            dz = da @ w1
            if e in need:
                dw1[e] = da.T @ z
        else:
            sg = 1.0 / (1.0 + np.exp(-fw["g"]))
            dgate = dhid * fw["u"] * (sg * (1.0 + fw["g"] * (1.0 - sg)))
            dup = dhid * silu(fw["g"])
            da = np.concatenate([dgate, dup], axis=1)
            dz = da @ w1
            if e in need:
                dw1[e] = da.T @ z
        dx[tt] += dz
    # gates -> probabilities
    p, idx = r["p"], r["idx"]
    dp = np.zeros((T, E))
    if renormalize:
        psel = np.take_along_axis(p, idx, axis=1)
        S = psel.sum(axis=1, keepdims=True)
        corr = np.sum(dg * r["gate"], axis=1, keepdims=True)
        np.put_along_axis(dp, idx, (dg - corr) / S, axis=1)
    else:
        np.put_along_axis(dp, idx, dg, axis=1)
    # eq. (4): d aux / d p_{t,e} = alpha * E * f_e / T
    dp += alpha * E * r["f"][None, :] / float(T)
    # eq. (1): softmax Jacobian (or the elementwise score's derivative)
    dh = score_grad(r["h"], p, dp, score)
    dw_r = dh.T @ x64
    dx += dh @ wr64
    return dict(dx=dx, dw_r=dw_r, dg=dg, dh=dh, dw1=dw1, dw2=dw2, route=r, slots=s)


def backward_sampled(x, w_r, bias, experts: ExpertSource, dy, *, tokens: Sequence[int],
                     experts_sampled: Sequence[int], k: int, act: str, cf: Optional[Tuple[int, int]],
                     count_assignments: bool = True, renormalize: bool = False, alpha: float = 0.01,
                     add_residual: bool = True, score: str = "softmax", sel_bias=None,
                     reroute: bool = False) -> dict:
    """The gradients of `backward` for a few tokens (dx, dg and dh rows) and a
    few experts (dw1, dw2), without evaluating every expert on every token:
    the same chain rule through eqs. (1), (2) and (4). Each expert the
    sampled tokens keep, or that is sampled itself, is fetched once; it gives
    the sampled tokens' gate gradients and expert-path dx terms, and, for a
    sampled expert, the weight gradients over every row it kept. Then, token
    by token, the gate gradients go through the renormalisation and the
    softmax Jacobian (plus the aux term, which depends on the batch only
    through f) to dh and the router's dx term. Routing and capacity always
    cover the whole batch."""
    x64, dy64 = _f64(x), _f64(dy)
    T, d = x64.shape
    wr64 = _f64(w_r)
    E = wr64.shape[0]
    r, C, s = _routing(x64, wr64, bias, k, renormalize, alpha, score, sel_bias, reroute, cf, count_assignments)
    p, idx, gate, slot = r["p"], r["idx"], r["gate"], s["slot"]
    toks = [int(t) for t in tokens]
    sampled = set(int(e) for e in experts_sampled)

    def expert_grads(z, dyv, g, w1, w2):
        fw = expert_ffn(z, w1, w2, act)
        dyp = g[:, None] * dyv
        dhid = dyp @ w2
        if act == "relu":
            da = dhid * (fw["a"] > 0)
        else:
            sg = 1.0 / (1.0 + np.exp(-fw["g"]))
            da = np.concatenate([dhid * fw["u"] * (sg * (1.0 + fw["g"] * (1.0 - sg))), dhid * silu(fw["g"])], axis=1)
        return fw, dyp, da

    acc = {t: dy64[t].copy() if add_residual else np.zeros(d) for t in toks}   # residual path
    kc = idx.shape[1]                                 # k columns (2 with rerouting)
    dg = {t: np.zeros(kc) for t in toks}
    pairs = {}                                        # expert -> the sampled tokens' kept pairs (t, j)
    for t in toks:
        for j in range(kc):
            if slot[t, j] >= 0:
                pairs.setdefault(int(idx[t, j]), []).append((t, j))
    dw1, dw2 = {}, {}
    for e in sorted(set(pairs) | sampled):
        w1, w2 = _expert(experts, e)
        if e in pairs:
            tt = np.array([t for t, _ in pairs[e]])
            jj = np.array([j for _, j in pairs[e]])
            fw, _, da = expert_grads(x64[tt], dy64[tt], gate[tt, jj], w1, w2)
            dz = da @ w1
            for n, (t, j) in enumerate(pairs[e]):
                dg[t][j] = float(np.dot(dy64[t], fw["y"][n]))
                acc[t] += dz[n]
        if e in sampled:
            tt, jj = np.nonzero((idx == e) & (slot >= 0))
            if len(tt) == 0:
                dw1[e], dw2[e] = np.zeros_like(w1), np.zeros_like(w2)
                continue
            fw, dyp, da = expert_grads(x64[tt], dy64[tt], gate[tt, jj], w1, w2)
            dw2[e] = dyp.T @ fw["hid"]
            dw1[e] = da.T @ x64[tt]
    dx, dh = {}, {}
    for t in toks:
        dp = np.zeros(E)
        if renormalize:
            psel = p[t, idx[t]]
            dp[idx[t]] = (dg[t] - np.dot(dg[t], gate[t])) / psel.sum()
        else:
            dp[idx[t]] = dg[t]
        dp += alpha * E * r["f"] / float(T)
        dh[t] = score_grad(r["h"][t:t + 1], p[t:t + 1], dp[None, :], score)[0]
        dx[t] = acc[t] + dh[t] @ wr64
    return dict(dx=dx, dg=dg, dh=dh, dw1=dw1, dw2=dw2, route=r, slots=s)


def loss(x, w_r, bias, experts: ExpertSource, dy, **kw) -> float:
    """L = <dY, out> + aux, the scalar whose gradient `backward` returns."""
    f = forward(x, w_r, bias, experts, **kw)
    return float(np.sum(_f64(dy) * f["out"])) + f["aux"]


# ------------------------------------------------------------------ expert-choice routing
def route_expert_choice(x, w_r, bias, C: int) -> dict:
    """Expert-choice routing ([Wiki] "Mixture-of-Experts", section 横断的知見: the
    experts pick their top-k tokens instead of the tokens picking experts).

    Read with the rest of the layer: the scores are eq. (1)'s softmax over the
    experts, p [T, E]; expert e takes the min(C, T) tokens with the largest
    p[:, e] (descending, ties to the lower token index), kept in ascending
    token order as its group of rows; the gate of a chosen (t, e) is p[t, e].
    A token can be chosen by any number of experts, or none. importance_e =
    sum_t p[t, e]; load_e = the number chosen. The balance is built in, so no
    auxiliary loss is formed.
    """
    h = router_logits(x, w_r, bias)
    T, E = h.shape
    p = softmax(h)
    Ce = min(C, T)
    chosen = np.zeros((E, Ce), dtype=np.int64)
    for e in range(E):
        order = sorted(range(T), key=lambda t: (-p[t, e], t))      # descending score, ties to the lower token
        chosen[e] = np.sort(order[:Ce])
    gate = np.take_along_axis(p.T, chosen, axis=1)                  # [E, Ce]
    load = np.full(E, Ce, dtype=np.int64)
    return dict(h=h, p=p, chosen=chosen, gate=gate, importance=p.sum(axis=0), load=load,
                offsets=np.arange(E + 1, dtype=np.int64) * Ce, row_token=chosen.reshape(-1))


def forward_expert_choice(x, w_r, bias, experts: ExpertSource, *, C: int, act: str,
                          add_residual: bool = True) -> dict:
    """out_t = x_t + sum over the experts e that chose t of p[t, e] E_e(x_t)."""
    x64 = _f64(x)
    r = route_expert_choice(x64, w_r, bias, C)
    out = x64.copy() if add_residual else np.zeros_like(x64)
    for e in range(r["p"].shape[1]):
        tt = r["chosen"][e]
        if len(tt) == 0:
            continue
        w1, w2 = _expert(experts, e)
        y = expert_ffn(x64[tt], w1, w2, act)["y"]
        out[tt] += r["gate"][e][:, None] * y              # tt has no repeats within one expert
    res = dict(r)
    res.update(out=out)
    return res


def backward_expert_choice(x, w_r, bias, experts: ExpertSource, dy, *, C: int, act: str,
                           add_residual: bool = True) -> dict:
    """Gradients of L = <dY, out> with the choices held constant: the chain rule
    through each chosen pair's gate p[t, e] and expert, then eq. (1)'s softmax
    Jacobian. dg [E, Ce] is the gradient at each chosen pair's gate."""
    x64, dy64 = _f64(x), _f64(dy)
    wr64 = _f64(w_r)
    r = route_expert_choice(x64, wr64, bias, C)
    T, E = r["p"].shape
    dx = dy64.copy() if add_residual else np.zeros_like(dy64)
    dg = np.zeros_like(r["gate"])
    dp = np.zeros((T, E))
    dw1, dw2 = {}, {}
    for e in range(E):
        tt = r["chosen"][e]
        w1, w2 = _expert(experts, e)
        if len(tt) == 0:
            dw1[e], dw2[e] = np.zeros_like(w1), np.zeros_like(w2)
            continue
        z = x64[tt]
        fw = expert_ffn(z, w1, w2, act)
        g = r["gate"][e][:, None]
        dg[e] = np.sum(dy64[tt] * fw["y"], axis=1)
        dp[tt, e] = dg[e]
        dyp = g * dy64[tt]
        dhid = dyp @ w2
        dw2[e] = dyp.T @ fw["hid"]
        if act == "relu":
            da = dhid * (fw["a"] > 0)
        else:
            sg = 1.0 / (1.0 + np.exp(-fw["g"]))
            da = np.concatenate([dhid * fw["u"] * (sg * (1.0 + fw["g"] * (1.0 - sg))), dhid * silu(fw["g"])], axis=1)
        dw1[e] = da.T @ z
        dx[tt] += da @ w1
    dh = score_grad(r["h"], r["p"], dp, "softmax")
    dx += dh @ wr64
    return dict(dx=dx, dw_r=dh.T @ x64, dg=dg, dh=dh, dw1=dw1, dw2=dw2, route=r)
