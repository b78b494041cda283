"""CPU oracle for router variants of the same layer (test infrastructure).

Like moe_oracle, this is plain fp64 numpy that only the tests may use. The
layer oracle (moe_oracle.route / forward / backward) takes its score
functions and selection from here.

Page followed: [Wiki] "Mixture-of-Experts" (notes.yuuk.io), section 横断的知見,
which names three changes to the router without giving formulas:

* sigmoid gating instead of the softmax (no zero-sum constraint across the
  experts), together with a learnable per-expert bias;
* sqrt(Softplus(.)) as the gating function that follows the sigmoid;
* auxiliary-loss-free load balancing: each token selects its experts with a
  per-expert correction bias added to the routing scores, while the weights
  of the selected experts are the original scores.

Readings taken (the plainest ones the page supports):

* score s_e = g(h_e), h = W_r x (+ fixed logit bias), with g the softmax over
  the experts, the elementwise sigmoid 1 / (1 + exp(-h)), or the elementwise
  sqrt(log(1 + exp(h)));
* selection: the k largest s_e + b_e per token (b = correction bias, zero when
  absent), descending, ties to the lower expert index;
* gates: s_e of the selected experts (the correction bias does not enter),
  divided by their sum when renormalising;
* correction-bias update after a batch, the sign rule of the method the page
  cites: b_e <- b_e + gamma * sign(mean_e(load) - load_e), so overloaded
  experts are pushed down and underloaded ones up (no change at the mean);
* with softmax scores and no correction bias, everything reduces to
  moe_oracle.route.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

SCORES = ("softmax", "sigmoid", "sqrt_softplus")


def scores(h: np.ndarray, kind: str) -> np.ndarray:
    """Routing scores from the logits h [T, E]."""
    h = np.asarray(h, dtype=np.float64)
    if kind == "softmax":
        z = np.exp(h - h.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if kind == "sigmoid":
        return 1.0 / (1.0 + np.exp(-h))
    if kind == "sqrt_softplus":
        return np.sqrt(np.logaddexp(0.0, h))   # log(1 + exp(h)) without overflow
    raise ValueError(f"unknown score function {kind!r}")


def select(s: np.ndarray, k: int, sel_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """Indices of the k largest s + b per token, largest first, ties to the lower index."""
    key = np.asarray(s, dtype=np.float64)
    if sel_bias is not None:
        key = key + np.asarray(sel_bias, dtype=np.float64)[None, :]
    order = np.argsort(-key, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def route_variant(h: np.ndarray, k: int, kind: str = "softmax", sel_bias: Optional[np.ndarray] = None,
                  renormalize: bool = False) -> dict:
    """Scores, selection (with the correction bias), gates (without it) and the per-expert load."""
    s = scores(h, kind)
    idx = select(s, k, sel_bias)
    gate = np.take_along_axis(s, idx, axis=1)
    if renormalize:
        gate = gate / gate.sum(axis=1, keepdims=True)
    load = np.bincount(idx.ravel(), minlength=s.shape[1]).astype(np.int64)
    return dict(s=s, idx=idx, gate=gate, load=load)


def update_bias(bias: np.ndarray, load: np.ndarray, gamma: float) -> np.ndarray:
    """b_e + gamma * sign(mean(load) - load_e)."""
    load = np.asarray(load, dtype=np.float64)
    return np.asarray(bias, dtype=np.float64) + gamma * np.sign(load.mean() - load)
