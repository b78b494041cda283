"""Seeded synthetic inputs for the sparsely-gated Mixture-of-Experts FFN layer.

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests. It holds workload shapes, seeds and random draws only: no step
of the layer (router, top-k, capacity, experts, combine) is computed here.

What the draws follow:

* x ~ N(0, 1) (rounded to bf16 for the bf16 workloads, kept fp32 otherwise).
* Router and expert weights ~ N(0, s / sqrt(fan_in)) with the reduced init
  scale s = 0.1 ("Mixture of Experts (MoE) を1から解説 — Switch Transformerの
  ルーティングと負荷分散", section 学習を安定させる3つの工夫, item 2, Table 3).
  The second argument is the standard deviation. fan_in is d_model for the
  router, the first expert matrix (and the SwiGLU gate/up matrices) and d_ff
  for the second expert matrix. Two workloads scale the router to give
  N(0, 1)-sized logits instead (router_std = 1/sqrt(d_model)).
* An optional fixed per-expert logit bias b_e = ln(r^-s / sum_r r^-s),
  r = e + 1 (a Zipf(s) prior over experts) that forces skewed routing.
* Margin conditioning: a token whose k+1 largest router logits are not
  separated by at least MARGIN (every consecutive gap, evaluated in fp64 on
  the exact rounded x) is redrawn from a child seed (token, attempt) until it
  passes. This makes the top-k set and its order unique, so any correct
  implementation must pick the same experts in the same order. It is a filter
  on the input distribution, not part of the layer.

Seeds are per workload, per tensor and per expert, so one expert's weights can
be regenerated alone (SeedSequence over [base seed, crc32(workload),
crc32(tensor), index, attempt]; numpy PCG64).
"""
from __future__ import annotations

import dataclasses
import math
import zlib
from typing import Optional, Tuple

import numpy as np

MARGIN = 1e-3


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MoE-layer problem: shapes, dtypes, capacity rule and init scales."""

    name: str
    T: int                      # tokens in one call
    d: int                      # d_model
    E: int                      # number of experts N
    k: int                      # top-k
    F: int                      # d_ff of one expert
    act: str                    # 'relu' | 'swiglu'
    dtype: str                  # 'f32' | 'bf16' (x, expert weights, activations)
    cf: Optional[Tuple[int, int]]  # capacity factor as (num, den); None = no limit
    count_assignments: bool = True  # capacity counts k*T assignments (True) or T tokens
    renormalize: bool = False   # gates renormalised over the k selected experts
    router_std: Optional[float] = None  # None -> 0.1/sqrt(d)
    expert_scale: float = 0.1   # expert std = expert_scale / sqrt(fan_in)
    zipf_s: Optional[float] = None
    alpha: float = 0.01         # load-balancing loss coefficient
    add_residual: bool = True   # out = x + MoE(x) (True) or MoE(x)
    score: str = "softmax"      # router score function: softmax | sigmoid | sqrt_softplus
    reroute: bool = False       # No-Token-Left-Behind: a top-1 token dropped by capacity tries its 2nd choice
    backward: bool = False      # the workload includes the backward pass
    seed: int = 49

    @property
    def nm(self) -> int:
        """Weight matrices per expert: 2 for ReLU (W1, W2), 3 for SwiGLU."""
        return 3 if self.act == "swiglu" else 2

    @property
    def R1(self) -> int:
        """Rows of the first expert matrix: F (ReLU) or 2F (SwiGLU gate; up)."""
        return 2 * self.F if self.act == "swiglu" else self.F

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads. Sizes follow the Switch-Transformer and fine-grained
# MoE shapes these pages discuss.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny-top1-f32", T=512, d=64, E=8, k=1, F=128, act="relu",
                 dtype="f32", cf=(1, 1), backward=True),
        Workload("switch-base-top1", T=8192, d=768, E=128, k=1, F=3072,
                 act="relu", dtype="bf16", cf=(5, 4)),
        Workload("gshard-top2-zipf", T=16384, d=1024, E=64, k=2, F=4096,
                 act="relu", dtype="bf16", cf=(2, 1),
                 router_std=1.0 / math.sqrt(1024), zipf_s=1.2),
        Workload("dropless-top8-swiglu", T=16384, d=2048, E=128, k=8, F=768,
                 act="swiglu", dtype="bf16", cf=None, renormalize=True,
                 router_std=1.0 / math.sqrt(2048), backward=True),
        Workload("large-top8-swiglu", T=4096, d=7168, E=256, k=8, F=2048,
                 act="swiglu", dtype="bf16", cf=(5, 4), backward=True),
    ]
}


# ----------------------------------------------------------------- seeding
def rng_for(w: Workload, tensor: str, *index: int) -> np.random.Generator:
    words = [w.seed, zlib.crc32(w.name.encode()), zlib.crc32(tensor.encode())]
    words += [int(i) for i in index]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(words)))


# ----------------------------------------------------------------- bf16 helpers
def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); float32 out."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    u = (u + (((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF))) \
        & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def _cast(w: Workload, a: np.ndarray) -> np.ndarray:
    return round_bf16(a) if w.dtype == "bf16" else a.astype(np.float32)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(shape, dtype=np.float32)
    out *= np.float32(std)
    return out


# ----------------------------------------------------------------- draws
def router_weight(w: Workload) -> np.ndarray:
    std = w.router_std if w.router_std is not None else w.expert_scale / math.sqrt(w.d)
    return _normal(rng_for(w, "w_r"), (w.E, w.d), std)


def logit_bias(w: Workload) -> Optional[np.ndarray]:
    if w.zipf_s is None:
        return None
    r = np.arange(1, w.E + 1, dtype=np.float64)
    q = r ** (-w.zipf_s)
    return np.log(q / q.sum()).astype(np.float32)


def _token_margin(x: np.ndarray, w_r: np.ndarray, b: Optional[np.ndarray], k: int) -> np.ndarray:
    h = x.astype(np.float64) @ w_r.astype(np.float64).T
    if b is not None:
        h += b.astype(np.float64)
    m = min(k + 1, h.shape[1])
    if m < 2:
        return np.full(h.shape[0], np.inf)
    top = -np.sort(-h, axis=1)[:, :m]
    return (top[:, :-1] - top[:, 1:]).min(axis=1)


def tokens(w: Workload, w_r: np.ndarray, b: Optional[np.ndarray],
           margin: float = MARGIN, max_attempts: int = 1000) -> np.ndarray:
    """x [T, d] with every token margin-conditioned against (w_r, b) (over the k + 1 largest logits; k = 2
    when the second choice matters too, with rerouting)."""
    kk = 2 if w.reroute else w.k
    x = _cast(w, _normal(rng_for(w, "x"), (w.T, w.d), 1.0))
    bad = np.nonzero(_token_margin(x, w_r, b, kk) < margin)[0]
    attempt = 0
    while bad.size:
        attempt += 1
        if attempt > max_attempts:
            raise RuntimeError(f"{w.name}: margin conditioning did not converge")
        for t in bad:
            x[t] = _cast(w, _normal(rng_for(w, "x-redraw", int(t), attempt), (w.d,), 1.0))
        still = _token_margin(x[bad], w_r, b, kk) < margin
        bad = bad[still]
    return x


def expert_weights(w: Workload, e: int) -> Tuple[np.ndarray, np.ndarray]:
    """(W1_e [R1, d], W2_e [d, F]); for SwiGLU W1_e stacks gate rows then up rows."""
    w1 = _cast(w, _normal(rng_for(w, "w1", e), (w.R1, w.d), w.expert_scale / math.sqrt(w.d)))
    w2 = _cast(w, _normal(rng_for(w, "w2", e), (w.d, w.F), w.expert_scale / math.sqrt(w.F)))
    return w1, w2


def all_expert_weights(w: Workload) -> Tuple[np.ndarray, np.ndarray]:
    w1 = np.empty((w.E, w.R1, w.d), np.float32)
    w2 = np.empty((w.E, w.d, w.F), np.float32)
    for e in range(w.E):
        w1[e], w2[e] = expert_weights(w, e)
    return w1, w2


def expert_weight_bits(w: Workload, threads: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Every expert's (W1, W2) of a bf16 workload as bf16 bit patterns, uint16
    [E, R1, d] and [E, d, F] (half the memory of float32), drawn expert by
    expert on a thread pool. The values are exactly expert_weights(w, e):
    each expert has its own generator, so the order the threads run in does
    not matter. from_bf16_bits() widens one expert back to float32."""
    if w.dtype != "bf16":
        raise ValueError("expert_weight_bits is for bf16 workloads")
    import concurrent.futures
    import os
    b1 = np.empty((w.E, w.R1, w.d), np.uint16)
    b2 = np.empty((w.E, w.d, w.F), np.uint16)

    def one(e):
        a, b = expert_weights(w, e)
        b1[e] = bf16_bits(a)
        b2[e] = bf16_bits(b)

    n = threads or min(32, os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=n) as ex:
        list(ex.map(one, range(w.E)))
    return b1, b2


def upstream_grad(w: Workload) -> np.ndarray:
    """dY [T, d] ~ N(0, 1), the gradient of the loss w.r.t. the layer output."""
    return _cast(w, _normal(rng_for(w, "dy"), (w.T, w.d), 1.0))


def make_inputs(w: Workload, experts: bool = True, dy: Optional[bool] = None) -> dict:
    """All inputs of one workload as float32 numpy arrays (bf16-exact where bf16)."""
    w_r = router_weight(w)
    b = logit_bias(w)
    out = {"w_r": w_r, "bias": b, "x": tokens(w, w_r, b)}
    if experts:
        out["w1"], out["w2"] = all_expert_weights(w)
    if dy if dy is not None else w.backward:
        out["dy"] = upstream_grad(w)
    return out
