"""Pins for the CPU oracle: each check ties it to something other than itself.

Closed forms from the pages' equations, invariants the pages state, brute
force on tiny inputs, textbook loops, a library routine the oracle does not
use, and central finite differences for the backward pass.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special

import moe_synth as syn
from oracle import moe_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


# ------------------------------------------------------------------ eq. (1)
def test_softmax_closed_form():
    g = GOLD["softmax"]
    p = O.softmax(np.array([g["h"]]))
    np.testing.assert_allclose(p[0], g["p"], rtol=0, atol=1e-15)


def test_softmax_rows_sum_to_one_and_match_library():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((300, 17)) * 8.0
    p = O.softmax(h)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12
    np.testing.assert_allclose(p, scipy.special.softmax(h, axis=1), rtol=1e-13, atol=1e-300)
    # a shift of one row by a constant leaves it unchanged
    np.testing.assert_allclose(O.softmax(h + 123.0), p, rtol=1e-12)


# ------------------------------------------------------------------ top-k
def _brute_topk(h, k):
    """Rank by counting: rank(e) = #{e' beating e}; beating = larger, or equal with lower index."""
    T, E = h.shape
    out = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        for e in range(E):
            rank = sum(1 for f in range(E) if h[t, f] > h[t, e] or (h[t, f] == h[t, e] and f < e))
            if rank < k:
                out[t, rank] = e
    return out


@pytest.mark.parametrize("k", [1, 2, 3, 8])
def test_topk_brute_force(k):
    rng = np.random.default_rng(k)
    h = rng.standard_normal((40, 8))
    h[0, :] = 0.5                     # all tied: order must be 0, 1, 2, ...
    h[1, 3] = h[1, 5] = h[1].max() + 1
    np.testing.assert_array_equal(O.top_k(h, k), _brute_topk(h, k))
    assert list(O.top_k(h, k)[0]) == list(range(k))
    if k >= 2:
        assert list(O.top_k(h, k)[1][:2]) == [3, 5]


# ------------------------------------------------------------------ eq. (4)
def test_aux_uniform_is_alpha():
    g = GOLD["aux_uniform"]
    E, m = 8, 5
    T = E * m
    x = np.zeros((T, E))
    x[np.arange(T), np.arange(T) % E] = 1.0
    w_r = 3.0 * np.eye(E)                      # h_t = 3 * onehot(t mod E)
    r = O.route(x, w_r, None, 1, False, g["alpha"])
    np.testing.assert_allclose(r["f"], 1.0 / E, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["P"], 1.0 / E, rtol=1e-14)
    assert abs(r["aux"] - g["loss"]) <= 1e-15


def test_aux_collapsed_limit():
    g = GOLD["aux_collapsed"]
    E = g["N"]
    x = np.ones((16, 1))
    w_r = np.zeros((E, 1))
    w_r[0, 0] = 60.0                           # p_0 = 1 - O(e^-60)
    r = O.route(x, w_r, None, 1, False, g["alpha"])
    assert np.all(r["idx"] == 0) and r["f"][0] == 1.0
    assert abs(r["aux"] - g["loss_limit"]) <= 1e-15


def test_route_statistics_brute_force():
    rng = np.random.default_rng(3)
    T, E, d, k = 50, 6, 5, 2
    x = rng.standard_normal((T, d))
    w_r = rng.standard_normal((E, d))
    r = O.route(x, w_r, None, k, False, 0.01)
    load = np.zeros(E, int)
    imp = np.zeros(E)
    for t in range(T):
        hs = [sum(w_r[e, i] * x[t, i] for i in range(d)) for e in range(E)]
        zs = [math.exp(v) for v in hs]
        for e in range(E):
            imp[e] += zs[e] / sum(zs)
        for e in _brute_topk(np.array([hs]), k)[0]:
            load[e] += 1
    np.testing.assert_array_equal(r["load"], load)
    np.testing.assert_allclose(r["importance"], imp, rtol=1e-12)
    assert abs(r["f"].sum() - 1.0) < 1e-15 and abs(r["P"].sum() - 1.0) < 1e-12
    np.testing.assert_allclose(np.take_along_axis(r["p"], r["idx"], 1), r["gate"], rtol=0)


def test_renormalized_gates_sum_to_one():
    rng = np.random.default_rng(4)
    r = O.route(rng.standard_normal((30, 4)), rng.standard_normal((7, 4)), None, 3, True, 0.01)
    np.testing.assert_allclose(r["gate"].sum(axis=1), 1.0, rtol=1e-14)


# ------------------------------------------------------------------ eq. (3)
def test_capacity_closed_forms():
    for c in GOLD["capacity"]["cases"]:
        cf = tuple(c["cf"])
        assert O.capacity(c["T"], c["E"], c["k"], cf, True) == c["assignments"], c
        assert O.capacity(c["T"], c["E"], c["k"], cf, False) == c["tokens"], c
    assert O.capacity(100, 8, 1, None) is None


def _brute_slots(idx, E, C):
    T, k = idx.shape
    slot = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            rank = sum(1 for u in range(t) if e in idx[u])
            if C is None or rank < C:
                slot[t, j] = rank
    return slot


@pytest.mark.parametrize("k,C", [(1, 3), (2, 5), (3, 0), (2, None), (1, 64)])
def test_slots_brute_force_and_invariants(k, C):
    rng = np.random.default_rng(10 + k)
    T, E = 48, 6
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    s = O.assign_slots(idx, E, C)
    np.testing.assert_array_equal(s["slot"], _brute_slots(idx, E, C))
    load = np.bincount(idx.ravel(), minlength=E)
    kept = load if C is None else np.minimum(load, C)
    np.testing.assert_array_equal(s["kept"], kept)
    assert s["offsets"][-1] == (s["slot"] >= 0).sum()
    if C is not None:
        assert np.all(s["kept"] <= C)
    # every kept pair owns exactly one row, inside its expert's group
    for t in range(T):
        for j in range(k):
            if s["slot"][t, j] >= 0:
                e = idx[t, j]
                row = s["offsets"][e] + s["slot"][t, j]
                assert s["offsets"][e] <= row < s["offsets"][e + 1]
                assert s["row_token"][row] == t


# ------------------------------------------------------------------ experts
def _ffn_loops(z, w1, w2, act):
    n, d = z.shape
    F = w2.shape[1]
    y = np.zeros((n, w2.shape[0]))
    for r in range(n):
        hid = []
        for f in range(F):
            a = sum(w1[f, i] * z[r, i] for i in range(d))
            if act == "relu":
                hid.append(max(a, 0.0))
            else:
                u = sum(w1[F + f, i] * z[r, i] for i in range(d))
                hid.append(a / (1.0 + math.exp(-a)) * u)
        for o in range(w2.shape[0]):
            y[r, o] = sum(w2[o, f] * hid[f] for f in range(F))
    return y


@pytest.mark.parametrize("act", ["relu", "swiglu"])
def test_expert_ffn_textbook_loops(act):
    rng = np.random.default_rng(5)
    d, F = 6, 5
    z = rng.standard_normal((4, d))
    w1 = rng.standard_normal(((2 if act == "swiglu" else 1) * F, d))
    w2 = rng.standard_normal((d, F))
    np.testing.assert_allclose(O.expert_ffn(z, w1, w2, act)["y"], _ffn_loops(z, w1, w2, act), rtol=1e-12, atol=1e-13)


def test_silu_closed_forms():
    assert O.silu(np.array(0.0)) == 0.0
    assert abs(O.silu(np.array(math.log(3.0))) - 0.75 * math.log(3.0)) < 1e-15   # sigma(ln 3) = 3/4
    assert abs(O.silu(np.array(-60.0))) < 1e-24


# ------------------------------------------------------------------ eq. (2)
@pytest.mark.parametrize("act,k,renorm", [("relu", 1, False), ("relu", 2, False), ("swiglu", 3, True)])
def test_infinite_capacity_equals_dense_masked(act, k, renorm):
    """With no drops, out = x + sum over top-k of g_i E_i(x), using every expert
    evaluated densely on every token and a brute-force top-k mask."""
    w = syn.Workload("pin", T=24, d=8, E=5, k=k, F=6, act=act, dtype="f32", cf=None,
                     renormalize=renorm, router_std=0.5)
    inp = syn.make_inputs(w)
    f = O.forward(inp["x"], inp["w_r"], None, (inp["w1"], inp["w2"]), k=k, act=act, cf=None,
                  renormalize=renorm)
    x = inp["x"].astype(np.float64)
    h = x @ inp["w_r"].astype(np.float64).T
    p = scipy.special.softmax(h, axis=1)
    top = _brute_topk(h, k)
    ref = x.copy()
    for t in range(w.T):
        ys = [_ffn_loops(x[t:t + 1], inp["w1"][e].astype(np.float64), inp["w2"][e].astype(np.float64), act)[0]
              for e in range(w.E)]
        mask = np.zeros(w.E)
        mask[top[t]] = 1.0
        gates = p[t] * mask
        if renorm:
            gates = gates / gates.sum()
        ref[t] += sum(gates[e] * ys[e] for e in range(w.E))
    np.testing.assert_allclose(f["out"], ref, rtol=1e-11, atol=1e-12)


def test_single_expert_is_plain_ffn():
    """E = 1, k = 1: p = 1, so the layer is x + FFN(x)."""
    rng = np.random.default_rng(6)
    T, d, F = 7, 5, 4
    x = rng.standard_normal((T, d))
    w1 = rng.standard_normal((1, F, d))
    w2 = rng.standard_normal((1, d, F))
    f = O.forward(x, rng.standard_normal((1, d)), None, (w1, w2), k=1, act="relu", cf=None)
    np.testing.assert_allclose(f["out"], x + _ffn_loops(x, w1[0], w2[0], "relu"), rtol=1e-12, atol=1e-13)
    assert f["aux"] == pytest.approx(0.01)   # N = 1: f = P = 1


def test_dropped_tokens_return_x_bitwise():
    w = syn.WORKLOADS["tiny-top1-f32"].with_(T=96)
    inp = syn.make_inputs(w)
    for C in (0, 3):
        cf = (C * w.E, w.T)      # gives capacity floor(T*cf/E) = C
        f = O.forward(inp["x"], inp["w_r"], None, (inp["w1"], inp["w2"]), k=1, act="relu", cf=cf)
        assert f["C"] == C
        dropped = np.all(f["slot"] < 0, axis=1)
        assert dropped.sum() >= (w.T - w.E * C)
        assert np.array_equal(f["out"][dropped], inp["x"][dropped].astype(np.float64))


# ------------------------------------------------------------------ backward
def _relu_pattern(pp, base, w):
    """Signs of every kept row's ReLU pre-activations (empty for SwiGLU)."""
    if w.act != "relu":
        return ()
    out = []
    for e in range(w.E):
        tt = np.nonzero(((base["idx"] == e) & (base["slot"] >= 0)).any(axis=1))[0]
        out.append((pp["x"][tt] @ pp["w1"][e].T) > 0)
    return out


def _fd_check(w, n_coords=60, eps=1e-4, seed=0, add_residual=True, score="softmax", sel_bias=None,
              reroute=False):
    """Central differences of L = <dY, out> + aux against the oracle's backward.

    eps = 1e-4: at 1e-6 the fp64 rounding of L divided by 2 eps already
    exceeds the 1e-6 relative bound on single coordinates. Samples where +-eps
    changes a routing decision or crosses a ReLU kink are skipped and counted.
    """
    inp = syn.make_inputs(w, dy=True)
    kw = dict(k=w.k, act=w.act, cf=w.cf, count_assignments=w.count_assignments,
              renormalize=w.renormalize, alpha=w.alpha, add_residual=add_residual, score=score,
              sel_bias=sel_bias, reroute=reroute)
    x = inp["x"].astype(np.float64)
    w_r = inp["w_r"].astype(np.float64)
    w1 = inp["w1"].astype(np.float64)
    w2 = inp["w2"].astype(np.float64)
    bias = inp["bias"]
    dy = inp["dy"].astype(np.float64)
    g = O.backward(x, w_r, bias, (w1, w2), dy, **kw)
    grads = {"x": g["dx"], "w_r": g["dw_r"],
             "w1": np.stack([g["dw1"][e] for e in range(w.E)]),
             "w2": np.stack([g["dw2"][e] for e in range(w.E)])}
    base = O.forward(x, w_r, bias, (w1, w2), **kw)
    params = {"x": x, "w_r": w_r, "w1": w1, "w2": w2}
    pattern0 = _relu_pattern(params, base, w)

    def L(pp):
        f = O.forward(pp["x"], pp["w_r"], bias, (pp["w1"], pp["w2"]), **kw)
        same = np.array_equal(f["idx"], base["idx"]) and np.array_equal(f["slot"], base["slot"])
        same = same and all(np.array_equal(a, b) for a, b in zip(_relu_pattern(pp, base, w), pattern0))
        return float(np.sum(dy * f["out"])) + f["aux"], same

    rng = np.random.default_rng(seed)
    checked = skipped = 0
    for name, arr in params.items():
        dirs = [rng.standard_normal(arr.shape)]                       # one random direction
        for _ in range(n_coords):                                      # and single coordinates
            v = np.zeros(arr.shape)
            v[tuple(rng.integers(0, s) for s in arr.shape)] = 1.0
            dirs.append(v)
        for v in dirs:
            plus = dict(params); plus[name] = arr + eps * v
            minus = dict(params); minus[name] = arr - eps * v
            lp, sp = L(plus)
            lm, sm = L(minus)
            if not (sp and sm):
                skipped += 1
                continue
            fd = (lp - lm) / (2 * eps)
            an = float(np.sum(grads[name] * v))
            scale = max(1.0, abs(an)) if np.count_nonzero(v) > 1 else max(1e-3, abs(an))
            assert abs(fd - an) <= 1e-6 * scale, f"{name}: fd {fd!r} vs analytic {an!r}"
            checked += 1
    return checked, skipped


def test_gradients_finite_differences_tiny():
    w = syn.WORKLOADS["tiny-top1-f32"].with_(T=128)
    checked, skipped = _fd_check(w)
    assert checked >= 200 and skipped <= checked // 10


def test_gradients_finite_differences_swiglu_renorm_capacity():
    w = syn.Workload("fd-swiglu", T=48, d=12, E=6, k=3, F=10, act="swiglu", dtype="f32", cf=(3, 4),
                     renormalize=True, router_std=0.4, zipf_s=1.2, backward=True)
    checked, skipped = _fd_check(w, n_coords=40)
    assert checked >= 150 and skipped <= checked // 10


def test_gradient_of_aux_term_alone():
    """With dY = 0 only eq. (4) contributes: d aux / d h = p * (c - <p, c>), c_e = alpha E f_e / T."""
    rng = np.random.default_rng(8)
    T, E, d = 20, 5, 3
    x, w_r = rng.standard_normal((T, d)), rng.standard_normal((E, d))
    w1, w2 = rng.standard_normal((E, 4, d)), rng.standard_normal((E, d, 4))
    g = O.backward(x, w_r, None, (w1, w2), np.zeros((T, d)), k=1, act="relu", cf=None, alpha=0.5)
    r = O.route(x, w_r, None, 1, False, 0.5)
    c = 0.5 * E * r["f"] / T
    dh = r["p"] * (c[None, :] - (r["p"] * c[None, :]).sum(axis=1, keepdims=True))
    np.testing.assert_allclose(g["dh"], dh, rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(g["dw_r"], dh.T @ x, rtol=1e-12, atol=1e-16)


@pytest.mark.parametrize("wl", [
    syn.Workload("sampled-relu", T=96, d=16, E=6, k=2, F=12, act="relu", dtype="f32", cf=(3, 4), backward=True),
    syn.Workload("sampled-swiglu", T=64, d=12, E=5, k=3, F=10, act="swiglu", dtype="f32", cf=None,
                 renormalize=True, router_std=0.4, zipf_s=1.2, backward=True),
])
def test_sampled_backward_matches_full_backward(wl):
    """The token-by-token / expert-by-expert gradients equal the full backward
    (itself pinned by finite differences above) on the rows they cover."""
    inp = syn.make_inputs(wl, dy=True)
    kw = dict(k=wl.k, act=wl.act, cf=wl.cf, count_assignments=wl.count_assignments, renormalize=wl.renormalize,
              alpha=wl.alpha)
    experts = (inp["w1"], inp["w2"])
    full = O.backward(inp["x"], inp["w_r"], inp["bias"], experts, inp["dy"], **kw)
    toks = [0, 7, wl.T - 1, wl.T // 2]
    exps = list(range(wl.E))
    smp = O.backward_sampled(inp["x"], inp["w_r"], inp["bias"], experts, inp["dy"], tokens=toks,
                             experts_sampled=exps, **kw)
    for t in toks:
        np.testing.assert_allclose(smp["dx"][t], full["dx"][t], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(smp["dg"][t], full["dg"][t], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(smp["dh"][t], full["dh"][t], rtol=1e-11, atol=1e-15)
    for e in exps:
        np.testing.assert_allclose(smp["dw1"][e], full["dw1"][e], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(smp["dw2"][e], full["dw2"][e], rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ sampled forward
@pytest.mark.parametrize("wl", [
    syn.Workload("fwd-sampled-drops", T=120, d=16, E=6, k=2, F=12, act="relu", dtype="f32", cf=(1, 2),
                 zipf_s=1.2, router_std=0.4),
    syn.Workload("fwd-sampled-renorm", T=90, d=12, E=7, k=3, F=10, act="swiglu", dtype="f32", cf=(3, 4),
                 renormalize=True, router_std=0.4),
    syn.Workload("fwd-sampled-top1", T=64, d=8, E=4, k=1, F=6, act="relu", dtype="f32", cf=(1, 1)),
])
def test_sampled_forward_matches_full_forward(wl):
    """forward(tokens=S) is the full forward restricted to S: its out rows equal
    forward()["out"][S] (the experts' GEMMs run on a subset of rows, so equal
    up to the BLAS's summation order), and routing, slots and statistics are
    the whole batch's. The cases drop tokens (capacity below the load,
    Zipf-skewed logits), take k > 1 and renormalise, and the sample holds
    tokens in any order, repeats none, and includes fully dropped tokens."""
    inp = syn.make_inputs(wl)
    kw = dict(k=wl.k, act=wl.act, cf=wl.cf, count_assignments=wl.count_assignments, renormalize=wl.renormalize,
              alpha=wl.alpha)
    experts = (inp["w1"], inp["w2"])
    full = O.forward(inp["x"], inp["w_r"], inp["bias"], experts, **kw)
    dropped = np.nonzero(np.all(full["slot"] < 0, axis=1))[0]
    assert (full["slot"] < 0).any()
    rng = np.random.default_rng(wl.T)
    S = [int(t) for t in dropped[:2]] + [int(t) for t in rng.choice(wl.T, wl.T // 3, replace=False)]
    S = list(dict.fromkeys(S))                                 # no repeats, arbitrary order
    assert any(t in S for t in dropped)
    part = O.forward(inp["x"], inp["w_r"], inp["bias"], experts, tokens=S, **kw)
    np.testing.assert_array_equal(part["tokens"], S)
    np.testing.assert_allclose(part["out"], full["out"][S], rtol=1e-13, atol=1e-15)
    for t in dropped:
        if t in S:
            assert np.array_equal(part["out"][S.index(int(t))], inp["x"][t].astype(np.float64))
    for key in ("idx", "slot", "kept", "offsets", "row_token", "load"):
        np.testing.assert_array_equal(part[key], full[key])
    np.testing.assert_allclose(part["gate"], full["gate"], rtol=0, atol=0)
    assert part["aux"] == full["aux"]


# ------------------------------------------------------------------ without the residual
def test_without_residual_single_expert_is_plain_ffn():
    """E = 1, k = 1, add_residual off: p = 1, so the layer is FFN(x) alone (textbook loops)."""
    rng = np.random.default_rng(16)
    T, d, F = 6, 5, 4
    x = rng.standard_normal((T, d))
    w1 = rng.standard_normal((1, 2 * F, d))
    w2 = rng.standard_normal((1, d, F))
    f = O.forward(x, rng.standard_normal((1, d)), None, (w1, w2), k=1, act="swiglu", cf=None, add_residual=False)
    np.testing.assert_allclose(f["out"], _ffn_loops(x, w1[0], w2[0], "swiglu"), rtol=1e-12, atol=1e-13)


def test_without_residual_dense_masked_and_dropped_tokens_are_zero():
    """No residual: out = sum over kept top-k of g_i E_i(x) from every expert evaluated densely (brute-force
    top-k mask, token-order capacity from the brute-force slots); fully dropped tokens give zeros."""
    w = syn.Workload("pin-nores", T=30, d=8, E=5, k=2, F=6, act="relu", dtype="f32", cf=(1, 2), router_std=0.5)
    inp = syn.make_inputs(w)
    f = O.forward(inp["x"], inp["w_r"], None, (inp["w1"], inp["w2"]), k=2, act="relu", cf=(1, 2),
                  add_residual=False)
    x = inp["x"].astype(np.float64)
    h = x @ inp["w_r"].astype(np.float64).T
    p = scipy.special.softmax(h, axis=1)
    top = _brute_topk(h, 2)
    slot = _brute_slots(top, w.E, O.capacity(w.T, w.E, 2, (1, 2)))
    ref = np.zeros_like(x)
    for t in range(w.T):
        for j in range(2):
            if slot[t, j] >= 0:
                e = top[t, j]
                y = _ffn_loops(x[t:t + 1], inp["w1"][e].astype(np.float64), inp["w2"][e].astype(np.float64), "relu")
                ref[t] += p[t, e] * y[0]
    assert (slot < 0).all(axis=1).any()
    np.testing.assert_allclose(f["out"], ref, rtol=1e-11, atol=1e-12)
    assert np.all(f["out"][(slot < 0).all(axis=1)] == 0.0)


def test_gradients_finite_differences_without_residual():
    w = syn.Workload("fd-nores", T=40, d=10, E=5, k=2, F=8, act="swiglu", dtype="f32", cf=(3, 4),
                     renormalize=True, router_std=0.4, backward=True)
    checked, skipped = _fd_check(w, n_coords=30, add_residual=False)
    assert checked >= 100 and skipped <= checked // 10


# ------------------------------------------------------------------ router variants in the layer
@pytest.mark.parametrize("score,biased", [("sigmoid", False), ("sigmoid", True), ("sqrt_softplus", False),
                                          ("sqrt_softplus", True), ("softmax", True)])
def test_gradients_finite_differences_router_variants(score, biased):
    """The layer's gradients with an elementwise score (its own derivative in place of the softmax Jacobian)
    and with a selection-only correction bias (constant choice, gates without the bias) against central
    differences of L = <dY, out> + aux."""
    w = syn.Workload(f"fd-{score}-{biased}", T=40, d=10, E=6, k=2, F=8, act="swiglu", dtype="f32", cf=(3, 4),
                     renormalize=biased, router_std=0.4, backward=True)
    b = np.random.default_rng(3).standard_normal(w.E) * 0.05 if biased else None
    checked, skipped = _fd_check(w, n_coords=25, score=score, sel_bias=b)
    assert checked >= 80 and skipped <= checked // 10


def test_route_with_variants_follows_the_variant_oracle():
    """moe_oracle.route with a score function and a correction bias chooses, gates and counts as
    router_variants.route_variant does on the same logits; the statistics sum the scores."""
    rng = np.random.default_rng(9)
    x, w_r = rng.standard_normal((50, 12)), rng.standard_normal((7, 12)) / 3.0
    b = rng.standard_normal(7) * 0.2
    from oracle import router_variants as RV
    for score in RV.SCORES:
        for sel in (None, b):
            r = O.route(x, w_r, None, 3, True, 0.01, score, sel)
            v = RV.route_variant(O.router_logits(x, w_r), 3, score, sel_bias=sel, renormalize=True)
            assert np.array_equal(r["idx"], v["idx"]) and np.array_equal(r["load"], v["load"])
            np.testing.assert_allclose(r["gate"], v["gate"], rtol=1e-15)
            np.testing.assert_allclose(r["importance"], v["s"].sum(axis=0), rtol=1e-13)


# ------------------------------------------------------------------ No-Token-Left-Behind
def _brute_reroute(first, second, E, C):
    """The two rounds spelled out with per-expert queues: round 1 keeps each expert's first C first-choice
    tokens (token order); round 2 walks the round-1 dropouts in token order and admits each to its second
    expert while that expert holds fewer than C."""
    T = len(first)
    slot = -np.ones((T, 2), dtype=np.int64)
    held = {e: [] for e in range(E)}
    for t in range(T):
        if len(held[first[t]]) < C:
            slot[t, 0] = len(held[first[t]])
            held[first[t]].append(t)
    for t in range(T):
        if slot[t, 0] < 0 and len(held[second[t]]) < C:
            slot[t, 1] = len(held[second[t]])
            held[second[t]].append(t)
    return slot, np.array([len(held[e]) for e in range(E)])


@pytest.mark.parametrize("C", [0, 2, 5, 40])
def test_reroute_slots_brute_force_and_invariants(C):
    rng = np.random.default_rng(30 + C)
    T, E = 60, 5
    idx2 = np.stack([rng.permutation(E)[:2] for _ in range(T)])
    idx2[:25, 0] = 1                                    # overload expert 1 so that round 2 has work
    s = O.assign_slots_reroute(idx2, E, C)
    slot, kept = _brute_reroute(idx2[:, 0], idx2[:, 1], E, C)
    np.testing.assert_array_equal(s["slot"], slot)
    np.testing.assert_array_equal(s["kept"], kept)
    assert np.all(s["kept"] <= C) and np.all(((s["slot"] >= 0).sum(axis=1)) <= 1)
    plain = O.assign_slots(idx2[:, :1], E, C)
    np.testing.assert_array_equal(s["slot"][:, 0], plain["slot"][:, 0])   # round 1 is the plain rule
    assert (s["slot"] >= 0).any(axis=1).sum() >= (plain["slot"] >= 0).sum()
    for t in range(T):
        for j in range(2):
            if s["slot"][t, j] >= 0:
                row = s["offsets"][idx2[t, j]] + s["slot"][t, j]
                assert s["row_token"][row] == t


def test_reroute_layer_gates_and_statistics():
    """The second-choice expert's probability is the gate of a rerouted token; load and f count first choices;
    a token is dropped for good only when both of its experts are full."""
    w = syn.Workload("reroute-pin", T=80, d=8, E=6, k=1, F=6, act="relu", dtype="f32", cf=(1, 2), router_std=0.6,
                     zipf_s=1.5)
    inp = syn.make_inputs(w)
    f = O.forward(inp["x"], inp["w_r"], inp["bias"], (inp["w1"], inp["w2"]), k=1, act="relu", cf=(1, 2),
                  reroute=True)
    base = O.forward(inp["x"], inp["w_r"], inp["bias"], (inp["w1"], inp["w2"]), k=1, act="relu", cf=(1, 2))
    assert f["idx"].shape == (w.T, 2) and np.array_equal(f["idx"][:, 0], base["idx"][:, 0])
    np.testing.assert_array_equal(f["load"], base["load"])
    assert f["aux"] == base["aux"]
    np.testing.assert_array_equal(f["gate"], np.take_along_axis(f["p"], f["idx"], axis=1))
    rerouted = f["slot"][:, 1] >= 0
    assert rerouted.any()
    x = inp["x"].astype(np.float64)
    for t in np.nonzero(rerouted)[0][:5]:
        e = f["idx"][t, 1]
        y = O.expert_ffn(x[t:t + 1], inp["w1"][e].astype(np.float64), inp["w2"][e].astype(np.float64), "relu")["y"]
        np.testing.assert_allclose(f["out"][t], x[t] + f["p"][t, e] * y[0], rtol=1e-12)
    C = f["C"]
    for t in np.nonzero((f["slot"] < 0).all(axis=1))[0]:
        assert f["kept"][f["idx"][t, 0]] == C and f["kept"][f["idx"][t, 1]] == C


def test_gradients_finite_differences_reroute():
    w = syn.Workload("fd-reroute", T=48, d=10, E=5, k=1, F=8, act="swiglu", dtype="f32", cf=(1, 2), router_std=0.5,
                     zipf_s=1.2, backward=True)
    checked, skipped = _fd_check(w, n_coords=30, reroute=True)
    assert checked >= 100 and skipped <= checked // 10


# ------------------------------------------------------------------ expert-choice routing
def test_expert_choice_brute_force_choice_and_dense_sum():
    """Each expert's chosen tokens by brute-force rank counting over its score column (ties to the lower
    token: a tie planted on purpose), and the layer equal to x plus a dense evaluation of every expert
    masked to the pairs chosen."""
    w = syn.Workload("ec-pin", T=20, d=6, E=4, k=1, F=5, act="relu", dtype="f32", cf=None, router_std=0.6)
    inp = syn.make_inputs(w)
    x = inp["x"].astype(np.float64)
    w_r = inp["w_r"].astype(np.float64)
    w_r[3] = w_r[2]                                   # experts 2 and 3 score every token alike
    C = 7
    f = O.forward_expert_choice(x, w_r, None, (inp["w1"], inp["w2"]), C=C, act="relu")
    p = scipy.special.softmax(x @ w_r.T, axis=1)
    for e in range(w.E):
        beats = lambda a, b: p[a, e] > p[b, e] or (p[a, e] == p[b, e] and a < b)
        top = sorted(t for t in range(w.T) if sum(beats(u, t) for u in range(w.T) if u != t) < C)
        assert f["chosen"][e].tolist() == top
    assert f["chosen"][2].tolist() == f["chosen"][3].tolist()
    ref = x.copy()
    for t in range(w.T):
        for e in range(w.E):
            if t in f["chosen"][e]:
                y = _ffn_loops(x[t:t + 1], inp["w1"][e].astype(np.float64), inp["w2"][e].astype(np.float64), "relu")
                ref[t] += p[t, e] * y[0]
    np.testing.assert_allclose(f["out"], ref, rtol=1e-12, atol=1e-13)
    assert np.all(f["load"] == C) and f["offsets"][-1] == w.E * C


def test_expert_choice_capacity_above_tokens_takes_every_token():
    """C >= T: every expert takes every token, so out = x + sum over all experts of p E(x) (the dense mixture)."""
    rng = np.random.default_rng(17)
    T, d, E, F = 6, 4, 3, 5
    x, w_r = rng.standard_normal((T, d)), rng.standard_normal((E, d))
    w1, w2 = rng.standard_normal((E, F, d)), rng.standard_normal((E, d, F))
    f = O.forward_expert_choice(x, w_r, None, (w1, w2), C=10, act="relu")
    p = scipy.special.softmax(x @ w_r.T, axis=1)
    ref = x + sum(p[:, e:e + 1] * _ffn_loops(x, w1[e], w2[e], "relu") for e in range(E))
    np.testing.assert_allclose(f["out"], ref, rtol=1e-12, atol=1e-13)


def test_expert_choice_gradients_finite_differences():
    w = syn.Workload("fd-ec", T=30, d=8, E=5, k=1, F=6, act="swiglu", dtype="f32", cf=None, router_std=0.5,
                     backward=True)
    inp = syn.make_inputs(w, dy=True)
    x, w_r = inp["x"].astype(np.float64), inp["w_r"].astype(np.float64)
    w1, w2, dy = inp["w1"].astype(np.float64), inp["w2"].astype(np.float64), inp["dy"].astype(np.float64)
    C = 9
    g = O.backward_expert_choice(x, w_r, None, (w1, w2), dy, C=C, act="swiglu")
    base = O.route_expert_choice(x, w_r, None, C)["chosen"]

    def L(xx, wr, a1, a2):
        f = O.forward_expert_choice(xx, wr, None, (a1, a2), C=C, act="swiglu")
        return float(np.sum(dy * f["out"])), np.array_equal(f["chosen"], base)

    grads = {"x": g["dx"], "w_r": g["dw_r"], "w1": np.stack([g["dw1"][e] for e in range(w.E)]),
             "w2": np.stack([g["dw2"][e] for e in range(w.E)])}
    params = {"x": x, "w_r": w_r, "w1": w1, "w2": w2}
    rng = np.random.default_rng(2)
    eps, checked, skipped = 1e-4, 0, 0
    for name, arr in params.items():
        for _ in range(25):
            v = np.zeros(arr.shape)
            v[tuple(rng.integers(0, s) for s in arr.shape)] = 1.0
            pp, mm = dict(params), dict(params)
            pp[name], mm[name] = arr + eps * v, arr - eps * v
            lp, sp = L(pp["x"], pp["w_r"], pp["w1"], pp["w2"])
            lm, sm = L(mm["x"], mm["w_r"], mm["w1"], mm["w2"])
            if not (sp and sm):
                skipped += 1
                continue
            an = float(np.sum(grads[name] * v))
            assert abs((lp - lm) / (2 * eps) - an) <= 1e-6 * max(1e-3, abs(an)), name
            checked += 1
    assert checked >= 80 and skipped <= checked // 10
