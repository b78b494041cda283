"""Pins of the router-variant oracle: closed forms of the score functions, a
hand-worked selection where the correction bias changes the choice but not
the gate, brute-force ranking, the bias update's sign rule, and the reduction
to the pinned softmax router."""
import itertools

import numpy as np
import pytest

from oracle import moe_oracle as O
from oracle import router_variants as RV


def test_score_closed_forms():
    z = np.zeros((1, 3))
    assert np.allclose(RV.scores(z, "sigmoid"), 0.5)
    assert np.allclose(RV.scores(z, "sqrt_softplus"), np.sqrt(np.log(2.0)))
    assert np.allclose(RV.scores(z, "softmax"), 1.0 / 3.0)
    h = np.array([[-3.0, -0.5, 0.25, 2.0, 40.0]])
    sig = RV.scores(h, "sigmoid")
    assert np.allclose(sig + RV.scores(-h, "sigmoid"), 1.0)                  # sigma(h) + sigma(-h) = 1
    sp = RV.scores(h, "sqrt_softplus") ** 2
    assert np.allclose(sp - RV.scores(-h, "sqrt_softplus") ** 2, h)           # softplus(h) - softplus(-h) = h
    assert np.isclose(sp[0, 4], 40.0)                                         # no overflow for large h


def test_bias_changes_the_choice_not_the_gate():
    # one token, four experts; sigmoid scores 0.7311 (h = 1.0) and 0.7109 (h = 0.9)
    h = np.array([[1.0, 0.9, 0.0, 0.0]])
    r0 = RV.route_variant(h, 1, "sigmoid")
    assert r0["idx"].tolist() == [[0]]
    r1 = RV.route_variant(h, 1, "sigmoid", sel_bias=np.array([0.0, 0.1, 0.0, 0.0]))
    assert r1["idx"].tolist() == [[1]]                                         # 0.7109 + 0.1 > 0.7311
    assert r1["gate"][0, 0] == pytest.approx(1.0 / (1.0 + np.exp(-0.9)))       # the bias is not in the gate


def test_selection_by_brute_force_ranking():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((16, 6))
    h[3, 2] = h[3, 4]                                                          # a tie: the lower index first
    b = rng.standard_normal(6) * 0.3
    for kind in RV.SCORES:
        s = RV.scores(h, kind)
        idx = RV.select(s, 3, b)
        for t in range(h.shape[0]):
            key = s[t] + b
            # expert e is chosen iff fewer than k others beat it (value first, then lower index)
            beats = lambda a, c: key[a] > key[c] or (key[a] == key[c] and a < c)
            chosen = sorted(e for e in range(6) if sum(beats(o, e) for o in range(6) if o != e) < 3)
            assert sorted(idx[t].tolist()) == chosen
            assert all(beats(idx[t][i], idx[t][i + 1]) for i in range(2))     # in order


def test_monotone_scores_without_bias_choose_the_top_logits():
    rng = np.random.default_rng(6)
    h = rng.standard_normal((32, 8))
    top = O.top_k(h, 2)
    for kind in RV.SCORES:
        assert np.array_equal(RV.route_variant(h, 2, kind)["idx"], top)


def test_renormalised_gates_sum_to_one():
    rng = np.random.default_rng(7)
    h = rng.standard_normal((20, 8))
    for kind in RV.SCORES:
        g = RV.route_variant(h, 3, kind, sel_bias=rng.standard_normal(8), renormalize=True)["gate"]
        assert np.allclose(g.sum(axis=1), 1.0)


def test_softmax_without_bias_is_the_pinned_router():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((24, 16))
    w_r = rng.standard_normal((8, 16)) / 4.0
    for renorm in (False, True):
        base = O.route(x, w_r, None, 2, renorm, 0.01)
        v = RV.route_variant(O.router_logits(x, w_r), 2, "softmax", renormalize=renorm)
        assert np.array_equal(v["idx"], base["idx"])
        assert np.allclose(v["gate"], base["gate"], rtol=0, atol=1e-15)
        assert np.array_equal(v["load"], base["load"])


def test_bias_update_sign_rule():
    b = np.array([0.5, 0.0, -0.25, 0.0])
    load = np.array([6, 2, 0, 4])                                              # mean 3
    assert RV.update_bias(b, load, 0.01).tolist() == pytest.approx([0.49, 0.01, -0.24, -0.01])
    assert RV.update_bias(b, np.array([3, 3, 3, 3]), 0.01).tolist() == b.tolist()   # balanced: no change
