"""The seeded input generator: reproducible, bf16-exact, margin-conditioned."""
import numpy as np
import pytest

import moe_synth as syn


def test_bf16_rounding_ties_to_even_and_exactness():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5e-3], np.float32)
    r = syn.round_bf16(vals)
    assert r[1] == 1.0                        # tie -> even mantissa
    assert r[2] == np.float32(1.0 + 4 * 2 ** -8)
    assert r[3] == 1.0
    assert np.array_equal(syn.round_bf16(r), r)
    assert np.array_equal(syn.from_bf16_bits(syn.bf16_bits(r)), r)


@pytest.mark.parametrize("name", ["tiny-top1-f32", "gshard-top2-zipf"])
def test_margin_conditioning_holds(name):
    w = syn.WORKLOADS[name]
    if w.T * w.d > 2_000_000:
        w = w.with_(T=2048)
    w_r, b = syn.router_weight(w), syn.logit_bias(w)
    x = syn.tokens(w, w_r, b)
    h = x.astype(np.float64) @ w_r.astype(np.float64).T + (0 if b is None else b.astype(np.float64))
    top = -np.sort(-h, axis=1)[:, : w.k + 1]
    assert (top[:, :-1] - top[:, 1:]).min() >= syn.MARGIN
    if w.dtype == "bf16":
        assert np.array_equal(syn.round_bf16(x), x)


def test_per_expert_regeneration_is_reproducible():
    w = syn.WORKLOADS["tiny-top1-f32"]
    w1, w2 = syn.all_expert_weights(w)
    a, b = syn.expert_weights(w, 5)
    assert np.array_equal(w1[5], a) and np.array_equal(w2[5], b)
    assert not np.array_equal(w1[4], w1[5])


def test_init_scale():
    w = syn.WORKLOADS["tiny-top1-f32"].with_(E=64)
    w1, w2 = syn.all_expert_weights(w)
    assert abs(w1.std() - 0.1 / np.sqrt(w.d)) < 0.02 * 0.1 / np.sqrt(w.d)
    assert abs(w2.std() - 0.1 / np.sqrt(w.F)) < 0.02 * 0.1 / np.sqrt(w.F)


def test_zipf_bias_is_a_log_distribution():
    w = syn.WORKLOADS["gshard-top2-zipf"]
    b = syn.logit_bias(w).astype(np.float64)
    assert abs(np.exp(b).sum() - 1.0) < 1e-6
    assert np.all(np.diff(b) < 0)
    assert abs((b[0] - b[1]) - 1.2 * np.log(2.0)) < 1e-5


def test_threaded_bit_draws_equal_the_per_expert_draws():
    w = syn.WORKLOADS["large-top8-swiglu"].with_(name="bits-small", E=6, d=64, F=32)
    b1, b2 = syn.expert_weight_bits(w, threads=3)
    assert b1.dtype == np.uint16 and b1.shape == (6, 64, 64) and b2.shape == (6, 64, 32)
    for e in range(w.E):
        a, b = syn.expert_weights(w, e)
        assert np.array_equal(syn.from_bf16_bits(b1[e]), a) and np.array_equal(syn.from_bf16_bits(b2[e]), b)
