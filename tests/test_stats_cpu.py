"""The logging figures the binding derives from the router's and the
dispatch's per-expert statistics, on hand-worked batches."""
import pytest

import sparse_mixture_experts_49_b300 as moe


def test_uniform_batch():
    # 8 tokens, top-1, 4 experts with 2 tokens each and equal mean probability
    s = moe.balance_stats(importance=[2.0] * 4, load=[2] * 4, kept=[2] * 4, T=8, k=1, alpha=0.01)
    assert s["drop_rate"] == 0.0
    assert s["max_over_mean_load"] == 1.0
    assert s["cv2_load"] == 0.0 and s["cv2_importance"] == 0.0
    assert s["aux"] == pytest.approx(0.01)            # uniform f = P = 1/E gives alpha (eq. (4))


def test_skewed_batch_with_drops():
    # 4 tokens, top-1, 2 experts: loads 3 / 1, capacity 2 keeps 2 / 1
    s = moe.balance_stats(importance=[2.5, 1.5], load=[3, 1], kept=[2, 1], T=4, k=1, alpha=0.01)
    assert s["drop_rate"] == pytest.approx(0.25)      # 1 of 4 assignments over capacity
    assert s["max_over_mean_load"] == pytest.approx(1.5)
    assert s["cv2_load"] == pytest.approx(1.0 / 4.0)  # variance 1, mean 2
    assert s["cv2_importance"] == pytest.approx(0.25 / 4.0)
    # alpha E sum f P = 0.01 * 2 * (3/4 * 2.5/4 + 1/4 * 1.5/4) = 0.01 * 1.125
    assert s["aux"] == pytest.approx(0.01125)


def test_top_k_normalisation():
    # top-2 over 2 experts: every token picks both, f = 1/2 each
    s = moe.balance_stats(importance=[3.0, 1.0], load=[4, 4], kept=[4, 4], T=4, k=2, alpha=0.01)
    assert s["drop_rate"] == 0.0
    # 0.01 * 2 * (1/2 * 3/4 + 1/2 * 1/4) = 0.01
    assert s["aux"] == pytest.approx(0.01)
