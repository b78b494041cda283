"""CUDA path vs the CPU oracle, through the C ABI, on seeded inputs.

Routing (top-k indices, load, slots, kept counts, group offsets, row owners)
must match bit for bit; the fp32 router's values within 1e-5 x max|ref| (fp32
layer) or 1e-4 x max|ref| (bf16 layers, tensor-core fp32 accumulation); the
layer's floating outputs and gradients within 2e-2 x max|ref| for bf16
experts (fp32 accumulation) and 1e-5 x max|ref| for the fp32 layer.
"""
import numpy as np
import pytest

import moe_synth as syn
from oracle import moe_oracle as O
from moe_cases import (SMALL, TOL_BF16, TOL_F32, TOL_ROUTER_BF16, assert_close, backward_intermediates,
                       check_router_values, check_routing, config_for, expert_reference, np64, oracle_kw, run_gpu)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_mixture_experts_49_b300 as moe
    moe.lib()   # fails loudly if the library is not built


def _ref_all(w, inp, backward, sel_bias=None):
    kw = dict(oracle_kw(w), sel_bias=sel_bias)
    experts = (inp["w1"], inp["w2"])
    f = O.forward(inp["x"], inp["w_r"], inp["bias"], experts, **kw)
    b = O.backward(inp["x"], inp["w_r"], inp["bias"], experts, inp["dy"], **kw) if backward else None
    return f, b


def _check_full(w, res, inp, f, b):
    tol = TOL_F32 if w.dtype == "f32" else TOL_BF16
    check_routing(res, f, w)
    check_router_values(res, f, w.dtype)
    assert res["device_error"] == 0
    assert np.array_equal(res["x_perm"], inp["x"].astype(np.float64)[f["row_token"]])
    h_ref, y_ref = expert_reference(w, inp, f)
    assert_close(res["h"], h_ref, tol, "h")
    assert_close(res["y_perm"], y_ref, tol, "y_perm")
    assert_close(res["out"], f["out"], tol, "out")
    dropped = np.all(f["slot"] < 0, axis=1)
    passthrough = inp["x"].astype(np.float64)[dropped] if w.add_residual else np.zeros((int(dropped.sum()), w.d))
    assert np.array_equal(res["out"][dropped], passthrough), "dropped tokens must return x (zeros without residual)"
    if b is not None:
        assert_close(res["dg"], b["dg"], tol, "dg")
        assert_close(res["dh"], b["dh"], tol, "dh")
        assert_close(res["dx"], b["dx"], tol, "dx")
        assert_close(res["dw_r"], b["dw_r"], tol, "dw_r")
        assert_close(res["dw1"], np.stack([b["dw1"][e] for e in range(w.E)]), tol, "dw1")
        assert_close(res["dw2"], np.stack([b["dw2"][e] for e in range(w.E)]), tol, "dw2")


def test_tiny_f32_forward_backward():
    w = syn.WORKLOADS["tiny-top1-f32"]
    inp = syn.make_inputs(w)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    _check_full(w, res, inp, f, b)


@pytest.mark.parametrize("name", list(SMALL))
def test_bf16_small_layers(name):
    w = SMALL[name]
    inp = syn.make_inputs(w, dy=w.backward)
    res = run_gpu(w, inp, backward=w.backward)
    f, b = _ref_all(w, inp, w.backward)
    _check_full(w, res, inp, f, b)


@pytest.mark.parametrize("name", ["tiny-top1-f32", "switch-small", "dropless-small"])
def test_deterministic(name):
    w = syn.WORKLOADS.get(name) or SMALL[name]
    inp = syn.make_inputs(w, dy=True)
    r1 = run_gpu(w, inp, backward=True)
    r2 = run_gpu(w, inp, backward=True)
    for key in ("out", "probs", "importance", "aux", "dx", "dw_r", "dw1", "dw2"):
        assert np.array_equal(np.asarray(r1[key]), np.asarray(r2[key])), key


@pytest.mark.parametrize("E,k", [(256, 2), (20, 1), (64, 8)])
def test_router_expert_counts_and_many_tiles(E, k):
    """49 token tiles (a ragged last one) with the K range split over CTAs:
    256 experts, a padded narrow layer (20 experts in 32 columns), top-8."""
    w = syn.Workload(f"many-tiles-{E}-{k}", T=6200, d=320, E=E, k=k, F=128, act="relu", dtype="bf16",
                     cf=(5, 4), router_std=1 / np.sqrt(320))
    inp = syn.make_inputs(w, dy=False)
    res = run_gpu(w, inp)
    f, _ = _ref_all(w, inp, False)
    _check_full(w, res, inp, f, None)


@pytest.mark.parametrize("T,E,k,renorm,d", [(200, 256, 8, False, 256), (130, 130, 3, True, 256),
                                            (96, 64, 2, False, 256), (1000, 128, 1, False, 256),
                                            (4000, 48, 4, True, 256), (300, 256, 8, False, 640),
                                            (2000, 100, 2, True, 520), (20000, 32, 1, False, 136)])
def test_router_cluster_splits(T, E, k, renorm, d):
    """The fused tensor-core router with d split over 8, 4, 2 or 1 CTAs of a cluster (few or many 128-token
    tiles; a partial last tile; K steps that do not divide evenly over the CTAs, and a partial last K step;
    130 and 100 experts in padded column ranges): routing bit-exact, values against the oracle, and every
    gate equal to the probability the same kernel wrote for its expert, bit for bit (the gates are not
    renormalised)."""
    w = syn.Workload(f"router-split-{T}-{E}-{k}-{d}", T=T, d=d, E=E, k=k, F=128, act="relu", dtype="bf16",
                     cf=(5, 4), renormalize=renorm, router_std=1 / np.sqrt(d))
    inp = syn.make_inputs(w, dy=False)
    res = run_gpu(w, inp)
    f, _ = _ref_all(w, inp, False)
    check_routing(res, f, w)
    check_router_values(res, f, w.dtype)
    assert res["device_error"] == 0
    if not renorm:
        assert np.array_equal(res["gate"], np.take_along_axis(res["probs"], res["idx"], axis=1))
    assert np.all(np.abs(res["probs"].sum(axis=1) - 1.0) <= 1e-5)


@pytest.mark.parametrize("name", ["switch-small", "gshard-small", "dropless-small", "top1-many-tiles"])
def test_fused_forward_call(name):
    """moe_forward (router, dispatch, expert GEMMs with the top-1 combine in the
    second one's epilogue) against the oracle and the separate calls."""
    if name == "top1-many-tiles":
        w = syn.Workload(name, T=6200, d=320, E=40, k=1, F=192, act="relu", dtype="bf16", cf=(1, 1),
                         router_std=1 / np.sqrt(320))
    else:
        w = SMALL[name]
    inp = syn.make_inputs(w, dy=False)
    res = run_gpu(w, inp, fused=True)
    sep = run_gpu(w, inp)
    f, _ = _ref_all(w, inp, False)
    check_routing(res, f, w)
    check_router_values(res, f, w.dtype)
    assert res["device_error"] == 0
    h_ref, _ = expert_reference(w, inp, f)
    assert_close(res["h"], h_ref, TOL_BF16, "h")
    assert_close(res["out"], f["out"], TOL_BF16, "out")
    assert_close(res["out"], sep["out"], TOL_BF16, "out vs separate calls")
    dropped = np.all(f["slot"] < 0, axis=1)
    assert dropped.any() == (w.cf is not None and (f["slot"] < 0).any())
    assert np.array_equal(res["out"][dropped], inp["x"].astype(np.float64)[dropped]), "dropped tokens must return x"


# ------------------------------------------------------------------ edge cases
def test_capacity_zero_drops_everything():
    w = SMALL["switch-small"].with_(cf=(0, 1), backward=True)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    assert np.all(res["slot"] == -1) and np.all(res["kept"] == 0)
    assert np.array_equal(res["out"], inp["x"].astype(np.float64))
    f, b = _ref_all(w, inp, True)
    assert_close(res["dx"], b["dx"], TOL_BF16, "dx")
    assert np.all(res["dw1"] == 0) and np.all(res["dw2"] == 0)


def test_single_token():
    w = SMALL["large-small"].with_(T=1, cf=None)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    _check_full(w, res, inp, f, b)


def test_k_equals_E():
    w = syn.Workload("k-eq-e", T=300, d=128, E=4, k=4, F=128, act="swiglu", dtype="bf16", cf=None,
                     renormalize=True, backward=True)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    _check_full(w, res, inp, f, b)


def test_replayed_routing_all_on_one_expert():
    """Caller-supplied top-k (replay of a recorded routing): every token on expert 3."""
    w = SMALL["switch-small"].with_(cf=None)
    inp = syn.make_inputs(w)
    idx = np.full((w.T, 1), 3, np.int64)
    res = run_gpu(w, inp, topk_idx=idx)
    assert np.array_equal(res["kept"], np.eye(w.E, dtype=np.int64)[3] * w.T)
    assert np.array_equal(res["slot"][:, 0], np.arange(w.T))
    x = inp["x"].astype(np.float64)
    y = O.expert_ffn(x, inp["w1"][3].astype(np.float64), inp["w2"][3].astype(np.float64), "relu")["y"]
    assert_close(res["out"], x + res["gate"][:, :1] * y, TOL_BF16, "out")


def test_bad_and_repeated_expert_indices_are_reported_and_dropped():
    import sparse_mixture_experts_49_b300 as moe
    w = SMALL["gshard-small"].with_(T=256, cf=None)
    inp = syn.make_inputs(w)
    idx = np.stack([np.arange(w.T) % w.E, (np.arange(w.T) + 1) % w.E], axis=1)
    idx[5, 1] = w.E + 3          # out of range
    res = run_gpu(w, inp, topk_idx=idx)
    assert res["device_error"] == moe.MOE_DEVERR_BAD_EXPERT
    assert res["slot"][5, 1] == -1 and res["slot"][5, 0] >= 0
    idx[5, 1] = idx[5, 0]        # repeated expert
    res = run_gpu(w, inp, topk_idx=idx)
    assert res["device_error"] == moe.MOE_DEVERR_DUP_EXPERT
    assert res["slot"][5, 1] == -1 and res["slot"][5, 0] >= 0


def test_empty_experts_and_heavy_skew():
    """Zipf-biased routing with a small capacity: many drops, some experts empty."""
    w = SMALL["gshard-small"].with_(cf=(1, 2), zipf_s=2.5)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    assert (f["load"] == 0).any() and (f["slot"] < 0).mean() > 0.3
    _check_full(w, res, inp, f, b)


# ------------------------------------------------------------------ grouped-GEMM tile modes
# Layers whose expert groups span several 256-row CTA-pair tiles with ragged
# ends, and weight-gradient GEMMs whose M is a multiple of 256 (pair-*) or not
# (dropless-small: d 320, 2F 384, read past M through the tensor map's zero fill).
PAIR_CASES = {
    "pair-relu": syn.Workload("pair-relu", T=2048, d=512, E=4, k=2, F=256, act="relu", dtype="bf16", cf=None,
                              backward=True),
    "pair-swiglu": syn.Workload("pair-swiglu", T=1536, d=512, E=6, k=4, F=256, act="swiglu", dtype="bf16",
                                cf=(5, 4), renormalize=True, backward=True),
    "dropless-small": SMALL["dropless-small"],
    "gshard-small": SMALL["gshard-small"],
    # capacity 192 (the most rows the unit-resident weight-gradient kernel takes: three K steps), skewed so
    # that the first experts are full, later ones partial and the last ones likely empty
    "wgrad-edge": syn.Workload("wgrad-edge", T=3072, d=256, E=16, k=1, F=256, act="relu", dtype="bf16", cf=(1, 1),
                               zipf_s=1.5, router_std=1 / 16, backward=True),
    "large-small": SMALL["large-small"],
    # three m-tiles for dW2 (d = 384: the weight-gradient kernel's units cover two, the last one runs past M)
    # and partial 128-column n-tiles (F = 320)
    "wgrad-odd": syn.Workload("wgrad-odd", T=1024, d=384, E=16, k=2, F=320, act="relu", dtype="bf16", cf=(5, 4),
                              router_std=1 / np.sqrt(384), backward=True),
}


@pytest.mark.parametrize("mode", ["1", "0", "dynamic", "wgrad-gemm"])
@pytest.mark.parametrize("name", list(PAIR_CASES))
def test_gemm_tile_modes(name, mode, monkeypatch):
    """Every expert GEMM forced onto CTA-pair tiles (MOE_GEMM_PAIR=1), onto
    one CTA per tile in the fixed order (0), or one CTA per tile handed out by
    the workspace's tile counter (MOE_GEMM_SCHED=dynamic), forward and
    backward, against the oracle; twice in a row for the counter, which every
    launch must leave at zero. With one CTA per tile, layers whose capacity
    is at most 192 rows take their weight gradients from the unit-resident
    kernel; MOE_WGRAD=gemm (wgrad-gemm) sends them to the grouped GEMM."""
    if mode == "wgrad-gemm":
        monkeypatch.setenv("MOE_WGRAD", "gemm")
        mode = "0"
    if mode == "dynamic":
        monkeypatch.setenv("MOE_GEMM_PAIR", "0")
        monkeypatch.setenv("MOE_GEMM_SCHED", "dynamic")
        w = PAIR_CASES[name]
        inp = syn.make_inputs(w, dy=True)
        import sparse_mixture_experts_49_b300 as moe
        layer = moe.MoELayer(config_for(moe, w))
        f, b = _ref_all(w, inp, True)
        for _ in range(2):
            res = run_gpu(w, inp, backward=True, layer=layer)
            _check_full(w, res, inp, f, b)
        return
    monkeypatch.setenv("MOE_GEMM_PAIR", mode)
    w = PAIR_CASES[name]
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    _check_full(w, res, inp, f, b)


@pytest.mark.parametrize("name", ["gshard-small", "large-small", "wgrad-odd", "pair-swiglu"])
def test_gemm_tail_windows(name, monkeypatch):
    """The last partial wave of grouped-M tiles cut into 128- or 64-column windows (the default) against whole
    tiles (MOE_GEMM_TAIL=0): every output and gradient bit for bit the same (a window's MMAs accumulate each
    output element over the same K steps in the same order), and both against the oracle. At these sizes
    every tile is in the last wave, so each GEMM runs on windows: ReLU and SwiGLU-backward staged epilogues,
    the plain TMA-store epilogue with K-major and MN-major weights, and the row-by-row path of group ends."""
    w = PAIR_CASES[name]
    inp = syn.make_inputs(w, dy=True)
    monkeypatch.setenv("MOE_GEMM_PAIR", "0")
    runs = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("MOE_GEMM_TAIL", mode)
        runs[mode] = run_gpu(w, inp, backward=True)
    monkeypatch.delenv("MOE_GEMM_TAIL")
    for key in ("out", "h", "y_perm", "dx", "dw_r", "dw1", "dw2"):
        if runs["1"][key] is None:
            continue
        assert np.array_equal(np.asarray(runs["1"][key]), np.asarray(runs["0"][key])), key
    f, b = _ref_all(w, inp, True)
    _check_full(w, runs["1"], inp, f, b)


@pytest.mark.parametrize("name", ["gshard-small", "large-small", "wgrad-odd", "pair-swiglu", "dropless-small"])
def test_gemm_short_tiles(name, monkeypatch):
    """m-tiles that hold at most 64 of their group's rows on M = 64 MMAs (the default; rows 16 q + i in TMEM lane
    32 q + i, stored row by row) against full 128-row tiles (MOE_GEMM_M64=0): every output and gradient bit for
    bit the same, and both against the oracle (forward and backward, every grouped-M epilogue)."""
    w = PAIR_CASES[name]
    inp = syn.make_inputs(w, dy=True)
    monkeypatch.setenv("MOE_GEMM_PAIR", "0")
    runs = {}
    for mode in ("1", "0"):
        monkeypatch.setenv("MOE_GEMM_M64", mode)
        runs[mode] = run_gpu(w, inp, backward=True)
    monkeypatch.delenv("MOE_GEMM_M64")
    for key in ("out", "h", "y_perm", "dx", "dw_r", "dw1", "dw2"):
        if runs["1"][key] is None:
            continue
        assert np.array_equal(np.asarray(runs["1"][key]), np.asarray(runs["0"][key])), key
    f, b = _ref_all(w, inp, True)
    _check_full(w, runs["1"], inp, f, b)


@pytest.mark.parametrize("mode", ["1", "0"])
def test_fused_top1_tile_modes(mode, monkeypatch):
    """moe_forward's combine epilogue (top-1) on both tile modes, groups of ~1000 rows."""
    monkeypatch.setenv("MOE_GEMM_PAIR", mode)
    w = syn.Workload("top1-pair", T=4096, d=256, E=4, k=1, F=512, act="relu", dtype="bf16", cf=(5, 4))
    inp = syn.make_inputs(w, dy=False)
    res = run_gpu(w, inp, fused=True)
    f, _ = _ref_all(w, inp, False)
    check_routing(res, f, w)
    assert res["device_error"] == 0
    assert_close(res["out"], f["out"], TOL_BF16, "out")


# ------------------------------------------------------------------ bounded waits
def test_bounded_wait_gives_up_and_reports_timeout():
    """The kernels' on-chip wait, run on a barrier nothing completes, gives up
    after its limit, records MOE_DEVERR_TIMEOUT and returns; the context stays
    usable (a layer runs correctly afterwards)."""
    import time
    import sparse_mixture_experts_49_b300 as moe
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert moe.moe_get_device_error(ws) == moe.MOE_DEVERR_NONE
    t0 = time.perf_counter()
    moe.moe_selftest_bounded_wait(ws)
    code = moe.moe_get_device_error(ws)
    dt = time.perf_counter() - t0
    assert code == moe.MOE_DEVERR_TIMEOUT
    assert 3.0 < dt < 30.0, dt
    assert moe.moe_get_device_error(ws) == moe.MOE_DEVERR_NONE   # read clears the word
    w = SMALL["switch-small"]
    inp = syn.make_inputs(w, dy=False)
    res = run_gpu(w, inp)
    f, _ = _ref_all(w, inp, False)
    _check_full(w, res, inp, f, None)


# ------------------------------------------------------------------ full sizes, sampled outputs
@pytest.mark.parametrize("name", ["switch-base-top1", "gshard-top2-zipf", "dropless-top8-swiglu"])
def test_full_size_forward_sampled(name):
    w = syn.WORKLOADS[name]
    inp = syn.make_inputs(w, dy=False)
    res = run_gpu(w, inp)
    sample = np.random.default_rng(7).choice(w.T, 256, replace=False)
    f = O.forward(inp["x"], inp["w_r"], inp["bias"], (inp["w1"], inp["w2"]), tokens=sample, **oracle_kw(w))
    check_routing(res, f, w)
    check_router_values(res, f, w.dtype)
    assert res["device_error"] == 0
    assert_close(res["out"][sample], f["out"], TOL_BF16, "out (sampled tokens)")


def test_full_size_dropless_backward_sampled():
    """The dropless top-8 SwiGLU layer at its full size, forward + backward as
    the benchmark runs it: routing bit-exact over the whole batch, dX on
    sampled tokens and dW1 / dW2 on sampled experts against the oracle's
    token-by-token / expert-by-expert backward."""
    import sparse_mixture_experts_49_b300 as moe
    w = syn.WORKLOADS["dropless-top8-swiglu"]
    inp = syn.make_inputs(w, dy=True)
    cfg = moe.make_config(T=w.T, d_model=w.d, n_experts=w.E, top_k=w.k, d_ff=w.F, act=w.act, dtype=w.dtype,
                          renormalize=w.renormalize, capacity=-1, aux_alpha=w.alpha)
    bf = torch.bfloat16
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(dt)
    L = moe.MoELayer(cfg)
    x, w_r, w1, w2, dy = dev(inp["x"], bf), dev(inp["w_r"], torch.float32), dev(inp["w1"], bf), \
        dev(inp["w2"], bf), dev(inp["dy"], bf)
    L.forward(x, w_r, w1, w2)
    dx, dw_r, dw1, dw2 = L.backward(dy)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    st = L.balance_stats()                        # logging figures from the layer's own statistics
    assert st["drop_rate"] == 0.0                 # dropless
    assert st["aux"] == pytest.approx(float(L.aux.item()), rel=1e-5)
    rng = np.random.default_rng(11)
    toks = sorted(rng.choice(w.T, 48, replace=False).tolist())
    exps = sorted(rng.choice(w.E, 3, replace=False).tolist())
    ref = O.backward_sampled(inp["x"], inp["w_r"], inp["bias"], (inp["w1"], inp["w2"]), inp["dy"], tokens=toks,
                             experts_sampled=exps, **oracle_kw(w))
    assert np.array_equal(L.topk_idx.cpu().numpy(), ref["route"]["idx"])
    assert np.array_equal(L.slot.cpu().numpy(), ref["slots"]["slot"])
    got_dx = dx[toks].float().cpu().numpy().astype(np.float64)
    assert_close(got_dx, np.stack([ref["dx"][t] for t in toks]), TOL_BF16, "dx (sampled tokens)")
    for e in exps:
        assert_close(dw1[e].float().cpu().numpy(), ref["dw1"][e], TOL_BF16, f"dw1[{e}]")
        assert_close(dw2[e].float().cpu().numpy(), ref["dw2"][e], TOL_BF16, f"dw2[{e}]")
    dg, dh = backward_intermediates(torch, moe, cfg, L, w.T, w.k, w.E)
    assert_close(dg[toks], np.stack([ref["dg"][t] for t in toks]), TOL_BF16, "dg (sampled tokens)")
    assert_close(dh[toks], np.stack([ref["dh"][t] for t in toks]), TOL_BF16, "dh (sampled tokens)")
    # dW_r = dh^T x over the whole batch, from the layer's own dh, in fp64
    assert_close(np64(dw_r), dh.T @ inp["x"].astype(np.float64), TOL_ROUTER_BF16, "dw_r vs dh^T x (fp64)")


def test_full_size_large_training_sampled():
    """The large fine-grained training layer at its full size (T 4096, d 7168, 256 experts, top-8, SwiGLU
    7168 -> 2048 -> 7168, capacity factor 1.25, alpha 0.01), forward + backward as the benchmark runs it, on
    the same moe_synth draws the benchmark times: routing bit-exact over the whole batch (the K-split router
    over 112 K blocks), the router's values, out, dX, dg and dh on 256 sampled tokens, dW1 and dW2 on 4
    sampled experts (grouped-K GEMMs over ~128 rows per expert), and dW_r equal to dh^T x in fp64 over the
    whole batch (the router gradient's token-range split)."""
    import sparse_mixture_experts_49_b300 as moe
    w = syn.WORKLOADS["large-top8-swiglu"]
    inp = syn.make_inputs(w, experts=False, dy=True)
    b1, b2 = syn.expert_weight_bits(w)
    cfg = config_for(moe, w)
    bf = torch.bfloat16
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(dt)
    L = moe.MoELayer(cfg)
    x, w_r, dy = dev(inp["x"], bf), dev(inp["w_r"], torch.float32), dev(inp["dy"], bf)
    w1 = torch.from_numpy(b1).view(bf).cuda()
    w2 = torch.from_numpy(b2).view(bf).cuda()
    L.forward(x, w_r, w1, w2)
    dx, dw_r, dw1, dw2 = L.backward(dy)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    experts = lambda e: (syn.from_bf16_bits(b1[e]), syn.from_bf16_bits(b2[e]))
    rng = np.random.default_rng(5)
    toks = sorted(rng.choice(w.T, 256, replace=False).tolist())
    exps = sorted(rng.choice(w.E, 4, replace=False).tolist())
    kw = oracle_kw(w)
    f = O.forward(inp["x"], inp["w_r"], inp["bias"], experts, tokens=toks, **kw)
    n = int(L.offsets[-1].item())
    res = dict(idx=np64(L.topk_idx), load=np64(L.load), slot=np64(L.slot), kept=np64(L.kept),
               offsets=np64(L.offsets), row_token=np64(L.row_token[:n]), probs=np64(L.probs),
               gate=np64(L.topk_gate), importance=np64(L.importance), aux=float(L.aux.item()))
    check_routing(res, f, w)
    assert (f["slot"] < 0).any() and f["C"] == 160
    check_router_values(res, f, w.dtype)
    assert_close(np64(L.out)[toks], f["out"], TOL_BF16, "out (sampled tokens)")
    ref = O.backward_sampled(inp["x"], inp["w_r"], inp["bias"], experts, inp["dy"], tokens=toks,
                             experts_sampled=exps, **kw)
    assert_close(np64(dx)[toks], np.stack([ref["dx"][t] for t in toks]), TOL_BF16, "dx (sampled tokens)")
    dg, dh = backward_intermediates(torch, moe, cfg, L, w.T, w.k, w.E)
    assert_close(dg[toks], np.stack([ref["dg"][t] for t in toks]), TOL_BF16, "dg (sampled tokens)")
    assert_close(dh[toks], np.stack([ref["dh"][t] for t in toks]), TOL_BF16, "dh (sampled tokens)")
    for e in exps:
        assert_close(np64(dw1[e]), ref["dw1"][e], TOL_BF16, f"dw1[{e}]")
        assert_close(np64(dw2[e]), ref["dw2"][e], TOL_BF16, f"dw2[{e}]")
    assert_close(np64(dw_r), dh.T @ inp["x"].astype(np.float64), TOL_ROUTER_BF16, "dw_r vs dh^T x (fp64)")


# ------------------------------------------------------------------ the layer without its residual
@pytest.mark.parametrize("name", ["switch-small", "gshard-small", "dropless-small"])
def test_without_residual(name):
    """add_residual = 0: out = MoE(x) (zeros for fully dropped tokens), dX without the dY term, on the
    separate calls and on moe_forward (top-1: the dispatch writes the zeros, the second GEMM's epilogue the
    gated sums)."""
    w = SMALL[name].with_(add_residual=False, backward=True)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    _check_full(w, res, inp, f, b)
    fused = run_gpu(w, inp, fused=True)
    assert_close(fused["out"], f["out"], TOL_BF16, "out (moe_forward)")
    dropped = np.all(f["slot"] < 0, axis=1)
    assert np.all(fused["out"][dropped] == 0.0)


# ------------------------------------------------------------------ router variants
def _variant_inputs(w, sel_bias):
    """Inputs whose variant selection keys (score + correction bias, fp64) keep every consecutive gap among
    the k + 1 largest at least the generator's margin, so that the choice and its order are unique: the
    first T of 3T margin-conditioned tokens that pass."""
    from oracle import router_variants as RV
    big = syn.make_inputs(w.with_(T=3 * w.T), dy=True)
    if sel_bias is None:
        keep = np.arange(w.T)
    else:
        h = O.router_logits(big["x"], big["w_r"], big["bias"])
        key = (O.softmax(h) if w.score == "softmax" else RV.scores(h, w.score)) + sel_bias[None, :]
        top = -np.sort(-key, axis=1)[:, : w.k + 1]
        keep = np.nonzero((top[:, :-1] - top[:, 1:]).min(axis=1) >= syn.MARGIN)[0][: w.T]
        assert len(keep) == w.T
    big["x"], big["dy"] = big["x"][keep], big["dy"][keep]
    return big


@pytest.mark.parametrize("score,biased", [("sigmoid", False), ("sigmoid", True), ("sqrt_softplus", False),
                                          ("sqrt_softplus", True), ("softmax", True)])
def test_router_variants(score, biased):
    """Sigmoid and sqrt(softplus) scores and the selection-only correction bias ([Wiki] "Mixture-of-Experts",
    section 横断的知見) through the whole layer, forward and backward, against the oracle: routing bit-exact,
    the scores within the router's tolerance, every gate the score of its expert, layer outputs and gradients
    within the bf16 tolerance. Cluster-split router (E 64 over 2 CTAs) and a single-CTA one (E 32)."""
    for E in (64, 32):
        w = syn.Workload(f"variant-{score}-{biased}-{E}", T=1500, d=256, E=E, k=4, F=192, act="swiglu",
                         dtype="bf16", cf=(5, 4), renormalize=biased, router_std=1 / 16, score=score, backward=True)
        sel = (np.random.default_rng(E).standard_normal(E) * 0.02).astype(np.float32) if biased else None
        inp = _variant_inputs(w, sel)
        res = run_gpu(w, inp, backward=True, select_bias=sel)
        f, b = _ref_all(w, inp, True, sel_bias=sel)
        _check_full(w, res, inp, f, b)
        if not w.renormalize:
            assert np.array_equal(res["gate"], np.take_along_axis(res["probs"], res["idx"], axis=1))


def test_select_bias_update_sign_rule():
    """b_e += gamma sign(mean(load) - load_e) on the GPU, bit for bit against the oracle's update rounded to
    fp32 (a correctly rounded fp32 sum), including experts exactly at the mean."""
    import sparse_mixture_experts_49_b300 as moe
    from oracle import router_variants as RV
    rng = np.random.default_rng(21)
    for E, T, k in [(64, 1000, 4), (256, 4096, 8), (7, 10, 3)]:
        cfg = moe.make_config(T=T, d_model=64, n_experts=E, top_k=k, d_ff=64)
        load = rng.multinomial(T * k, np.ones(E) / E).astype(np.int32)
        if E == 7:
            load = np.array([4, 5, 3, 6, 4, 4, 4], np.int32)      # mean 30 / 7: no expert at the mean
        if E == 64:                                              # 8 experts exactly at the mean 62: no change
            load = np.concatenate([np.full(8, 62), rng.multinomial(56 * 62, np.ones(56) / 56)]).astype(np.int32)
            assert load.sum() == 64 * 62
        b = (rng.standard_normal(E) * 0.01).astype(np.float32)
        bd = torch.from_numpy(b).cuda()
        moe.moe_select_bias_update(cfg, torch.from_numpy(load).cuda(), bd, 0.001)
        torch.cuda.synchronize()
        ref = RV.update_bias(b.astype(np.float64), load, np.float64(np.float32(0.001))).astype(np.float32)
        assert np.array_equal(bd.cpu().numpy(), ref)


# ------------------------------------------------------------------ sizes that are not tile multiples
@pytest.mark.parametrize("act,k", [("relu", 1), ("swiglu", 2), ("relu", 3)])
def test_dims_multiple_of_8(act, k):
    """d_model 136 and d_ff 200 (multiples of 8, not of the 64-wide K step or the 128/256-wide N tiles):
    K tails come from the tensor maps' zero fill, N tails are clipped by the tile stores and masked in 8-column
    vectors elsewhere (the SwiGLU halves have a map each). Forward + backward on the separate calls, and
    moe_forward (top-1: the combine epilogue)."""
    w = syn.Workload(f"dims8-{act}-{k}", T=700, d=136, E=12, k=k, F=200, act=act, dtype="bf16", cf=(5, 4),
                     router_std=1 / np.sqrt(136), backward=True)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    _check_full(w, res, inp, f, b)
    fused = run_gpu(w, inp, fused=True)
    assert_close(fused["out"], f["out"], TOL_BF16, "out (moe_forward)")


# ------------------------------------------------------------------ No-Token-Left-Behind
@pytest.mark.parametrize("T,cf", [(1000, (3, 4)), (6200, (1, 2))])
def test_reroute_second_choice(T, cf):
    """Top-1 layers with rerouting ([Switch] section 論文の限界と、まだ分かっていないこと): the two-round
    slots (first choices, then the round-1 dropouts' second choices into the room left) bit-exact against
    the oracle over one and many dispatch blocks, forward and backward values within tolerance, and
    moe_forward on the same layer."""
    w = syn.Workload(f"reroute-{T}", T=T, d=256, E=16, k=1, F=256, act="relu", dtype="bf16", cf=cf, zipf_s=1.2,
                     router_std=1 / 16, reroute=True, backward=True)
    inp = syn.make_inputs(w, dy=True)
    res = run_gpu(w, inp, backward=True)
    f, b = _ref_all(w, inp, True)
    assert (f["slot"][:, 1] >= 0).any() and (f["slot"] < 0).all(axis=1).any()
    _check_full(w, res, inp, f, b)
    fused = run_gpu(w, inp, fused=True)
    check_routing(fused, f, w)
    assert_close(fused["out"], f["out"], TOL_BF16, "out (moe_forward)")


# ------------------------------------------------------------------ expert-choice routing
@pytest.mark.parametrize("T,E,C,act,dtype", [(1000, 16, 160, "swiglu", "bf16"), (700, 24, 50, "relu", "bf16"),
                                              (300, 8, 400, "relu", "bf16"), (512, 8, 96, "relu", "f32")])
def test_expert_choice(T, E, C, act, dtype):
    """Expert-choice routing ([Wiki] "Mixture-of-Experts", section 横断的知見): each expert's chosen tokens
    (its rows, in token order) bit-exact against the oracle, the gates and probabilities within the router's
    tolerance, the layer output and every gradient within the layer's; C above T takes every token. The
    inputs keep each expert's C-th and (C+1)-th scores at least 5e-5 apart (relative), far above fp32 error."""
    import sparse_mixture_experts_49_b300 as moe
    w = syn.Workload(f"ec-{T}-{E}-{C}", T=T, d=256 if dtype == "bf16" else 64, E=E, k=1, F=192 if dtype == "bf16" else 128,
                     act=act, dtype=dtype, cf=None, router_std=1 / 16 if dtype == "bf16" else None, backward=True)
    inp = syn.make_inputs(w, dy=True)
    cfg = moe.make_config(T=w.T, d_model=w.d, n_experts=w.E, top_k=1, d_ff=w.F, act=act, dtype=dtype, capacity=C,
                          expert_choice=True)
    L = moe.MoELayer(cfg)
    dt = L.dt
    from moe_cases import to_dev
    x, w_r = to_dev(torch, inp["x"], dt), to_dev(torch, inp["w_r"], torch.float32)
    w1, w2, dy = to_dev(torch, inp["w1"], dt), to_dev(torch, inp["w2"], dt), to_dev(torch, inp["dy"], dt)
    out = L.forward(x, w_r, w1, w2)
    dx, dw_r, dw1, dw2 = L.backward(dy)
    torch.cuda.synchronize()
    assert L.device_error() == 0
    f = O.forward_expert_choice(inp["x"], inp["w_r"], None, (inp["w1"], inp["w2"]), C=C, act=act)
    b = O.backward_expert_choice(inp["x"], inp["w_r"], None, (inp["w1"], inp["w2"]), inp["dy"], C=C, act=act)
    Ce = min(C, T)
    rows = E * Ce
    assert np.array_equal(np64(L.row_token[:rows]), f["row_token"])
    assert np.array_equal(np64(L.offsets), f["offsets"])
    tol_r = TOL_F32 if dtype == "f32" else TOL_ROUTER_BF16
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert_close(np64(L.probs), f["p"], tol_r, "probs")
    assert_close(np64(L.row_gate[:rows]), f["gate"].reshape(-1), tol_r, "row gates")
    assert_close(np64(L.importance), f["importance"], tol_r, "importance")
    assert_close(np64(out), f["out"], tol, "out")
    assert_close(np64(dx), b["dx"], tol, "dx")
    assert_close(np64(dw_r), b["dw_r"], tol, "dw_r")
    assert_close(np64(dw1), np.stack([b["dw1"][e] for e in range(E)]), tol, "dw1")
    assert_close(np64(dw2), np.stack([b["dw2"][e] for e in range(E)]), tol, "dw2")
    _, dh = backward_intermediates(torch, moe, cfg, L, T, 1, E)
    assert_close(dh, b["dh"], tol, "dh")
