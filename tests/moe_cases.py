"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np

import moe_synth as syn
from oracle import moe_oracle as O

TOL_BF16 = 2e-2    # max|err| <= TOL * max|ref| for bf16 experts with fp32 accumulation
TOL_F32 = 1e-5     # fp32 layer (CUDA-core fp32 throughout)
# fp32 router of a bf16 layer: the logits are exact bf16 x bf16 products summed
# in fp32 by the tensor core over d <= 7168 terms. With u = 2^-24 the typical
# rounding error of such a sum grows like sqrt(d) u sum|x_i w_i|, about
# 85 x 6e-8 x 30 = 1.5e-4 in a logit of size ~3 at d = 7168; probabilities
# inherit it relative to p. 1e-4 x max|ref| bounds that with margin and is
# still 200x tighter than the bf16 layer's 2e-2.
TOL_ROUTER_BF16 = 1e-4

# Small versions of the workload families: several 128 x 256 tiles, ragged
# tails (T, group sizes, F not a multiple of the tile), drops and empty experts.
SMALL = {
    "switch-small": syn.Workload("switch-small", T=1000, d=256, E=16, k=1, F=512, act="relu", dtype="bf16",
                                 cf=(5, 4)),
    "gshard-small": syn.Workload("gshard-small", T=2048, d=256, E=16, k=2, F=448, act="relu", dtype="bf16",
                                 cf=(2, 1), router_std=1 / 16, zipf_s=1.2, backward=True),
    "dropless-small": syn.Workload("dropless-small", T=1024, d=320, E=32, k=8, F=192, act="swiglu",
                                   dtype="bf16", cf=None, renormalize=True, router_std=1 / np.sqrt(320),
                                   backward=True),
    "large-small": syn.Workload("large-small", T=512, d=512, E=64, k=8, F=256, act="swiglu", dtype="bf16",
                                cf=(5, 4), backward=True),
}


def abi_capacity(moe, w) -> int:
    if w.cf is None:
        return -1
    return moe.moe_capacity(w.T, w.E, w.k, w.cf[0], w.cf[1], w.count_assignments)


def config_for(moe, w):
    return moe.make_config(T=w.T, d_model=w.d, n_experts=w.E, top_k=w.k, d_ff=w.F, act=w.act, dtype=w.dtype,
                           renormalize=w.renormalize, capacity=abi_capacity(moe, w), aux_alpha=w.alpha,
                           add_residual=w.add_residual, score=w.score, reroute=w.reroute)


def to_dev(torch, a, dtype):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to("cuda").to(dtype).contiguous()


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != __import__("torch").int32 \
        else t.cpu().numpy().astype(np.int64)


def run_gpu(w, inp, backward=False, topk_idx=None, layer=None, fused=False, select_bias=None):
    import torch
    import sparse_mixture_experts_49_b300 as moe
    cfg = config_for(moe, w)
    layer = layer or moe.MoELayer(cfg)
    dt = layer.dt
    x = to_dev(torch, inp["x"], dt)
    w_r = to_dev(torch, inp["w_r"], torch.float32)
    bias = to_dev(torch, inp["bias"], torch.float32)
    w1 = to_dev(torch, inp["w1"], dt)
    w2 = to_dev(torch, inp["w2"], dt)
    idx_t = None if topk_idx is None else torch.from_numpy(np.asarray(topk_idx, np.int32)).cuda()
    sel = None if select_bias is None else to_dev(torch, select_bias, torch.float32)
    if fused:
        layer.infer(x, w_r, w1, w2, bias)
    else:
        layer.forward(x, w_r, w1, w2, bias, idx_t, select_bias=sel)
    res = {}
    if backward:
        dy = to_dev(torch, inp["dy"], dt)
        dx, dw_r, dw1, dw2 = layer.backward(dy)
        dg, dh = backward_intermediates(torch, moe, cfg, layer, w.T, 2 if w.reroute else w.k, w.E)
        res.update(dx=np64(dx), dw_r=np64(dw_r), dw1=np64(dw1), dw2=np64(dw2), dg=dg, dh=dh)
    torch.cuda.synchronize()
    res.update(out=np64(layer.out), probs=np64(layer.probs), idx=np64(layer.topk_idx), gate=np64(layer.topk_gate),
               importance=np64(layer.importance), load=np64(layer.load), aux=float(layer.aux.item()),
               slot=np64(layer.slot), kept=np64(layer.kept), offsets=np64(layer.offsets))
    n = int(res["offsets"][-1])
    res["row_token"] = np64(layer.row_token[:n])
    res["x_perm"] = np64(layer.x_perm[:n])
    res["h"] = np64(layer.h[:n])
    res["y_perm"] = None if (fused and w.k == 1) else np64(layer.y_perm[:n])   # top-1 moe_forward writes no y_perm
    res["device_error"] = layer.device_error()
    return res


def oracle_kw(w):
    return dict(k=w.k, act=w.act, cf=w.cf, count_assignments=w.count_assignments, renormalize=w.renormalize,
                alpha=w.alpha, add_residual=w.add_residual, score=w.score, reroute=w.reroute)


def assert_close(got, ref, tol, what):
    """max|got - ref| <= tol * max|ref|; returns the measured ratio max|err| / max|ref| (printed, so that a run
    with -rP records the margin each check had)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    assert err <= tol * scale + 1e-30, f"{what}: max|err| {err:.3e} > {tol} x max|ref| {scale:.3e}"
    ratio = err / scale if scale > 0 else 0.0
    print(f"[tol] {what}: max|err|/max|ref| = {ratio:.3e} (bound {tol:g})")
    return ratio


def backward_intermediates(torch, moe, cfg, layer, T, k, E):
    """dg [T, k] and dh [T, E] (fp32) of the last moe_backward, read from the layer's workspace."""
    inter = moe.moe_backward_intermediates(cfg, layer.ws)
    torch.cuda.synchronize()
    base = layer.ws.data_ptr()
    dg = layer.ws[inter["dg"] - base: inter["dg"] - base + T * k * 4].view(torch.float32).view(T, k)
    dh = layer.ws[inter["dh"] - base: inter["dh"] - base + T * E * 4].view(torch.float32).view(T, E)
    return np64(dg), np64(dh)


def check_routing(res, ref, w):
    """Top-k indices, load, slots, kept counts, offsets and row ownership: bit-exact."""
    assert np.array_equal(res["idx"], ref["idx"]), "topk_idx differs"
    assert np.array_equal(res["load"], ref["load"]), "load differs"
    assert np.array_equal(res["slot"], ref["slot"]), "slot differs"
    assert np.array_equal(res["kept"], ref["kept"]), "kept differs"
    assert np.array_equal(res["offsets"], ref["offsets"]), "offsets differ"
    assert np.array_equal(res["row_token"], ref["row_token"]), "row_token differs"


def check_router_values(res, ref, dtype="f32"):
    tol = TOL_F32 if dtype == "f32" else TOL_ROUTER_BF16
    assert_close(res["probs"], ref["p"], tol, "probs")
    assert_close(res["gate"], ref["gate"], tol, "gates")
    assert_close(res["importance"], ref["importance"], tol, "importance")
    assert abs(res["aux"] - ref["aux"]) <= tol * abs(ref["aux"]) + 1e-9, ("aux", res["aux"], ref["aux"])


def expert_reference(w, inp, ref):
    """Oracle h and y for the packed rows, in the packed order."""
    x = inp["x"].astype(np.float64)
    hs, ys = [], []
    for e in range(w.E):
        lo, hi = int(ref["offsets"][e]), int(ref["offsets"][e + 1])
        if hi == lo:
            continue
        toks = ref["row_token"][lo:hi]
        f = O.expert_ffn(x[toks], inp["w1"][e].astype(np.float64), inp["w2"][e].astype(np.float64), w.act)
        hs.append(f["hid"])
        ys.append(f["y"])
    if not hs:
        return np.zeros((0, w.F)), np.zeros((0, w.d))
    return np.concatenate(hs), np.concatenate(ys)
