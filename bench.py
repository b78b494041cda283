"""Benchmark of the MoE FFN layer on B300.

One step = one pass of the whole layer over one batch. By default that is
the forward pass (router -> dispatch -> expert grouped GEMM -> combine, as
the single moe_forward call) of the Switch-Base-like top-1 workload: T = 8192 tokens (16 x 512), d_model 768,
128 experts, ReLU FFN 768 -> 3072 -> 768, capacity factor 1.25, bf16
activations and experts with an fp32 router. `--workload` picks another of
the bf16 workloads and `--pass fwdbwd` adds the backward pass (moe_backward)
to every step. Inputs are seeded synthetic data of the workload's shape,
resident in HBM before timing. The L2 cache is flushed (a 256 MiB write)
before every timed step, outside the step's CUDA events.

Prints one JSON line. `--impl reference` times the CPU oracle instead (the
reference arm of this build: a plain fp64 restatement of the layer).
Under torchrun (N > 1) every rank runs its own independent batch (data-
parallel replicas, no collective on the data path); time = max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as syn  # noqa: E402

WORKLOAD = "switch-base-top1"
METRIC = "MoE-layer tokens/s fwd & fwd+bwd; grouped-GEMM % bf16 peak; dispatch % HBM BW"
L2_FLUSH_BYTES = 256 << 20
# kernels of the library per call of the bf16 layer: router (W_r split, tensor-core logits, selection +
# statistics) 3, dispatch (count + scan, slots + row copy) 2, grouped GEMM 2, combine 1. moe_forward runs
# the same, but top-1 layers combine inside the second grouped-GEMM launch.
def forward_launches(w, fused_call: bool) -> int:
    combine = 0 if (fused_call and w.k == 1) else 1
    return 3 + 2 + 2 + combine
# moe_backward of the bf16 layer: combine backward 1, grouped GEMMs 4, router logit gradient 1, W_r split 1,
# router gradient GEMMs 2, dW_r part sum 1, unpermute-reduce 1
LAUNCHES_BACKWARD = 11


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    """Largest `value` across ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 9 for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": reasons}


# ---------------------------------------------------------------- measured DRAM traffic (from an ncu capture)
def gemm_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "common.cuh"):
        h.update(open(os.path.join(ROOT, "sparse_mixture_experts_49_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def gemm_traffic(workload):
    """dram read+write bytes per moe_expert_gemm call, from profiles/traffic.json, or None when the
    counters were taken on a different version of the GEMM kernel source."""
    try:
        t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[workload]
        return t["gemm_bytes_per_call"] if t.get("source_hash") == gemm_source_hash() else None
    except Exception:
        return None


# ---------------------------------------------------------------- algorithmic traffic and flops
def algorithmic(w, K_a: int, E_used: int):
    """Bytes / FLOPs each call must move or do (kept assignments only; the weights of the E_used experts
    that keep at least one token, read once; the expert-gradient outputs cover all E experts)."""
    s = 2  # bf16
    d, F, E, T, k, R1 = w.d, w.F, w.E, w.T, w.k, w.R1
    router_b = T * d * s + E * d * 4 + T * k * 8 + T * E * 4   # x, W_r, idx+gate, probs
    dispatch_b = T * d * s + K_a * d * s + T * k * 4 * 3 + K_a * 4
    act_b = K_a * F * s * 2 + (K_a * 2 * F * s if w.act == "swiglu" else 0)   # h out+in, pre-activations out
    gemm_b = w.nm * E_used * F * d * s + K_a * d * s * 2 + act_b   # weights, x_perm in, y_perm out, activations
    combine_b = T * d * s * 2 + K_a * d * s + T * k * 12
    gemm_flops = 2 * K_a * d * F * w.nm
    # backward: combine bwd (dY, y_perm in; dYp out), four grouped GEMMs (weights in, weight gradients out,
    # dYp / h / pre-activations / dA / x_perm in, dA and dXp out), router gradient, unpermute-reduce
    bwd_gemm_b = (w.nm * (E_used + E) * F * d * s + 2 * K_a * d * s + K_a * F * s
                  + (K_a * 2 * F * s if w.act == "swiglu" else 0)
                  + 3 * K_a * R1 * s + K_a * d * s + K_a * d * s)
    backward_b = (T * d * s + 2 * K_a * d * s + bwd_gemm_b + T * E * 4 * 2 + T * d * s + E * d * 4 * 2
                  + T * d * 4 * 2 + T * d * s * 2 + K_a * d * s)
    backward_flops = 2 * gemm_flops + 4 * T * E * d
    return dict(router=router_b, dispatch=dispatch_b, gemm=gemm_b, combine=combine_b, gemm_flops=gemm_flops,
                backward=backward_b, backward_flops=backward_flops, bwd_gemm_flops=2 * gemm_flops)


# ---------------------------------------------------------------- inputs on the device
DEVICE_DRAW_BYTES = 8 << 30   # expert weights above this size are drawn on the GPU (host draws take minutes)


def device_inputs(w, want_dy: bool):
    """x, W_r, bias (and dY) from moe_synth (margin-conditioned); expert weights per expert from moe_synth,
    or, for the largest workloads, from torch's seeded Philox generator on the GPU with the same
    distribution N(0, 0.1 / sqrt(fan_in)), rounded to bf16."""
    import torch
    bf = torch.bfloat16
    inp = syn.make_inputs(w, experts=False, dy=want_dy)
    dev = {"x": torch.from_numpy(inp["x"]).cuda().to(bf), "w_r": torch.from_numpy(inp["w_r"]).cuda(),
           "bias": None if inp["bias"] is None else torch.from_numpy(inp["bias"]).cuda(),
           "dy": torch.from_numpy(inp["dy"]).cuda().to(bf) if want_dy else None}
    w1 = torch.empty(w.E, w.R1, w.d, dtype=bf, device="cuda")
    w2 = torch.empty(w.E, w.d, w.F, dtype=bf, device="cuda")
    host_draw = w.E * (w.R1 * w.d + w.d * w.F) * 2 <= DEVICE_DRAW_BYTES
    if host_draw:
        for e in range(w.E):
            a, b = syn.expert_weights(w, e)
            w1[e].copy_(torch.from_numpy(a).to(bf))
            w2[e].copy_(torch.from_numpy(b).to(bf))
    else:
        g = torch.Generator(device="cuda")
        for e in range(w.E):
            g.manual_seed(w.seed * 1000003 + e)
            w1[e].copy_(torch.randn(w.R1, w.d, generator=g, device="cuda") * (w.expert_scale / math.sqrt(w.d)))
            w2[e].copy_(torch.randn(w.d, w.F, generator=g, device="cuda") * (w.expert_scale / math.sqrt(w.F)))
    dev["w1"], dev["w2"] = w1, w2
    dev["weights"] = "moe_synth (host, per expert)" if host_draw else "torch Philox on the GPU, seeded per expert"
    return inp, dev


# ---------------------------------------------------------------- our arm
def bench_workload(args):
    """The named workload, or a reduced case of it (--tokens / --experts) with its own seeds."""
    w = syn.WORKLOADS[args.workload]
    if args.tokens is None and args.experts is None:
        return w
    T = args.tokens or w.T
    E = args.experts or w.E
    return w.with_(name=f"{w.name}-T{T}-E{E}", T=T, E=E)


def run_ours(args):
    import torch
    import sparse_mixture_experts_49_b300 as moe
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    w = bench_workload(args)
    bwd = args.pass_ == "fwdbwd"
    inp, dv = device_inputs(w, bwd)
    cap = -1 if w.cf is None else moe.moe_capacity(w.T, w.E, w.k, w.cf[0], w.cf[1], w.count_assignments)
    cfg = moe.make_config(T=w.T, d_model=w.d, n_experts=w.E, top_k=w.k, d_ff=w.F, act=w.act, dtype=w.dtype,
                          renormalize=w.renormalize, capacity=cap, aux_alpha=w.alpha)
    stream = torch.cuda.current_stream()
    L = moe.MoELayer(cfg)
    x, w_r, bias, w1, w2, dy = dv["x"], dv["w_r"], dv["bias"], dv["w1"], dv["w2"], dv["dy"]
    if bwd:
        dx = torch.empty_like(x)
        dw_r = torch.empty(w.E, w.d, dtype=torch.float32, device="cuda")
        dw1 = torch.empty_like(w1)
        dw2 = torch.empty_like(w2)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    ev = lambda: torch.cuda.Event(enable_timing=True)
    calls = ["router", "dispatch", "gemm", "combine"] + (["backward"] if bwd else [])
    saved = dict(x=x, w_r=w_r, w1=w1, w2=w2, probs=L.probs, topk_idx=L.topk_idx, topk_gate=L.topk_gate,
                 slot=L.slot, expert_offsets=L.offsets, load=L.load, x_perm=L.x_perm, pre_act=L.pre_act, h=L.h,
                 y_perm=L.y_perm)
    pre_act = L.pre_act if bwd else None

    def step(marks=None):
        if marks: marks[0].record(torch.cuda.current_stream())
        moe.moe_router(cfg, x, w_r, bias, L.probs, L.topk_idx, L.topk_gate, L.importance, L.load, L.aux, L.ws)
        if marks: marks[1].record(torch.cuda.current_stream())
        moe.moe_dispatch(cfg, x, L.topk_idx, L.slot, L.kept, L.offsets, L.row_token, L.x_perm, L.ws)
        if marks: marks[2].record(torch.cuda.current_stream())
        moe.moe_expert_gemm(cfg, L.x_perm, L.offsets, w1, w2, pre_act, L.h, L.y_perm, L.ws)
        if marks: marks[3].record(torch.cuda.current_stream())
        moe.moe_combine(cfg, x, L.y_perm, L.topk_idx, L.topk_gate, L.slot, L.offsets, L.out)
        if marks: marks[4].record(torch.cuda.current_stream())
        if bwd:
            moe.moe_backward(cfg, saved, dy, dx, dw_r, dw1, dw2, L.ws)
            if marks: marks[5].record(torch.cuda.current_stream())

    def step_fused():
        # the whole forward layer in one call (inference): no y_perm and no combine launch for top-1
        # (inference: the [T, E] probabilities are only needed by the backward pass and are not written)
        moe.moe_forward(cfg, x, w_r, bias, w1, w2, None, L.topk_idx, L.topk_gate, L.importance, L.load, L.aux,
                        L.slot, L.kept, L.offsets, L.row_token, L.x_perm, L.h, L.y_perm if w.k > 1 else None, L.out,
                        L.ws)

    timed_step = step if bwd else step_fused

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise RuntimeError("device error during warm-up")
    K_a = int(L.offsets[-1].item())
    E_used = int((L.kept > 0).sum().item())   # experts whose weights the GEMMs read

    # per-call breakdown (eager launches, CUDA events between the ABI calls)
    n_eager = min(args.steps, 200)
    nc = len(calls)
    marks = [[ev() for _ in range(nc + 1)] for _ in range(n_eager)]
    for i in range(n_eager):
        flush.zero_()
        step(marks[i])
    torch.cuda.synchronize()
    per_call = {c: [m[j].elapsed_time(m[j + 1]) for m in marks] for j, c in enumerate(calls)}
    eager_ms = statistics.mean(m[0].elapsed_time(m[nc]) for m in marks)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        for _ in range(args.warmup):
            flush.zero_()
            g.replay()
        torch.cuda.synchronize()
        return g

    # per-call times inside a CUDA graph of the separate calls, with timing events between the calls (no host
    # launch gaps); the eager figures above are the fallback
    per_call_source = "eager"
    try:
        gm = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nc + 1)]
        g_m = capture(lambda: step(gm))
        reps = []
        for _ in range(min(args.steps, 100)):
            flush.zero_()
            g_m.replay()
            torch.cuda.synchronize()
            reps.append([gm[j].elapsed_time(gm[j + 1]) for j in range(nc)])
        per_call = {c: [r[j] for r in reps] for j, c in enumerate(calls)}
        per_call_source = "graph"
        del g_m
    except Exception as exc:  # events inside captured graphs not available: keep the eager figures
        per_call_source = f"eager ({type(exc).__name__})"

    # the separate ABI calls as one graph (reported beside the timed step for forward-only workloads)
    unfused_ms = None
    if not bwd:
        g_sep = capture(step)
        ue = [(ev(), ev()) for _ in range(n_eager)]
        for a_, b_ in ue:
            flush.zero_()
            a_.record(stream)
            g_sep.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        unfused_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in ue)
        del g_sep

    # the timed steps: the whole step captured once in a CUDA graph, replayed
    graph = capture(timed_step)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    s_ev = [ev() for _ in range(args.steps)]
    e_ev = [ev() for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()
        s_ev[i].record(stream)
        graph.replay()
        e_ev[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    clk = clocks.stop()
    if L.device_error() != 0:
        raise RuntimeError("device error during the timed steps")
    per_step = [a.elapsed_time(b) for a, b in zip(s_ev, e_ev)]
    ms_step = statistics.mean(per_step)
    total_ms = max_over_ranks(sum(per_step), world)
    value = world * w.T * args.steps / (total_ms / 1e3)

    # end to end: pinned host x (and dY) in, host out (and dX) back, through the same C-ABI calls. The copies
    # run on their own streams, double-buffered, so step i's upload and step i-1's download overlap step i's
    # compute; every step still moves its own input up and its own result down inside the timed region.
    bf = torch.bfloat16
    x_host = torch.from_numpy(inp["x"]).to(bf).pin_memory()
    out_host = [torch.empty(w.T, w.d, dtype=bf).pin_memory() for _ in range(2)]
    xb = [torch.empty_like(x) for _ in range(2)]
    ob = [torch.empty_like(x) for _ in range(2)]
    if bwd:
        dy_host = torch.from_numpy(inp["dy"]).to(bf).pin_memory()
        dx_host = [torch.empty(w.T, w.d, dtype=bf).pin_memory() for _ in range(2)]
        dyb = [torch.empty_like(x) for _ in range(2)]
        dxb = [torch.empty_like(x) for _ in range(2)]

    def io_step(b):
        if not bwd:
            moe.moe_forward(cfg, xb[b], w_r, bias, w1, w2, None, L.topk_idx, L.topk_gate, L.importance, L.load,
                            L.aux, L.slot, L.kept, L.offsets, L.row_token, L.x_perm, L.h,
                            L.y_perm if w.k > 1 else None, ob[b], L.ws)
            return
        moe.moe_router(cfg, xb[b], w_r, bias, L.probs, L.topk_idx, L.topk_gate, L.importance, L.load, L.aux, L.ws)
        moe.moe_dispatch(cfg, xb[b], L.topk_idx, L.slot, L.kept, L.offsets, L.row_token, L.x_perm, L.ws)
        moe.moe_expert_gemm(cfg, L.x_perm, L.offsets, w1, w2, pre_act, L.h, L.y_perm, L.ws)
        moe.moe_combine(cfg, xb[b], L.y_perm, L.topk_idx, L.topk_gate, L.slot, L.offsets, ob[b])
        sv = dict(saved, x=xb[b])
        moe.moe_backward(cfg, sv, dyb[b], dxb[b], dw_r, dw1, dw2, L.ws)

    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(10, args.steps // 4)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(s_up)
    for i in range(e2e_steps):
        b = i & 1
        with torch.cuda.stream(s_up):
            if i >= 2:
                s_up.wait_event(comp_done[b])            # xb[b] (dyb[b]) no longer read
            xb[b].copy_(x_host, non_blocking=True)
            if bwd:
                dyb[b].copy_(dy_host, non_blocking=True)
            up_done[b].record(s_up)
        stream.wait_event(up_done[b])
        if i >= 2:
            stream.wait_event(down_done[b])              # ob[b] (dxb[b]) already downloaded
        io_step(b)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(comp_done[b])
            out_host[b].copy_(ob[b], non_blocking=True)
            if bwd:
                dx_host[b].copy_(dxb[b], non_blocking=True)
            down_done[b].record(s_down)
    s_down.wait_event(down_done[(e2e_steps - 1) & 1])
    e1.record(s_down)
    torch.cuda.synchronize()
    if L.device_error() != 0:
        raise RuntimeError("device error during the end-to-end steps")
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * w.T * e2e_steps / (e2e_ms / 1e3)
    io_bytes = w.T * w.d * 2 * (2 if bwd else 1)

    hbm, tflops, tflops_sus, peak_src = load_peaks()
    alg = algorithmic(w, K_a, E_used)
    mean_call = {c: statistics.mean(v) for c, v in per_call.items()}
    kernels = {}
    for c in calls:
        gbs = alg[c] / (mean_call[c] * 1e-3) / 1e9
        kernels[c] = {"ms": round(mean_call[c], 5), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}
    gemm_tf = alg["gemm_flops"] / (mean_call["gemm"] * 1e-3) / 1e12
    kernels["gemm"].update({"TFLOP/s": round(gemm_tf, 1), "frac_bf16_peak": round(gemm_tf / tflops, 4)})
    if bwd:
        btf = alg["bwd_gemm_flops"] / (mean_call["backward"] * 1e-3) / 1e12
        kernels["backward"].update({"gemm_TFLOP/s": round(btf, 1), "frac_bf16_peak": round(btf / tflops, 4)})
    gemm_gbs = alg["gemm"] / (mean_call["gemm"] * 1e-3) / 1e9
    # the binding roof of the forward grouped GEMM: max(FLOPs / tensor peak, bytes / HBM peak)
    tensor_bound = alg["gemm_flops"] / (tflops * 1e12) > alg["gemm"] / (hbm * 1e9)
    traffic = gemm_traffic(w.name)
    if tensor_bound:
        # a contraction timed inside a long step under the power cap is held to the sustained bf16 peak; one that
        # ran at full clock, to the burst peak
        capped = "sw_power_cap" in (clk.get("reasons") or []) and tflops_sus > 0
        peak_t = tflops_sus if capped else tflops
        roof = {"bound": "tensor", "achieved": round(gemm_tf, 1), "peak": peak_t, "unit": "TFLOP/s",
                "frac": round(gemm_tf / peak_t, 4), "peak_kind": "sustained (power cap active)" if capped else "burst",
                "frac_of_burst_peak": round(gemm_tf / tflops, 4)}
    else:
        roof = {"bound": "hbm", "achieved": round(gemm_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gemm_gbs / hbm, 4)}
    roof.update({"kernel": "moe_expert_gemm (forward grouped GEMM, 2 launches)", "traffic": traffic,
                 "peak_source": peak_src, "algorithmic_bytes_per_call": alg["gemm"],
                 "algorithmic_flops_per_call": alg["gemm_flops"]})
    launches = forward_launches(w, not bwd) + (LAUNCHES_BACKWARD if bwd else 0)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "pass": args.pass_, "T": w.T, "d_model": w.d, "experts": w.E,
                   "top_k": w.k, "d_ff": w.F, "act": w.act, "renormalize": w.renormalize,
                   "capacity_factor": None if w.cf is None else f"{w.cf[0]}/{w.cf[1]}", "capacity": cap,
                   "capacity_reading": "floor(k*T*cf/E)" if w.cf is not None else "none (dropless)",
                   "kept_assignments": K_a, "experts_with_tokens": E_used, "expert_weights": dv["weights"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every timed step (256 MiB write, outside the step's events)"},
        "roofline": roof,
        "kernels": kernels,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                "d2h_bytes_per_step": io_bytes, "call": "moe_forward" if not bwd else "separate calls + moe_backward",
                "overlap": "uploads and downloads on their own streams, double-buffered, overlapping compute"},
        "gpu_launches": launches * args.steps,
        "eager_ms_per_step": round(eager_ms, 5),
        "step_call": "moe_forward (one call: router, dispatch, expert GEMMs, combine fused into the second GEMM "
                     "for top-1)" if not bwd else
                     "moe_router, moe_dispatch, moe_expert_gemm, moe_combine, moe_backward",
        "separate_calls_graph_ms_per_step": None if unfused_ms is None else round(unfused_ms, 5),
        "timing": "step replayed as one CUDA graph; per-call figures from the separate ABI calls with events "
                  "between them, replayed as a CUDA graph (per_call_source)",
        "per_call_source": per_call_source,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall1 - t_wall0, 3),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, inp, bwd)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- the oracle, timed on the host cores
def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


HOST_F64_WEIGHTS_MAX = 16 << 30   # the oracle's fp64 copy of the expert weights must fit in host RAM


def _oracle_weights(w):
    if w.E * (w.R1 * w.d + w.d * w.F) * 8 > HOST_F64_WEIGHTS_MAX:
        return None
    w1, w2 = syn.all_expert_weights(w)
    return w1.astype(np.float64), w2.astype(np.float64)


def _oracle_step(w, inp, Ts, weights, bwd):
    from oracle import moe_oracle as O
    kw = dict(k=w.k, act=w.act, cf=w.cf, count_assignments=w.count_assignments, renormalize=w.renormalize,
              alpha=w.alpha)
    x = inp["x"][:Ts]
    O.forward(x, inp["w_r"], inp["bias"], weights, **kw)
    if bwd:
        O.backward(x, inp["w_r"], inp["bias"], weights, inp["dy"][:Ts], **kw)


def _oracle_batch(w, inp, weights, bwd, budget_s):
    """Largest batch of the first Ts tokens (T halved until one step fits the budget)."""
    Ts = w.T
    while Ts > 64:
        t0 = time.perf_counter()
        _oracle_step(w.with_(T=Ts), inp, Ts, weights, bwd)
        if time.perf_counter() - t0 <= budget_s:
            break
        Ts //= 2
    return Ts


def _sample_text(w, Ts, bwd):
    what = "forward + backward" if bwd else "forward"
    part = f"the full batch (T={w.T})" if Ts == w.T else f"the first {Ts} of the {w.T} tokens as one batch " \
                                                          "(same capacity factor)"
    return f"one {what} of {part} of {w.name}, fp64 numpy oracle, expert weights widened to fp64 before timing"


def cpu_baseline(w, inp, bwd):
    weights = _oracle_weights(w)
    if weights is None:
        return {"value": None, "unit": "tokens/s", "cores": _oracle_threads(), "kind": "oracle",
                "sample": f"not run: the oracle's fp64 expert weights of {w.name} exceed {HOST_F64_WEIGHTS_MAX >> 30} GiB "
                          "of host memory"}
    Ts = _oracle_batch(w, inp, weights, bwd, 20.0)
    # the sampled batch, repeated until at least 10 s of CPU work have been timed
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(w.with_(T=Ts), inp, Ts, weights, bwd)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0:
            break
    return {"value": round(Ts * reps / dt, 1), "unit": "tokens/s", "cores": _oracle_threads(), "kind": "oracle",
            "sample": _sample_text(w, Ts, bwd) + f", {reps} time(s); {dt:.2f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = bench_workload(args)
    bwd = args.pass_ == "fwdbwd"
    inp = syn.make_inputs(w, experts=False, dy=bwd)
    weights = _oracle_weights(w)
    if weights is None:
        print(json.dumps({"impl": "reference", "unavailable": f"the oracle's fp64 expert weights of {w.name} do not "
                                                              "fit in host memory"}), flush=True)
        return
    budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    Ts = _oracle_batch(w, inp, weights, bwd, budget)
    ws = w.with_(T=Ts)
    for _ in range(args.warmup):
        _oracle_step(ws, inp, Ts, weights, bwd)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(ws, inp, Ts, weights, bwd)
    dt = time.perf_counter() - t0
    value = Ts * args.steps / dt
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name, "pass": args.pass_, "T_sample": Ts},
           "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": _oracle_threads(),
                            "kind": "oracle", "sample": "each step: " + _sample_text(w, Ts, bwd)},
           "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


BENCH_WORKLOADS = [n for n, w in syn.WORKLOADS.items() if w.dtype == "bf16"]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=BENCH_WORKLOADS, default=WORKLOAD)
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "fwdbwd"], default=None,
                    help="default: fwdbwd for the workloads that include the backward pass, else fwd")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (smaller cases of the same kernels, e.g. for profiling)")
    ap.add_argument("--experts", type=int, default=None, help="override E (with the same per-expert shapes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.pass_ is None:
        args.pass_ = "fwdbwd" if syn.WORKLOADS[args.workload].backward else "fwd"
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
