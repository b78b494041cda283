"""Benchmark of the MoE FFN layer on B300.

One step = one pass of the whole layer over one batch. By default that is
the forward and backward pass (moe_router -> moe_dispatch -> moe_expert_gemm
-> moe_combine -> moe_backward) of the large fine-grained training layer:
T = 4096 tokens, d_model 7168, 256 experts, top-8, SwiGLU FFN
7168 -> 2048 -> 7168, capacity factor 1.25, bf16 experts with an fp32
router and the alpha = 0.01 load-balancing loss in the backward pass.
`--workload` picks another bf16 workload; `--pass fwd` times the forward
alone, as the single moe_forward call. Inputs (tokens, router weights, every
expert's weights, the upstream gradient) are the seeded synthetic draws of
moe_synth, the same the parity tests give the oracle; they are resident in
HBM before timing. The L2 cache is flushed (a 256 MiB write) before every
timed step, outside the step's CUDA events.

Besides the step time the JSON line carries, per kernel of the step, its
launch duration inside the step (the captured step graph with every kernel
node between two event-record nodes, replayed after an L2 flush), its
algorithmic bytes and FLOPs, and the fraction of the measured HBM or
sustained bf16 peak they reach; the `roofline` object is the step's longest
grouped-GEMM launch, timed in the timed steps themselves by two event-record
nodes added around its kernel node in the timed graph.

Prints one JSON line. `--impl reference` times the CPU oracle instead (the
reference arm of this build: a plain fp64 restatement of the layer).
Under torchrun (N > 1) every rank runs its own independent batch (data-
parallel replicas, no collective on the data path); time = max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as syn  # noqa: E402

WORKLOAD = "large-top8-swiglu"
METRIC = "MoE-layer tokens/s fwd & fwd+bwd; grouped-GEMM % bf16 peak; dispatch % HBM BW"
L2_FLUSH_BYTES = 256 << 20
GEMM_ROLES = ("gemm1", "gemm2", "gemm2_combine", "dH", "dW2", "dXp", "dW1")
CSRC = os.path.join(ROOT, "sparse_mixture_experts_49_b300", "csrc")


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

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

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


# ---------------------------------------------------------------- algorithmic traffic and flops
def algorithmic(w, K_a: int, E_used: int):
    """Bytes / FLOPs each ABI call must move or do (kept assignments only; the weights of the E_used experts
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


def gemm_launch_algorithmic(role: str, w, K_a: int, E_used: int, training: bool):
    """(bytes, FLOPs) one grouped-GEMM launch must move / do: the weights of the experts that keep tokens read
    once (weight-gradient outputs: every expert's written once), the packed activation rows it reads and
    writes once, kept rows only."""
    s = 2
    d, F, E, R1 = w.d, w.F, w.E, w.R1
    swiglu = w.act == "swiglu"
    if role == "gemm1":       # x_perm W1^T -> h (+ SwiGLU pre-activations when training)
        b = E_used * R1 * d * s + K_a * d * s + K_a * F * s + (K_a * 2 * F * s if swiglu and training else 0)
        return b, 2 * K_a * R1 * d
    if role == "gemm2":       # h W2^T -> y_perm
        return E_used * d * F * s + K_a * F * s + K_a * d * s, 2 * K_a * d * F
    if role == "gemm2_combine":   # h W2^T, gated residual sum into out (kept rows: x read, out written)
        return E_used * d * F * s + K_a * F * s + 2 * K_a * d * s, 2 * K_a * d * F
    if role == "dH":          # dYp W2 -> activation backward -> dA (reads the saved pre-activations or h)
        saved = K_a * 2 * F * s if swiglu else K_a * F * s
        return E_used * d * F * s + K_a * d * s + saved + K_a * R1 * s, 2 * K_a * d * F
    if role == "dW2":         # dYp^T h per expert -> dW2 (all E written)
        return E * d * F * s + K_a * d * s + K_a * F * s, 2 * K_a * d * F
    if role == "dXp":         # dA W1 -> dXp
        return E_used * R1 * d * s + K_a * R1 * s + K_a * d * s, 2 * K_a * R1 * d
    if role == "dW1":         # dA^T x_perm per expert -> dW1 (all E written)
        return E * R1 * d * s + K_a * R1 * s + K_a * d * s, 2 * K_a * R1 * d
    raise ValueError(role)


# ---------------------------------------------------------------- kernel roles from their names
_GEMM_ARGS = re.compile(r"grouped_gemm_kernel<(\d+), (\d+), (\d+), (\d+), (\d+)>")
# the ABI call each library kernel belongs to (kernel name -> call)
_CALL_OF = [("router_dh", "backward"), ("router_wsplit6", "backward"), ("router_dwr_sum", "backward"),
            ("router", "router"), ("dispatch", "dispatch"), ("combine_backward", "backward"),
            ("unpermute", "backward"), ("combine", "combine")]


def demangle(names):
    """C++ names of mangled kernel symbols (c++filt; the names unchanged when it is missing)."""
    try:
        r = subprocess.run(["c++filt"], input="\n".join(names), capture_output=True, text=True, timeout=30)
        out = r.stdout.splitlines()
        if r.returncode == 0 and len(out) == len(names):
            return out
    except Exception:
        pass
    return list(names)


def kernel_roles(names):
    """(role, ABI call) of each launch of one step, in launch order, from the demangled kernel names:
    grouped-GEMM launches by their template arguments (PAIR, GROUP_K, A_MN, B_MN, EPI) and position (the first
    grouped-K launch of the backward pass is dW2, the second dW1), every other kernel by its own name."""
    roles, gk = [], 0
    for n in names:
        if "wgrad_kernel" in n:   # the weight gradients' own kernel: dW2, then dW1, like the grouped-K GEMMs
            roles.append(("dW2" if gk == 0 else "dW1", "backward"))
            gk += 1
            continue
        m = _GEMM_ARGS.search(n)
        if m:
            _, group_k, _, b_mn, epi = (int(v) for v in m.groups())
            if epi == 5:
                roles.append(("router_grad_dW_r" if group_k else "router_grad_dX_r", "backward"))
            elif group_k:
                roles.append(("dW2" if gk == 0 else "dW1", "backward"))
                gk += 1
            elif epi in (1, 2):
                roles.append(("gemm1", "gemm"))
            elif epi == 6:
                roles.append(("gemm2_combine", "gemm"))
            elif epi in (3, 4):
                roles.append(("dH", "backward"))
            elif b_mn:
                roles.append(("dXp", "backward"))
            else:
                roles.append(("gemm2", "gemm"))
            continue
        head = re.split(r"[<(]", n.replace("(anonymous namespace)", "anon").replace("void ", "", 1), maxsplit=1)[0]
        ident = head.split("::")[-1].strip()
        call = next((c for key, c in _CALL_OF if key in ident), "other")
        roles.append((ident, call))
    return roles


def source_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(CSRC, f), "rb").read())
    return h.hexdigest()[:16]


# the sources each kernel role is built from (a measured traffic figure holds while they are unchanged)
def role_sources(role: str):
    if role.startswith("dW"):
        return ("gemm_tc.cu", "wgrad.cu", "common.cuh")
    if role.startswith(("gemm", "dH", "dXp", "router_grad")):
        return ("gemm_tc.cu", "common.cuh")
    if role.startswith("router"):
        return ("router.cu", "common.cuh") if "dh" not in role and "split6" not in role and "dwr" not in role \
            else ("backward.cu", "common.cuh")
    if role.startswith("dispatch"):
        return ("dispatch.cu", "common.cuh")
    return ("combine.cu", "common.cuh")


def measured_traffic(workload: str, role: str):
    """dram read + write bytes per launch of `role` from profiles/traffic.json, or None when the counters were
    taken on a different version of the kernel's source (or not at all)."""
    try:
        t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))[workload][role]
        return t["dram_bytes_per_launch"] if t.get("source_hash") == source_hash(role_sources(role)) else None
    except Exception:
        return None


# ---------------------------------------------------------------- per-kernel times by replaying graph nodes
def _drv_ok(res):
    from cuda.bindings import driver as drv
    err = res[0] if isinstance(res, tuple) else res
    if err != drv.CUresult.CUDA_SUCCESS:
        raise RuntimeError(f"CUDA driver call failed: {err}")
    return res[1:] if isinstance(res, tuple) else None


def _listing(fn, *head):
    """(nodes) of a driver graph query, whichever of its signatures the bindings expose (some also return edge
    data): the first list in the result is the nodes, the last integer the count."""
    n = [v for v in _drv_ok(fn(*head, 0)) if isinstance(v, int)][-1]
    if n == 0:
        return []
    return list(next(v for v in _drv_ok(fn(*head, n)) if isinstance(v, (list, tuple))))


def graph_kernels(graph):
    """Kernel nodes of a captured graph in launch order (every node after its dependencies, ready nodes in
    creation order), with {key: node}, {key: ancestors} and {key: group id} (see concurrent_groups)."""
    from cuda.bindings import driver as drv
    nodes = _listing(drv.cuGraphGetNodes, graph)
    by_key = {int(n): n for n in nodes}
    pos = {int(n): i for i, n in enumerate(nodes)}          # creation order
    deps = {int(n): [int(d) for d in _listing(drv.cuGraphNodeGetDependencies, n)] for n in nodes}
    order = topological_order(deps, pos)
    anc = {}
    for k in order:
        anc[k] = set(deps[k]).union(*(anc[d] for d in deps[k])) if deps[k] else set()
    kern = [k for k in order
            if _drv_ok(drv.cuGraphNodeGetType(by_key[k]))[0] == drv.CUgraphNodeType.CU_GRAPH_NODE_TYPE_KERNEL]
    return by_key, kern, anc, concurrent_groups(kern, anc)


def kernel_name(node):
    from cuda.bindings import driver as drv
    params = _drv_ok(drv.cuGraphKernelNodeGetParams(node))[0]
    func = params.func
    if not int(func):
        func = _drv_ok(drv.cuKernelGetFunction(params.kern))[0]
    name = _drv_ok(drv.cuFuncGetName(func))[0]
    return name.decode() if isinstance(name, bytes) else str(name)


class Bracketed:
    """A captured graph in which each of the given kernel nodes sits between two event-record nodes (before:
    after the node's dependencies; after: before its dependents), instantiated. `launch(stream, events)` sets
    every record node's event for this launch ({key: (start, end)}) and launches the graph; the events are
    recorded on the stream the graph runs on, right around the kernel, inside the graph's own run."""

    def __init__(self, graph, by_key, keys):
        from cuda.bindings import driver as drv
        self.drv = drv
        ev0 = _drv_ok(drv.cuEventCreate(0))[0]
        self.placeholder = ev0
        self.nodes = {}
        for k in keys:
            kn = by_key[k]
            before = _listing(drv.cuGraphNodeGetDependencies, kn)
            after = _listing(drv.cuGraphNodeGetDependentNodes, kn)
            a = _drv_ok(drv.cuGraphAddEventRecordNode(graph, before, len(before), ev0))[0]
            if before:
                _drv_ok(drv.cuGraphRemoveDependencies(graph, before, [kn] * len(before), None, len(before)))
            _drv_ok(drv.cuGraphAddDependencies(graph, [a], [kn], None, 1))
            b = _drv_ok(drv.cuGraphAddEventRecordNode(graph, [kn], 1, ev0))[0]
            if after:
                _drv_ok(drv.cuGraphRemoveDependencies(graph, [kn] * len(after), after, None, len(after)))
                _drv_ok(drv.cuGraphAddDependencies(graph, [b] * len(after), after, None, len(after)))
            self.nodes[k] = (a, b)
        self.exec = _drv_ok(drv.cuGraphInstantiate(graph, 0))[0]

    def new_events(self):
        return {k: (_drv_ok(self.drv.cuEventCreate(0))[0], _drv_ok(self.drv.cuEventCreate(0))[0])
                for k in self.nodes}

    def launch(self, stream, events=None):
        drv = self.drv
        if events:
            for k, (a, b) in self.nodes.items():
                _drv_ok(drv.cuGraphExecEventRecordNodeSetEvent(self.exec, a, events[k][0]))
                _drv_ok(drv.cuGraphExecEventRecordNodeSetEvent(self.exec, b, events[k][1]))
        _drv_ok(drv.cuGraphLaunch(self.exec, drv.CUstream(stream.cuda_stream)))

    def elapsed(self, e0, e1):
        return float(_drv_ok(self.drv.cuEventElapsedTime(e0, e1))[0])

    def destroy_events(self, events):
        for a, b in events.values():
            _drv_ok(self.drv.cuEventDestroy(a))
            _drv_ok(self.drv.cuEventDestroy(b))

    def close(self):
        _drv_ok(self.drv.cuGraphExecDestroy(self.exec))
        _drv_ok(self.drv.cuEventDestroy(self.placeholder))


def capture_graph(step, stream):
    """`step` captured into a kept (not yet instantiated) torch CUDA graph; returns (the torch graph, which
    owns the capture, and the raw driver graph)."""
    import torch
    from cuda.bindings import driver as drv
    g = torch.cuda.CUDAGraph(keep_graph=True)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    return g, drv.CUgraph(g.raw_cuda_graph())


def time_kernels_in_step(step, stream, flush, reps: int):
    """Per-kernel launch times inside the step: `step` captured into a CUDA graph with every kernel node
    between two event-record nodes, replayed `reps` times (each after an L2 flush), each kernel timed from its
    own pair of events. Kernel nodes that the step can run side by side (consecutive in launch order, with no
    path between them in the graph, as when a call forks onto a second stream) form a group, timed from the
    earliest start to the latest end of its members. Returns ([(mangled name, mean ms, group)] in launch
    order, {group: mean ms} for groups of two or more)."""
    import torch
    g, graph = capture_graph(step, stream)
    by_key, kern, anc, group_of = graph_kernels(graph)
    names = [kernel_name(by_key[k]) for k in kern]
    br = Bracketed(graph, by_key, kern)
    for _ in range(2):                            # warm-up launches
        flush.zero_()
        br.launch(stream)
    torch.cuda.synchronize()
    runs = []
    for _ in range(reps):
        evs = br.new_events()
        flush.zero_()
        br.launch(stream, evs)
        runs.append(evs)
    torch.cuda.synchronize()
    first = kern[0]                               # the step's first kernel precedes every other one
    per = {k: [] for k in kern}
    span = {}
    for evs in runs:
        ref = evs[first][0]
        t = {k: (br.elapsed(ref, evs[k][0]), br.elapsed(ref, evs[k][1])) for k in kern}
        for k in kern:
            per[k].append(t[k][1] - t[k][0])
        for gid in set(group_of.values()):
            mem = [k for k in kern if group_of[k] == gid]
            if len(mem) > 1:
                span.setdefault(gid, []).append(max(t[k][1] for k in mem) - min(t[k][0] for k in mem))
        br.destroy_events(evs)
    br.close()
    del g
    out = [(names[i], statistics.mean(per[k]), group_of[k]) for i, k in enumerate(kern)]
    return out, {gid: statistics.mean(v) for gid, v in span.items()}


def topological_order(deps, pos):
    """Node keys in an order that puts every node after its dependencies, ready nodes taken in creation order
    (`pos`); raises on a cycle."""
    indeg = {k: len(v) for k, v in deps.items()}
    children = {k: [] for k in deps}
    for k, ds in deps.items():
        for d in ds:
            children[d].append(k)
    ready = sorted((k for k, n in indeg.items() if n == 0), key=pos.get)
    order = []
    while ready:
        k = ready.pop(0)
        order.append(k)
        for c in children[k]:
            indeg[c] -= 1
            if indeg[c] == 0:
                ready.append(c)
        ready.sort(key=pos.get)
    if len(order) != len(deps):
        raise RuntimeError("the captured step graph has a cycle")
    return order


def concurrent_groups(kern, anc):
    """Group ids of kernel nodes (in launch order): a node joins the current group when no node of it is an
    ancestor or a descendant of the node (they can run side by side), else it opens the next group."""
    group_of, cur, gid = {}, [], 0
    for k in kern:
        if cur and all(c not in anc[k] and k not in anc[c] for c in cur):
            cur.append(k)
        else:
            gid += 1 if cur else 0
            cur = [k]
        group_of[k] = gid
    return group_of


# ---------------------------------------------------------------- inputs on the device
def device_inputs(w, want_dy: bool):
    """x, W_r, bias (and dY) from moe_synth (margin-conditioned), and every expert's weights from moe_synth's
    per-expert draws (threaded), uploaded as bf16."""
    import torch
    bf = torch.bfloat16
    inp = syn.make_inputs(w, experts=False, dy=want_dy)
    dev = {"x": torch.from_numpy(inp["x"]).cuda().to(bf), "w_r": torch.from_numpy(inp["w_r"]).cuda(),
           "bias": None if inp["bias"] is None else torch.from_numpy(inp["bias"]).cuda(),
           "dy": torch.from_numpy(inp["dy"]).cuda().to(bf) if want_dy else None}
    t0 = time.perf_counter()
    b1, b2 = syn.expert_weight_bits(w)
    t_draw = time.perf_counter() - t0
    dev["w1"] = torch.from_numpy(b1).view(bf).cuda()
    dev["w2"] = torch.from_numpy(b2).view(bf).cuda()
    del b1, b2
    dev["weights"] = f"moe_synth per-expert draws (host, {t_draw:.1f} s on {min(32, os.cpu_count() or 1)} threads)"
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
    # launch gaps); eager launches with events between the calls are the fallback
    nc = len(calls)
    n_rep = max(3, min(args.steps, 100))
    per_call_source = "graph"
    try:
        gm = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nc + 1)]
        g_m = capture(lambda: step(gm))
        reps = []
        for _ in range(n_rep):
            flush.zero_()
            g_m.replay()
            torch.cuda.synchronize()
            reps.append([gm[j].elapsed_time(gm[j + 1]) for j in range(nc)])
        per_call = {c: [r[j] for r in reps] for j, c in enumerate(calls)}
        del g_m
    except Exception as exc:  # events inside captured graphs not available
        per_call_source = f"eager ({type(exc).__name__})"
        marks = [[ev() for _ in range(nc + 1)] for _ in range(n_rep)]
        for i in range(n_rep):
            flush.zero_()
            step(marks[i])
        torch.cuda.synchronize()
        per_call = {c: [m[j].elapsed_time(m[j + 1]) for m in marks] for j, c in enumerate(calls)}

    # per-kernel launch times inside the step (every kernel node of the step graph between two event-record
    # nodes), in launch order
    try:
        launches, group_ms = time_kernels_in_step(timed_step, stream, flush, reps=max(3, min(args.steps, 20)))
        launch_error = None
    except Exception as exc:
        launches, group_ms, launch_error = [], {}, f"{type(exc).__name__}: {exc}"[:300]
    names = demangle([n for n, _, _ in launches])
    roles = kernel_roles(names)
    # the launch the roofline reports: the longest grouped-GEMM launch that runs alone
    solo = [i for i, ((_, ms, gid), (role, _)) in enumerate(zip(launches, roles))
            if role in GEMM_ROLES and gid not in group_ms]
    top_index = max(solo, key=lambda i: launches[i][1]) if solo else None

    # the timed steps: the whole step captured once in a CUDA graph and replayed; the reported launch sits
    # between two event-record nodes of that graph, so its duration comes from the timed steps themselves
    live = None
    try:
        if top_index is None:
            raise RuntimeError("no solo grouped-GEMM launch")
        g_t, raw_t = capture_graph(timed_step, stream)
        by_key_t, kern_t, _, _ = graph_kernels(raw_t)
        if len(kern_t) != len(launches) or demangle([kernel_name(by_key_t[kern_t[top_index]])]) != [names[top_index]]:
            raise RuntimeError("the step graph changed between captures")
        live = Bracketed(raw_t, by_key_t, [kern_t[top_index]])
        for _ in range(args.warmup):
            flush.zero_()
            live.launch(stream)
        torch.cuda.synchronize()
        run_step = lambda i: live.launch(stream, live_ev[i])
        live_ev = [live.new_events() for _ in range(args.steps)]
        timed_how = "graph (driver launch), the reported launch bracketed by event-record nodes"
    except Exception as exc:
        live, live_error = None, f"{type(exc).__name__}: {exc}"[:200]
        graph = capture(timed_step)
        run_step = lambda i: graph.replay()
        timed_how = f"graph (torch replay; no live launch timing: {live_error})"
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
        run_step(i)
        e_ev[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    clk = clocks.stop()
    live_ms = None
    if live is not None:
        (k_top,) = live.nodes.keys()
        live_ms = [live.elapsed(*evs[k_top]) for evs in live_ev]
        for evs in live_ev:
            live.destroy_events(evs)
        live.close()
        del g_t
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

    hbm, tflops_burst, tflops_sus, peak_src = load_peaks()
    # every time below is taken inside the running step, so a contraction is set against the sustained bf16
    # figure (the burst one is for a kernel timed alone)
    tflops = tflops_sus if tflops_sus > 0 else tflops_burst
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

    # per launch: the grouped GEMMs against max(FLOPs / tensor peak, bytes / HBM peak); the token kernels'
    # launch times are summed per call and set against the call's algorithmic bytes
    table, call_launch_ms = [], {}

    def against_bound(row, b, f, ms):
        t_hbm, t_tc = b / (hbm * 1e9), f / (tflops * 1e12)
        row.update({"bytes": b, "flops": f, "GB/s": round(b / (ms * 1e-3) / 1e9, 1),
                    "TFLOP/s": round(f / (ms * 1e-3) / 1e12, 1), "bound": "tensor" if t_tc > t_hbm else "hbm",
                    "frac_of_bound": round(max(t_hbm, t_tc) * 1e3 / ms, 4),
                    "frac_bf16_peak": round(f / (ms * 1e-3) / 1e12 / tflops, 4)})
        return row

    for idx, ((_, ms, gid), name, (role, call)) in enumerate(zip(launches, names, roles)):
        row = {"kernel": role, "call": call, "ms": round(ms, 5), "index": idx}
        if gid in group_ms:
            row["group"] = gid
        if role in GEMM_ROLES:
            against_bound(row, *gemm_launch_algorithmic(role, w, K_a, E_used, bwd), ms)
            row["traffic"] = measured_traffic(w.name, role)
        else:
            call_launch_ms[call] = call_launch_ms.get(call, 0.0) + ms
            row["traffic"] = measured_traffic(w.name, role)
        row["name"] = name[:120]
        table.append(row)
    # launches the step runs side by side, replayed together
    concurrent = []
    for gid, ms in group_ms.items():
        rows = [r for r in table if r.get("group") == gid]
        unit = {"kernels": [r["kernel"] for r in rows], "ms": round(ms, 5), "name": " + ".join(r["kernel"] for r in rows)}
        if all("bytes" in r for r in rows):
            against_bound(unit, sum(r["bytes"] for r in rows), sum(r["flops"] for r in rows), ms)
            trs = [r["traffic"] for r in rows]
            unit["traffic"] = sum(trs) if all(t is not None for t in trs) else None
        concurrent.append(unit)
    for c in ("router", "dispatch", "combine"):
        if c in call_launch_ms and call_launch_ms[c] > 0:
            gbs = alg[c] / (call_launch_ms[c] * 1e-3) / 1e9
            kernels[c].update({"launches_ms": round(call_launch_ms[c], 5), "launches_GB/s": round(gbs, 1),
                               "launches_frac_hbm": round(gbs / hbm, 4)})

    # the dominant unit: the longest grouped-GEMM launch that runs alone, or the longest group of GEMM
    # launches that run side by side (timed together)
    gemm_rows = [r for r in table if "bytes" in r and "group" not in r] + [u for u in concurrent if "bytes" in u]
    if gemm_rows:
        top = max(gemm_rows, key=lambda r: r["ms"])
        side_by_side = "kernels" in top
        top_ms, timing = top["ms"], ("the group's launches inside the step graph, from the first start to the "
                                     "last end" if side_by_side else "the launch inside the step graph") + \
            ", between event-record nodes added around each kernel node, L2 flushed before each step"
        if not side_by_side and live_ms and top.get("index") == top_index:
            top_ms = statistics.mean(live_ms)
            timing = ("this launch in every timed step, between two event-record nodes added around its kernel "
                      "node in the timed step graph (CUDA events on the launching stream); mean over the timed "
                      "steps")
            top = dict(against_bound(dict(top), top["bytes"], top["flops"], top_ms))
        if top["bound"] == "tensor":
            roof = {"bound": "tensor", "achieved": top["TFLOP/s"], "peak": tflops, "unit": "TFLOP/s",
                    "frac": round(top["TFLOP/s"] / tflops, 4),
                    "peak_kind": "sustained (kernel timed inside the step)" if tflops_sus > 0 else "burst"}
        else:
            roof = {"bound": "hbm", "achieved": top["GB/s"], "peak": hbm, "unit": "GB/s",
                    "frac": round(top["GB/s"] / hbm, 4)}
        roof.update({"traffic": top["traffic"],
                     "kernel": (f"{top['name']} (launched side by side on two streams, each on its share of the "
                                f"SMs)") if side_by_side else f"{top['kernel']} ({top['name']})",
                     "launch_ms": round(top_ms, 5), "algorithmic_bytes_per_launch": top["bytes"],
                     "algorithmic_flops_per_launch": top["flops"], "peak_source": peak_src, "timing": timing})
    else:   # per-launch replay unavailable: the forward grouped-GEMM call (two launches) from the per-call events
        gemm_gbs = alg["gemm"] / (mean_call["gemm"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gemm_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(gemm_gbs / hbm, 4), "traffic": None, "peak_source": peak_src,
                "kernel": "moe_expert_gemm (forward grouped GEMM call, 2 launches)",
                "algorithmic_bytes_per_call": alg["gemm"]}
    # the whole step against the HBM time of its algorithmic bytes
    step_bytes = alg["router"] + alg["dispatch"] + alg["gemm"] + alg["combine"] + (alg["backward"] if bwd else 0)
    step_floor_ms = step_bytes / (hbm * 1e9) * 1e3
    n_launch = len(launches) if launches else None
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "pass": args.pass_, "T": w.T, "d_model": w.d, "experts": w.E,
                   "top_k": w.k, "d_ff": w.F, "act": w.act, "renormalize": w.renormalize,
                   "capacity_factor": None if w.cf is None else f"{w.cf[0]}/{w.cf[1]}", "capacity": cap,
                   "capacity_reading": "floor(k*T*cf/E)" if w.cf is not None else "none (dropless)",
                   "aux_alpha": w.alpha, "kept_assignments": K_a, "experts_with_tokens": E_used,
                   "expert_weights": dv["weights"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed before every timed step (256 MiB write, outside the step's events)"},
        "roofline": roof,
        "step_roofline": {"algorithmic_bytes": step_bytes, "hbm_floor_ms": round(step_floor_ms, 4),
                          "frac": round(step_floor_ms / ms_step, 4), "peak": hbm, "unit": "GB/s"},
        "kernels": kernels,
        "launches": table if table else {"error": launch_error},
        "concurrent_launches": concurrent,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                "d2h_bytes_per_step": io_bytes, "call": "moe_forward" if not bwd else "separate calls + moe_backward",
                "overlap": "uploads and downloads on their own streams, double-buffered, overlapping compute"},
        "gpu_launches": n_launch * args.steps if n_launch else None,
        "gpu_launches_per_step": n_launch,
        "step_call": "moe_forward (one call: router, dispatch, expert GEMMs, combine fused into the second GEMM "
                     "for top-1)" if not bwd else
                     "moe_router, moe_dispatch, moe_expert_gemm, moe_combine, moe_backward",
        "timing": f"step replayed as one CUDA graph ({timed_how}); per-call figures from the separate ABI calls "
                  "with events between them, replayed as a CUDA graph (per_call_source); per-launch figures from "
                  "the step graph with every kernel node between two event-record nodes, replayed",
        "peaks": {"hbm_gbs": hbm, "bf16_tflops_used": tflops, "bf16_tflops_burst": tflops_burst,
                  "bf16_tflops_sustained": tflops_sus or None, "source": peak_src},
        "per_call_source": per_call_source,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall1 - t_wall0, 3),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, bwd)
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


HOST_F64_WEIGHTS_MAX = 8 << 30   # the oracle's fp64 copy of a sample's expert weights


def _f64_weight_bytes(w) -> int:
    return w.E * (w.R1 * w.d + w.d * w.F) * 8


def oracle_sample(w):
    """The workload the oracle is timed on, and how it stands for w.

    When the fp64 expert weights fit HOST_F64_WEIGHTS_MAX, w itself (a batch of its first tokens, chosen by
    time). Otherwise the same layer with fewer experts: E' = E / 2^j experts and T' = T E' / E tokens (its
    own seeded draws), so every expert's GEMM shape, the capacity, k and the rows per expert are w's, and
    the per-token work is w's (the router's E-dependent share aside)."""
    if _f64_weight_bytes(w) <= HOST_F64_WEIGHTS_MAX:
        return w, None
    E = w.E
    while E > 1 and _f64_weight_bytes(w.with_(E=E)) > HOST_F64_WEIGHTS_MAX:
        E //= 2
    T = max(1, w.T * E // w.E)
    ws = w.with_(name=f"{w.name}-T{T}-E{E}", T=T, E=E)
    return ws, (f"the same layer with {E} of the {w.E} experts and {T} of the {w.T} tokens (T E'/E; its own "
                f"seeded draws): every expert GEMM shape, k, the capacity ({_capacity(ws)}) and the rows per "
                "expert are the full layer's, so its tokens/s stands for the full layer's; the oracle runs it "
                "expert by expert through its callable expert source")


def _capacity(w):
    from oracle import moe_oracle as O
    return O.capacity(w.T, w.E, w.k, w.cf, w.count_assignments)


def _oracle_inputs(ws, bwd):
    inp = syn.make_inputs(ws, experts=False, dy=bwd)
    w1, w2 = syn.all_expert_weights(ws)
    weights = (w1.astype(np.float64), w2.astype(np.float64))
    del w1, w2
    return inp, weights


def _oracle_step(w, inp, Ts, weights, bwd):
    from oracle import moe_oracle as O
    kw = dict(k=w.k, act=w.act, cf=w.cf, count_assignments=w.count_assignments, renormalize=w.renormalize,
              alpha=w.alpha)
    x = inp["x"][:Ts]
    experts = lambda e: (weights[0][e], weights[1][e])    # one expert at a time, already fp64
    O.forward(x, inp["w_r"], inp["bias"], experts, **kw)
    if bwd:
        O.backward(x, inp["w_r"], inp["bias"], experts, inp["dy"][:Ts], **kw)


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


def _sample_text(ws, Ts, bwd, how):
    what = "forward + backward" if bwd else "forward"
    part = f"the full batch (T={ws.T})" if Ts == ws.T else f"the first {Ts} of the {ws.T} tokens as one batch " \
                                                           "(same capacity factor)"
    text = f"one {what} of {part} of {ws.name}, fp64 numpy oracle, expert weights widened to fp64 before timing"
    return text + (f"; {how}" if how else "")


def cpu_baseline(w, bwd):
    ws, how = oracle_sample(w)
    inp, weights = _oracle_inputs(ws, bwd)
    Ts = _oracle_batch(ws, inp, weights, bwd, 20.0)
    # the sampled batch, repeated until at least 10 s of CPU work have been timed
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(ws.with_(T=Ts), inp, Ts, weights, bwd)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0:
            break
    return {"value": round(Ts * reps / dt, 1), "unit": "tokens/s", "cores": _oracle_threads(), "kind": "oracle",
            "sample": _sample_text(ws, Ts, bwd, how) + f", {reps} time(s); {dt:.2f} s"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = bench_workload(args)
    bwd = args.pass_ == "fwdbwd"
    ws, how = oracle_sample(w)
    inp, weights = _oracle_inputs(ws, bwd)
    budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    Ts = _oracle_batch(ws, inp, weights, bwd, budget)
    wt = ws.with_(T=Ts)
    for _ in range(args.warmup):
        _oracle_step(wt, inp, Ts, weights, bwd)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(wt, inp, Ts, weights, bwd)
    dt = time.perf_counter() - t0
    value = Ts * args.steps / dt
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name, "pass": args.pass_, "sample_workload": ws.name, "T_sample": Ts},
           "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": _oracle_threads(),
                            "kind": "oracle", "sample": "each step: " + _sample_text(ws, Ts, bwd, how)},
           "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


BENCH_WORKLOADS = [n for n, w in syn.WORKLOADS.items() if w.dtype == "bf16"]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
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
