"""bench.py's bookkeeping on the CPU: the algorithmic bytes and FLOPs its
roofline figures divide by, counted here element by element from the
workload shapes, and the kernel-launch counts it reports."""
import importlib.util
import os

import pytest

import moe_synth as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_switch_base_gemm_bytes_and_flops():
    b = _bench()
    w = syn.WORKLOADS["switch-base-top1"]          # T 8192, d 768, E 128, k 1, F 3072, ReLU
    K_a = 8088                                     # kept rows of the seeded batch (capacity 80)
    a = b.algorithmic(w, K_a, 128)
    weights = 2 * 128 * 3072 * 768 * 2             # W1 and W2 of every expert, bf16, read once
    x_in_y_out = 2 * K_a * 768 * 2                 # x_perm read, y_perm written
    h = 2 * K_a * 3072 * 2                         # h written by GEMM 1, read by GEMM 2
    assert a["gemm"] == weights + x_in_y_out + h == 1332191232
    assert a["gemm_flops"] == 2 * 2 * K_a * 768 * 3072 == 76327944192


def test_dropless_gemm_flops_and_dispatch_bytes():
    b = _bench()
    w = syn.WORKLOADS["dropless-top8-swiglu"]      # T 16384, d 2048, E 128, k 8, F 768, SwiGLU, no capacity
    K_a = 16384 * 8
    a = b.algorithmic(w, K_a, 128)
    assert a["gemm_flops"] == 3 * 2 * K_a * 2048 * 768 == 1236950581248
    x_read = 16384 * 2048 * 2
    rows_written = K_a * 2048 * 2
    routing = 16384 * 8 * 4 * 3 + K_a * 4         # idx, slot in/out; row owners
    assert a["dispatch"] == x_read + rows_written + routing == 606076928
    combine = 2 * 16384 * 2048 * 2 + K_a * 2048 * 2 + 16384 * 8 * 12   # x in, out, kept y rows, idx/gate/slot
    assert a["combine"] == combine
    assert a["backward_flops"] == 2 * a["gemm_flops"] + 4 * 16384 * 128 * 2048


def test_skewed_layer_counts_only_experts_that_keep_tokens():
    b = _bench()
    w = syn.WORKLOADS["gshard-top2-zipf"]
    all_experts = b.algorithmic(w, 9532, 64)["gemm"]
    used = b.algorithmic(w, 9532, 55)["gemm"]
    assert all_experts - used == 9 * 2 * 4096 * 1024 * 2    # the weights of the 9 empty experts


def test_grouped_gemm_launch_bytes_large_training():
    """Per-launch algorithmic bytes of the large training layer's six grouped-GEMM launches, element by element:
    together they are the forward call's and the backward GEMMs' bytes."""
    b = _bench()
    w = syn.WORKLOADS["large-top8-swiglu"]         # d 7168, F 2048, E 256, SwiGLU (R1 = 4096)
    K_a, E_used, d, F, R1, E = 32749, 256, 7168, 2048, 4096, 256
    g = {r: b.gemm_launch_algorithmic(r, w, K_a, E_used, True) for r in ("gemm1", "gemm2", "dH", "dW2", "dXp", "dW1")}
    assert g["gemm1"] == (E_used * R1 * d * 2 + K_a * d * 2 + K_a * F * 2 + K_a * 2 * F * 2, 2 * K_a * R1 * d)
    assert g["gemm2"] == (E_used * d * F * 2 + K_a * F * 2 + K_a * d * 2, 2 * K_a * d * F)
    assert g["dW1"] == (E * R1 * d * 2 + K_a * R1 * 2 + K_a * d * 2, 2 * K_a * R1 * d)
    assert g["dW2"] == (E * d * F * 2 + K_a * d * 2 + K_a * F * 2, 2 * K_a * d * F)
    assert g["dH"][0] == E_used * d * F * 2 + K_a * d * 2 + K_a * 2 * F * 2 + K_a * R1 * 2
    assert g["dXp"][0] == E_used * R1 * d * 2 + K_a * R1 * 2 + K_a * d * 2
    a = b.algorithmic(w, K_a, E_used)
    assert g["gemm1"][0] + g["gemm2"][0] == a["gemm"]           # the forward call's two launches
    assert g["gemm1"][1] + g["gemm2"][1] == a["gemm_flops"]
    assert sum(g[r][1] for r in ("dH", "dW2", "dXp", "dW1")) == a["bwd_gemm_flops"]


def test_kernel_roles_from_demangled_names():
    b = _bench()
    gemm = "void moe::tc::grouped_gemm_kernel<{}>(CUtensorMap_st, CUtensorMap_st, CUtensorMap_st, CUtensorMap_st, moe::tc::Args)"
    names = [
        "moe::(anonymous namespace)::router_split_kernel(float const*, int, int, int, __nv_bfloat16*)",
        "void moe::(anonymous namespace)::rt::router_tc_kernel<256>(CUtensorMap_st, CUtensorMap_st, moe::(anonymous namespace)::rt::Args)",
        "void moe::(anonymous namespace)::router_select_kernel<8>(float const*, int, moe::(anonymous namespace)::RouterArgs)",
        "void moe::(anonymous namespace)::dispatch_count_kernel<8>(int const*, int, int, int, long)",
        "void moe::(anonymous namespace)::dispatch_place_kernel<__nv_bfloat16, 8>(__nv_bfloat16 const*)",
        gemm.format("0, 0, 0, 0, 2"), gemm.format("0, 0, 0, 0, 0"),
        "void moe::(anonymous namespace)::combine_kernel<__nv_bfloat16, 8>(__nv_bfloat16 const*)",
        "void moe::(anonymous namespace)::combine_backward_kernel<__nv_bfloat16, 8>(__nv_bfloat16 const*)",
        gemm.format("0, 0, 0, 1, 4"), gemm.format("0, 1, 1, 1, 0"), gemm.format("0, 0, 0, 1, 0"),
        gemm.format("0, 1, 1, 1, 0"),
        "void moe::(anonymous namespace)::router_dh_kernel<8>(float const*)",
        "moe::(anonymous namespace)::router_wsplit6_kernel(float const*, int, int, int, __nv_bfloat16*)",
        gemm.format("0, 0, 0, 1, 5"), gemm.format("0, 1, 1, 1, 5"),
        "moe::(anonymous namespace)::router_dwr_sum_kernel(float const*, int, int, int, int, float*)",
        "void moe::(anonymous namespace)::unpermute_kernel<__nv_bfloat16, 8>(__nv_bfloat16 const*)",
    ]
    roles = b.kernel_roles(names)
    assert [r for r, _ in roles] == [
        "router_split_kernel", "router_tc_kernel", "router_select_kernel", "dispatch_count_kernel",
        "dispatch_place_kernel", "gemm1", "gemm2", "combine_kernel", "combine_backward_kernel", "dH", "dW2", "dXp",
        "dW1", "router_dh_kernel", "router_wsplit6_kernel", "router_grad_dX_r", "router_grad_dW_r",
        "router_dwr_sum_kernel", "unpermute_kernel"]
    assert [c for _, c in roles] == ["router"] * 3 + ["dispatch"] * 2 + ["gemm"] * 2 + ["combine"] + ["backward"] * 11
    assert b.kernel_roles([gemm.format("0, 0, 0, 0, 6")]) == [("gemm2_combine", "gemm")]
    wg = "moe::wg::wgrad_kernel(CUtensorMap_st, CUtensorMap_st, CUtensorMap_st, moe::wg::Args)"
    assert b.kernel_roles([gemm.format("0, 0, 0, 1, 4"), wg, gemm.format("0, 0, 0, 1, 0"), wg]) == [
        ("dH", "backward"), ("dW2", "backward"), ("dXp", "backward"), ("dW1", "backward")]


def test_oracle_sample_of_the_large_layer_keeps_every_per_expert_shape():
    b = _bench()
    w = syn.WORKLOADS["large-top8-swiglu"]
    ws, how = b.oracle_sample(w)
    assert how and ws.E == 16 and ws.T == 256 and (ws.d, ws.F, ws.k, ws.act, ws.cf) == (w.d, w.F, w.k, w.act, w.cf)
    assert b._capacity(ws) == b._capacity(w) == 160                  # C = floor(k T cf / E) is unchanged
    assert b._f64_weight_bytes(ws) <= b.HOST_F64_WEIGHTS_MAX
    small = syn.WORKLOADS["switch-base-top1"]
    assert b.oracle_sample(small) == (small, None)


def test_step_graph_order_and_side_by_side_groups():
    """The backward GEMMs on two streams: the main stream runs dH then dXp, the side stream dW2 then dW1 (after
    dH). Launch order follows the dependencies; dH with dW2 and dXp with dW1 form the side-by-side groups."""
    b = _bench()
    # creation order: cb (combine backward), dH, dW2, dXp, dW1, dh (router), unp
    deps = {"cb": [], "dH": ["cb"], "dW2": ["cb"], "dXp": ["dH"], "dW1": ["dW2", "dH"], "dh": ["dXp", "dW1"],
            "unp": ["dh"]}
    pos = {k: i for i, k in enumerate(deps)}
    order = b.topological_order(deps, pos)
    assert order == ["cb", "dH", "dW2", "dXp", "dW1", "dh", "unp"]
    anc = {}
    for k in order:
        anc[k] = set(deps[k]).union(*(anc[d] for d in deps[k])) if deps[k] else set()
    g = b.concurrent_groups(order, anc)
    assert g["dH"] == g["dW2"] and g["dXp"] == g["dW1"]
    assert len({g["cb"], g["dH"], g["dXp"], g["dh"], g["unp"]}) == 5
    # a chain: every node its own group
    chain = {"a": [], "b": ["a"], "c": ["b"]}
    o = b.topological_order(chain, {"a": 0, "b": 1, "c": 2})
    an = {"a": set(), "b": {"a"}, "c": {"a", "b"}}
    assert sorted(b.concurrent_groups(o, an).values()) == [0, 1, 2]
    with pytest.raises(RuntimeError):
        b.topological_order({"a": ["b"], "b": ["a"]}, {"a": 0, "b": 1})
