"""bench.py's bookkeeping on the CPU: the algorithmic bytes and FLOPs its
roofline figures divide by, counted here element by element from the
workload shapes, and the kernel-launch counts it reports."""
import importlib.util
import os

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


def test_launch_counts():
    b = _bench()
    top1 = syn.WORKLOADS["switch-base-top1"]
    top8 = syn.WORKLOADS["dropless-top8-swiglu"]
    # router 3 (split, logits, selection), dispatch 2, grouped GEMM 2, combine 1 unless fused into GEMM 2 (top-1)
    assert b.forward_launches(top1, True) == 7
    assert b.forward_launches(top1, False) == 8
    assert b.forward_launches(top8, True) == 8
    assert b.LAUNCHES_BACKWARD == 11
