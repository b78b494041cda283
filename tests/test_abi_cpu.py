"""The C-ABI library without a GPU: it loads, exports what include/moe.h
declares, sizes its workspace, and rejects bad arguments on the host before
any launch."""
import ctypes
import os
import re

import pytest

import sparse_mixture_experts_49_b300 as moe
from oracle import moe_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from sparse_mixture_experts_49_b300 import build
    build.build()


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = header_functions()
    assert len(names) >= 13
    L = moe.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(moe.EXPORTED)


def test_capacity_matches_oracle_reading():
    for T, E, k, cf in [(512, 8, 1, (1, 1)), (8192, 128, 1, (5, 4)), (16384, 64, 2, (2, 1)),
                        (4096, 256, 8, (5, 4)), (1000, 7, 3, (3, 2)), (1, 256, 8, (1, 1))]:
        for count in (True, False):
            assert moe.moe_capacity(T, E, k, cf[0], cf[1], count) == O.capacity(T, E, k, cf, count)
    assert moe.moe_capacity(10, 0, 1, 1, 1) == -1
    assert moe.moe_capacity(10, 4, 1, 1, 0) == -1


def cfg(**kw):
    base = dict(T=1000, d_model=256, n_experts=16, top_k=2, d_ff=512, act="relu", dtype="bf16", capacity=250)
    base.update(kw)
    return moe.make_config(**base)


def test_rows_and_workspace_size():
    c = cfg()
    assert moe.moe_max_rows(c) == min(1000 * 2, 16 * 250)
    assert moe.moe_max_rows(cfg(capacity=-1)) == 2000
    assert moe.moe_max_rows(cfg(capacity=10)) == 160
    assert moe.moe_workspace_size(c) > 2000 * 256 * 2
    assert moe.moe_workspace_size(cfg(act="swiglu")) > moe.moe_workspace_size(c)


@pytest.mark.parametrize("kw,status", [
    (dict(top_k=17), moe.MOE_ERR_INVALID_ARG),          # k > E
    (dict(n_experts=300, top_k=2), moe.MOE_ERR_UNSUPPORTED),
    (dict(top_k=9, n_experts=16), moe.MOE_ERR_UNSUPPORTED),
    (dict(d_model=204), moe.MOE_ERR_ALIGNMENT),          # bf16 needs multiples of 8 (16-byte rows)
    (dict(d_ff=100), moe.MOE_ERR_ALIGNMENT),
    (dict(dtype="f32", d_model=66), moe.MOE_ERR_ALIGNMENT),
    (dict(T=0), moe.MOE_ERR_INVALID_ARG),
])
def test_config_validation(kw, status):
    with pytest.raises(moe.MoEError) as e:
        moe.moe_workspace_size(cfg(**kw))
    assert e.value.status == status


def test_bf16_sizes_multiple_of_8_are_accepted():
    for d, F in [(136, 200), (8, 8), (4104, 1000)]:
        assert moe.moe_workspace_size(cfg(d_model=d, d_ff=F)) > 0
        assert moe.moe_workspace_size(cfg(d_model=d, d_ff=F, act="swiglu")) > 0


def test_config_bad_fields():
    c = cfg()
    c.act = 7
    with pytest.raises(moe.MoEError):
        moe.moe_workspace_size(c)
    for field, bad in (("add_residual", 2), ("score", 3), ("renormalize", -1)):
        c = cfg()
        setattr(c, field, bad)
        with pytest.raises(moe.MoEError) as e:
            moe.moe_workspace_size(c)
        assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as e:                     # router variants: bf16 layers only
        moe.moe_workspace_size(cfg(dtype="f32", score="sigmoid"))
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    c = cfg()
    c.reroute = 2
    with pytest.raises(moe.MoEError):
        moe.moe_workspace_size(c)
    with pytest.raises(moe.MoEError) as e:                     # rerouting: top-1 layers only
        moe.moe_workspace_size(cfg(reroute=True))               # (top_k 2)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
    rr = cfg(top_k=1, reroute=True)
    assert moe.moe_max_rows(rr) == min(1000, 16 * 250)          # at most one kept assignment per token
    c = cfg()
    c.aux_alpha = float("nan")
    with pytest.raises(moe.MoEError):
        moe.moe_workspace_size(c)


def test_null_and_misaligned_pointers_rejected_before_launch():
    L = moe.lib()
    c = cfg()
    P = 1 << 20                   # fake, 16-byte aligned addresses: never dereferenced on these paths
    null = None
    # a required pointer missing -> invalid argument
    st = L.moe_router(ctypes.byref(c), null, P, null, null, P, P, P, P, null, P, null)
    assert st == moe.MOE_ERR_INVALID_ARG
    # a misaligned pointer -> alignment error
    st = L.moe_dispatch(ctypes.byref(c), P + 4, P, P, P, P, P, P, P, null)
    assert st == moe.MOE_ERR_ALIGNMENT
    # ReLU takes no pre-activation buffer
    st = L.moe_expert_gemm(ctypes.byref(c), P, P, P, P, P, P, P, P, null)
    assert st == moe.MOE_ERR_INVALID_ARG
    # combine output may not alias its inputs
    st = L.moe_combine(ctypes.byref(c), P, P + 256, P, P, P, P, P, null)
    assert st == moe.MOE_ERR_INVALID_ARG
    # backward without the saved state
    st = L.moe_backward(ctypes.byref(c), None, P, P, P, P, P, P, null)
    assert st == moe.MOE_ERR_INVALID_ARG
    # SwiGLU backward needs the saved pre-activations
    s = moe.moe_saved(**{n: P for n, _ in moe.moe_saved._fields_})
    s.pre_act = None
    st = L.moe_backward(ctypes.byref(cfg(act="swiglu")), ctypes.byref(s), P, P, P, P, P, P, null)
    assert st == moe.MOE_ERR_INVALID_ARG
    # the bounded-wait self-test needs a workspace
    assert L.moe_selftest_bounded_wait(null, null) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_bounded_wait(P + 4, null) == moe.MOE_ERR_ALIGNMENT


def test_forward_call_validation():
    L = moe.lib()
    P = 1 << 20
    null = None

    def fwd(c, **over):
        a = dict(x=P, w_r=P, bias=null, w1=P, w2=P, probs=null, idx=P, gate=P, imp=P, load=P, aux=null, slot=P,
                 kept=P, offsets=P, row_token=P, x_perm=P, h=P, y_perm=P, out=P + 4096, ws=P)
        a.update(over)
        return L.moe_forward(ctypes.byref(c), *a.values(), null)

    assert fwd(cfg(dtype="f32", d_model=64, d_ff=128)) == moe.MOE_ERR_UNSUPPORTED   # bf16 only
    assert fwd(cfg(), y_perm=null) == moe.MOE_ERR_INVALID_ARG      # top-2 combines through y_perm
    assert fwd(cfg(), out=P) == moe.MOE_ERR_INVALID_ARG            # out may not alias x
    assert fwd(cfg(), h=P + 8) == moe.MOE_ERR_ALIGNMENT
    assert fwd(cfg(), row_token=null) == moe.MOE_ERR_INVALID_ARG
    assert fwd(cfg(), x_perm=null) == moe.MOE_ERR_INVALID_ARG


def test_status_strings():
    L = moe.lib()
    for s in range(6):
        assert L.moe_status_string(s)
    assert L.moe_status_string(99) == b"unknown status"


def test_backward_intermediates_are_inside_the_workspace():
    c = cfg(act="swiglu")
    base = 1 << 24
    out = moe.moe_backward_intermediates(c, base)
    size = moe.moe_workspace_size(c)
    for v in out.values():
        assert base <= v < base + size and v % 256 == 0
