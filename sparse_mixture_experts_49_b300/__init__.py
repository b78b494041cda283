"""Sparsely-gated Mixture-of-Experts FFN layer on one B300: Python binding.

A thin ctypes layer over libmoe.so (declared in include/moe.h). Each function
has the C entry point's name and arguments; it checks and marshals torch
tensors (device pointers, sizes, the current CUDA stream) and nothing else:
every step of the layer runs in the library's CUDA kernels. If the library
is not built, the first call raises MoEError; there is no fallback.

`MoELayer` strings the calls together (router -> dispatch -> expert GEMMs ->
combine, and the backward pass) with buffers allocated through torch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_ALIGNMENT, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(6)
MOE_ACT_RELU, MOE_ACT_SWIGLU = 0, 1
MOE_F32, MOE_BF16 = 0, 1
MOE_SCORE_SOFTMAX, MOE_SCORE_SIGMOID, MOE_SCORE_SQRT_SOFTPLUS = 0, 1, 2
SCORES = {"softmax": MOE_SCORE_SOFTMAX, "sigmoid": MOE_SCORE_SIGMOID, "sqrt_softplus": MOE_SCORE_SQRT_SOFTPLUS}
MOE_DEVERR_NONE, MOE_DEVERR_BAD_EXPERT, MOE_DEVERR_DUP_EXPERT, MOE_DEVERR_TIMEOUT = range(4)
MOE_NOALLOC_MAX_TOKENS = 32768

EXPORTED = [
    "moe_capacity", "moe_max_rows", "moe_workspace_size", "moe_workspace_init", "moe_router",
    "moe_router_biased", "moe_select_bias_update", "moe_router_expert_choice", "moe_dispatch_expert_choice",
    "moe_combine_expert_choice", "moe_backward_expert_choice",
    "moe_dispatch", "moe_dispatch_noalloc", "moe_expert_gemm", "moe_combine", "moe_forward", "moe_backward",
    "moe_backward_intermediates",
    "moe_get_device_error", "moe_selftest_bounded_wait", "moe_status_string", "moe_last_cuda_error",
]


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("act", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("add_residual", ctypes.c_int32),
        ("score", ctypes.c_int32), ("capacity", ctypes.c_int64), ("aux_alpha", ctypes.c_float),
        ("reroute", ctypes.c_int32), ("expert_choice", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]


class moe_saved_expert_choice(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "x", "w_r", "w1", "w2", "probs", "row_token", "row_gate", "expert_offsets", "x_perm", "pre_act", "h",
        "y_perm")]


class moe_saved(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "x", "w_r", "w1", "w2", "probs", "topk_idx", "topk_gate", "slot", "expert_offsets", "load",
        "x_perm", "pre_act", "h", "y_perm")]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library (raises MoEError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoEError(MOE_ERR_CUDA, f"{LIB_PATH} is missing: build it with "
                                         "sparse_mixture_experts_49_b300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        C = ctypes.POINTER(moe_config)
        sig = {
            "moe_capacity": (I64, [I64, I32, I32, I32, I32, I32]),
            "moe_max_rows": (I64, [C]),
            "moe_workspace_size": (ctypes.c_int, [C, ctypes.POINTER(SZ)]),
            "moe_workspace_init": (ctypes.c_int, [C, P, P]),
            "moe_router": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P, P, P]),
            "moe_router_biased": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P, P, P, P]),
            "moe_select_bias_update": (ctypes.c_int, [C, P, P, ctypes.c_float, P]),
            "moe_router_expert_choice": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P, P]),
            "moe_dispatch_expert_choice": (ctypes.c_int, [C, P, P, P, P]),
            "moe_combine_expert_choice": (ctypes.c_int, [C, P, P, P, P, P, P, P]),
            "moe_backward_expert_choice": (ctypes.c_int, [C, ctypes.POINTER(moe_saved_expert_choice), P, P, P, P, P,
                                                          P, P]),
            "moe_dispatch": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P]),
            "moe_dispatch_noalloc": (ctypes.c_int, [C, P, P, P, P, P, P, P, P]),
            "moe_expert_gemm": (ctypes.c_int, [C, P, P, P, P, P, P, P, P, P]),
            "moe_combine": (ctypes.c_int, [C, P, P, P, P, P, P, P, P]),
            "moe_forward": (ctypes.c_int, [C] + [P] * 21),
            "moe_backward": (ctypes.c_int, [C, ctypes.POINTER(moe_saved), P, P, P, P, P, P, P]),
            "moe_backward_intermediates": (ctypes.c_int, [C, P, ctypes.POINTER(P), ctypes.POINTER(P),
                                                          ctypes.POINTER(P), ctypes.POINTER(P),
                                                          ctypes.POINTER(P)]),
            "moe_get_device_error": (ctypes.c_int, [P, P, ctypes.POINTER(I32)]),
            "moe_selftest_bounded_wait": (ctypes.c_int, [P, P]),
            "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "moe_last_cuda_error": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != MOE_OK:
        L = lib()
        msg = L.moe_status_string(status).decode()
        if status == MOE_ERR_CUDA:
            msg += ": " + L.moe_last_cuda_error().decode()
        raise MoEError(status, f"{what}: {msg}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise MoEError(MOE_ERR_INVALID_ARG, "tensors passed to the MoE library must be on the GPU")
    if not t.is_contiguous():
        raise MoEError(MOE_ERR_INVALID_ARG, "tensors passed to the MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def make_config(T: int, d_model: int, n_experts: int, top_k: int, d_ff: int, act: str = "relu",
                dtype: str = "bf16", renormalize: bool = False, capacity: int = -1,
                aux_alpha: float = 0.01, add_residual: bool = True, score: str = "softmax",
                reroute: bool = False, expert_choice: bool = False) -> moe_config:
    return moe_config(T=T, d_model=d_model, n_experts=n_experts, top_k=top_k, d_ff=d_ff,
                      act=MOE_ACT_SWIGLU if act == "swiglu" else MOE_ACT_RELU,
                      dtype=MOE_BF16 if dtype == "bf16" else MOE_F32, renormalize=int(renormalize),
                      add_residual=int(add_residual), score=SCORES[score],
                      capacity=-1 if capacity is None else int(capacity), aux_alpha=float(aux_alpha),
                      reroute=int(reroute), expert_choice=int(expert_choice), reserved=0)


# ---------------------------------------------------------------- entry points (same names as the C ABI)
def moe_capacity(T: int, E: int, k: int, cf_num: int, cf_den: int, count_assignments: bool = True) -> int:
    return lib().moe_capacity(T, E, k, cf_num, cf_den, int(count_assignments))


def moe_max_rows(cfg: moe_config) -> int:
    r = lib().moe_max_rows(ctypes.byref(cfg))
    if r < 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_max_rows: invalid config")
    return r


def moe_workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_workspace_init(cfg, ws, stream=None):
    _check(lib().moe_workspace_init(ctypes.byref(cfg), _ptr(ws), _stream(stream)), "moe_workspace_init")


def moe_router(cfg, x, w_r, logit_bias, probs, topk_idx, topk_gate, importance, load, aux_loss, ws, stream=None):
    _check(lib().moe_router(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_bias), _ptr(probs), _ptr(topk_idx),
                            _ptr(topk_gate), _ptr(importance), _ptr(load), _ptr(aux_loss), _ptr(ws),
                            _stream(stream)), "moe_router")


def moe_router_biased(cfg, x, w_r, logit_bias, select_bias, probs, topk_idx, topk_gate, importance, load, aux_loss,
                      ws, stream=None):
    """moe_router with a selection-only correction bias (the experts are chosen on score + bias; the gates are
    the scores)."""
    _check(lib().moe_router_biased(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_bias), _ptr(select_bias),
                                   _ptr(probs), _ptr(topk_idx), _ptr(topk_gate), _ptr(importance), _ptr(load),
                                   _ptr(aux_loss), _ptr(ws), _stream(stream)), "moe_router_biased")


def moe_select_bias_update(cfg, load, select_bias, gamma: float, stream=None):
    """select_bias[e] += gamma * sign(mean(load) - load[e]), in place."""
    _check(lib().moe_select_bias_update(ctypes.byref(cfg), _ptr(load), _ptr(select_bias), float(gamma),
                                        _stream(stream)), "moe_select_bias_update")


def moe_router_expert_choice(cfg, x, w_r, logit_bias, probs, row_token, row_gate, expert_offsets, importance, ws,
                             stream=None):
    """Expert-choice routing: each expert takes the min(C, T) tokens with the largest softmax scores."""
    _check(lib().moe_router_expert_choice(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_bias), _ptr(probs),
                                          _ptr(row_token), _ptr(row_gate), _ptr(expert_offsets), _ptr(importance),
                                          _ptr(ws), _stream(stream)), "moe_router_expert_choice")


def moe_dispatch_expert_choice(cfg, x, row_token, x_perm, stream=None):
    _check(lib().moe_dispatch_expert_choice(ctypes.byref(cfg), _ptr(x), _ptr(row_token), _ptr(x_perm),
                                            _stream(stream)), "moe_dispatch_expert_choice")


def moe_combine_expert_choice(cfg, x, y_perm, row_token, row_gate, out, ws, stream=None):
    _check(lib().moe_combine_expert_choice(ctypes.byref(cfg), _ptr(x), _ptr(y_perm), _ptr(row_token), _ptr(row_gate),
                                           _ptr(out), _ptr(ws), _stream(stream)), "moe_combine_expert_choice")


def moe_backward_expert_choice(cfg, saved: dict, dy, dx, dw_r, dw1, dw2, ws, stream=None):
    sv = moe_saved_expert_choice(**{k: _ptr(saved.get(k)) for k, _ in moe_saved_expert_choice._fields_})
    _check(lib().moe_backward_expert_choice(ctypes.byref(cfg), ctypes.byref(sv), _ptr(dy), _ptr(dx), _ptr(dw_r),
                                            _ptr(dw1), _ptr(dw2), _ptr(ws), _stream(stream)),
           "moe_backward_expert_choice")


def moe_dispatch(cfg, x, topk_idx, slot, kept, expert_offsets, row_token, x_perm, ws, stream=None):
    _check(lib().moe_dispatch(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(slot), _ptr(kept),
                              _ptr(expert_offsets), _ptr(row_token), _ptr(x_perm), _ptr(ws), _stream(stream)),
           "moe_dispatch")


def moe_dispatch_noalloc(cfg, x, topk_idx, slot, kept, expert_offsets, row_token, x_perm, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate device memory at all: the
    scratch is a fixed array inside the library (T <= MOE_NOALLOC_MAX_TOKENS; calls that overlap on
    the GPU race; bad expert indices are dropped but not reported)."""
    _check(lib().moe_dispatch_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(slot), _ptr(kept),
                                      _ptr(expert_offsets), _ptr(row_token), _ptr(x_perm), _stream(stream)),
           "moe_dispatch_noalloc")


def moe_expert_gemm(cfg, x_perm, expert_offsets, w1, w2, pre_act, h, y_perm, ws, stream=None):
    _check(lib().moe_expert_gemm(ctypes.byref(cfg), _ptr(x_perm), _ptr(expert_offsets), _ptr(w1), _ptr(w2),
                                 _ptr(pre_act), _ptr(h), _ptr(y_perm), _ptr(ws), _stream(stream)),
           "moe_expert_gemm")


def moe_combine(cfg, x, y_perm, topk_idx, topk_gate, slot, expert_offsets, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(x), _ptr(y_perm), _ptr(topk_idx), _ptr(topk_gate),
                             _ptr(slot), _ptr(expert_offsets), _ptr(out), _stream(stream)), "moe_combine")


def moe_forward(cfg, x, w_r, logit_bias, w1, w2, probs, topk_idx, topk_gate, importance, load, aux_loss, slot, kept,
                expert_offsets, row_token, x_perm, h, y_perm, out, ws, stream=None):
    """The whole forward layer in one call (inference; top-1 layers combine inside the second expert GEMM)."""
    _check(lib().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_r), _ptr(logit_bias), _ptr(w1), _ptr(w2), _ptr(probs),
                             _ptr(topk_idx), _ptr(topk_gate), _ptr(importance), _ptr(load), _ptr(aux_loss), _ptr(slot),
                             _ptr(kept), _ptr(expert_offsets), _ptr(row_token), _ptr(x_perm), _ptr(h), _ptr(y_perm),
                             _ptr(out), _ptr(ws), _stream(stream)), "moe_forward")


def moe_backward(cfg, saved: dict, dy, dx, dw_r, dw1, dw2, ws, stream=None):
    sv = moe_saved(**{k: _ptr(saved.get(k)) for k, _ in moe_saved._fields_})
    _check(lib().moe_backward(ctypes.byref(cfg), ctypes.byref(sv), _ptr(dy), _ptr(dx), _ptr(dw_r), _ptr(dw1),
                              _ptr(dw2), _ptr(ws), _stream(stream)), "moe_backward")


def moe_backward_intermediates(cfg, ws) -> dict:
    ps = [ctypes.c_void_p() for _ in range(5)]
    _check(lib().moe_backward_intermediates(ctypes.byref(cfg), _ptr(ws), *[ctypes.byref(p) for p in ps]),
           "moe_backward_intermediates")
    return dict(zip(["dyp", "da", "dxp", "dg", "dh"], [p.value for p in ps]))


def moe_get_device_error(ws, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().moe_get_device_error(_ptr(ws), _stream(stream), ctypes.byref(code)), "moe_get_device_error")
    return code.value


def moe_selftest_bounded_wait(ws, stream=None) -> None:
    """Runs the kernels' bounded on-chip wait on a barrier nothing completes; the wait gives up after its
    limit (about 4 s) and records MOE_DEVERR_TIMEOUT in the workspace's error word (read it with
    moe_get_device_error)."""
    _check(lib().moe_selftest_bounded_wait(_ptr(ws), _stream(stream)), "moe_selftest_bounded_wait")


# ---------------------------------------------------------------- logging figures
def _host(a):
    """A torch tensor (any device) or array-like as a float64 numpy array."""
    import numpy as np
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.float64)


def balance_stats(importance, load, kept, T: int, k: int, alpha: float = 0.01) -> dict:
    """Load-balance figures of one routed batch, for logging, from the router's per-expert importance
    (sum over tokens of the routing probability) and load (top-k assignments), and the dispatch's kept counts:

    - drop_rate = 1 - sum(kept) / (T k), the share of assignments over capacity;
    - max_over_mean_load = max(load) / mean(load);
    - cv2_importance, cv2_load: squared coefficients of variation (population variance / mean^2);
    - aux = alpha E sum_e f_e P_e with f_e = load_e / (T k) and P_e = importance_e / T, the
      load-balancing loss the router also returns ("Mixture of Experts (MoE) を1から解説 — Switch
      Transformerのルーティングと負荷分散", eq. (4))."""
    imp, ld, kp = _host(importance), _host(load), _host(kept)
    E = ld.shape[0]
    mean_ld = ld.mean()
    f = ld / (T * k)
    P = imp / T
    return {
        "drop_rate": 1.0 - kp.sum() / (T * k),
        "max_over_mean_load": float(ld.max() / mean_ld) if mean_ld > 0 else 0.0,
        "cv2_importance": float(imp.var() / imp.mean() ** 2) if imp.mean() > 0 else 0.0,
        "cv2_load": float(ld.var() / mean_ld ** 2) if mean_ld > 0 else 0.0,
        "aux": float(alpha * E * (f * P).sum()),
    }


# ---------------------------------------------------------------- convenience wrapper
class MoELayer:
    """Buffers for one layer shape, and the forward/backward call sequences."""

    def __init__(self, cfg: moe_config, device="cuda", stream=None):
        import torch
        self.cfg = cfg
        self.stream = stream
        self.dt = torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32
        T, d, E, k, F = cfg.T, cfg.d_model, cfg.n_experts, cfg.top_k, cfg.d_ff
        if cfg.reroute:
            k = 2   # columns: first choice, second candidate
        R1 = 2 * F if cfg.act == MOE_ACT_SWIGLU else F
        self.rows = moe_max_rows(cfg)
        dev = torch.device(device)
        z = lambda *s, dtype=self.dt: torch.empty(*s, dtype=dtype, device=dev)
        self.ws = torch.zeros(moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
        self.probs = z(T, E, dtype=torch.float32)
        self.topk_idx = z(T, k, dtype=torch.int32)
        self.topk_gate = z(T, k, dtype=torch.float32)
        self.importance = z(E, dtype=torch.float32)
        self.load = z(E, dtype=torch.int32)
        self.aux = z(1, dtype=torch.float32)
        self.slot = z(T, k, dtype=torch.int32)
        self.kept = z(E, dtype=torch.int32)
        self.offsets = z(E + 1, dtype=torch.int32)
        self.row_token = z(max(self.rows, 1), dtype=torch.int32)
        self.x_perm = z(max(self.rows, 1), d)
        self.pre_act = z(max(self.rows, 1), 2 * F) if cfg.act == MOE_ACT_SWIGLU else None
        self.h = z(max(self.rows, 1), F)
        self.y_perm = z(max(self.rows, 1), d)
        self.out = z(T, d)
        self.row_gate = z(max(self.rows, 1), dtype=torch.float32) if cfg.expert_choice else None
        self.R1 = R1
        moe_workspace_init(cfg, self.ws, stream)

    def forward(self, x, w_r, w1, w2, logit_bias=None, topk_idx=None, select_bias=None):
        """out = x + MoE(x) (MoE(x) alone without the residual). If topk_idx is given, the router's choice is
        replaced by it (replay); select_bias is the selection-only correction bias (moe_router_biased)."""
        c, s = self.cfg, self.stream
        if c.expert_choice:
            # expert-choice routing: the experts pick their tokens (groups of min(C, T) rows each)
            moe_router_expert_choice(c, x, w_r, logit_bias, self.probs, self.row_token, self.row_gate, self.offsets,
                                     self.importance, self.ws, s)
            moe_dispatch_expert_choice(c, x, self.row_token, self.x_perm, s)
            moe_expert_gemm(c, self.x_perm, self.offsets, w1, w2, self.pre_act, self.h, self.y_perm, self.ws, s)
            moe_combine_expert_choice(c, x, self.y_perm, self.row_token, self.row_gate, self.out, self.ws, s)
            self._saved = dict(x=x, w_r=w_r, w1=w1, w2=w2, probs=self.probs, row_token=self.row_token,
                               row_gate=self.row_gate, expert_offsets=self.offsets, x_perm=self.x_perm,
                               pre_act=self.pre_act, h=self.h, y_perm=self.y_perm)
            return self.out
        if select_bias is None:
            moe_router(c, x, w_r, logit_bias, self.probs, self.topk_idx, self.topk_gate, self.importance,
                       self.load, self.aux, self.ws, s)
        else:
            moe_router_biased(c, x, w_r, logit_bias, select_bias, self.probs, self.topk_idx, self.topk_gate,
                              self.importance, self.load, self.aux, self.ws, s)
        idx = self.topk_idx if topk_idx is None else topk_idx
        moe_dispatch(c, x, idx, self.slot, self.kept, self.offsets, self.row_token, self.x_perm, self.ws, s)
        moe_expert_gemm(c, self.x_perm, self.offsets, w1, w2, self.pre_act, self.h, self.y_perm, self.ws, s)
        moe_combine(c, x, self.y_perm, idx, self.topk_gate, self.slot, self.offsets, self.out, s)
        self._saved = dict(x=x, w_r=w_r, w1=w1, w2=w2, probs=self.probs, topk_idx=idx, topk_gate=self.topk_gate,
                           slot=self.slot, expert_offsets=self.offsets, load=self.load, x_perm=self.x_perm,
                           pre_act=self.pre_act, h=self.h, y_perm=self.y_perm)
        return self.out

    def infer(self, x, w_r, w1, w2, logit_bias=None):
        """out = x + MoE(x) through moe_forward (one call; nothing kept for the backward pass)."""
        c = self.cfg
        moe_forward(c, x, w_r, logit_bias, w1, w2, self.probs, self.topk_idx, self.topk_gate, self.importance,
                    self.load, self.aux, self.slot, self.kept, self.offsets, self.row_token, self.x_perm, self.h,
                    self.y_perm if (c.top_k > 1 or c.reroute) else None, self.out, self.ws, self.stream)
        return self.out

    def backward(self, dy, dx=None, dw_r=None, dw1=None, dw2=None):
        import torch
        c = self.cfg
        dev = dy.device
        dx = dx if dx is not None else torch.empty_like(dy)
        dw_r = dw_r if dw_r is not None else torch.empty(c.n_experts, c.d_model, dtype=torch.float32, device=dev)
        dw1 = dw1 if dw1 is not None else torch.empty(c.n_experts, self.R1, c.d_model, dtype=self.dt, device=dev)
        dw2 = dw2 if dw2 is not None else torch.empty(c.n_experts, c.d_model, c.d_ff, dtype=self.dt, device=dev)
        if c.expert_choice:
            moe_backward_expert_choice(c, self._saved, dy, dx, dw_r, dw1, dw2, self.ws, self.stream)
        else:
            moe_backward(c, self._saved, dy, dx, dw_r, dw1, dw2, self.ws, self.stream)
        return dx, dw_r, dw1, dw2

    def balance_stats(self) -> dict:
        """balance_stats() of the last routed batch (synchronises the device first)."""
        import torch
        torch.cuda.synchronize()
        c = self.cfg
        return balance_stats(self.importance, self.load, self.kept, c.T, c.top_k, c.aux_alpha)

    def device_error(self) -> int:
        return moe_get_device_error(self.ws, self.stream)
