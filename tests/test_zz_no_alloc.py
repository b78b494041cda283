"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device
memory at all (no workspace to pass), against the workspace-based
moe_dispatch on the same inputs.

The entry point keeps its scratch in a fixed array inside the library,
shared by every call, so it is checked on two calls in a row whose routings
differ: the second call must not see anything the first one left behind.
Dispatch is integer and copy work, so the comparison is bit for bit.
This file is collected last on purpose.
"""
import numpy as np
import pytest

import moe_synth as syn
import sparse_mixture_experts_49_b300 as moe
from moe_cases import config_for

FAKE = 1 << 20   # a 16-byte-aligned address that is never dereferenced


def test_rejects_more_tokens_than_the_fixed_scratch_holds():
    c = moe.make_config(T=moe.MOE_NOALLOC_MAX_TOKENS + 1, d_model=256, n_experts=16, top_k=2, d_ff=512)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_dispatch_noalloc(c, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, stream=0)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_dispatch_matches_workspace_dispatch_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [
        syn.Workload("noalloc-a", T=3000, d=256, E=32, k=2, F=256, act="relu", dtype="bf16", cf=(5, 4)),
        syn.Workload("noalloc-b", T=1100, d=320, E=16, k=4, F=256, act="relu", dtype="bf16", cf=(1, 1)),
        # the fixed array's exact bound: T = MOE_NOALLOC_MAX_TOKENS tokens over 256 experts
        syn.Workload("noalloc-max", T=moe.MOE_NOALLOC_MAX_TOKENS, d=128, E=256, k=2, F=256, act="relu",
                     dtype="bf16", cf=(5, 4)),
    ]
    for w in cases:
        cfg = config_for(moe, w)
        rng = np.random.default_rng(w.T)
        x = torch.from_numpy(syn.round_bf16(rng.standard_normal((w.T, w.d)).astype(np.float32))).cuda()
        x = x.to(torch.bfloat16)
        idx = np.stack([rng.permutation(w.E)[:w.k] for _ in range(w.T)]).astype(np.int32)
        idx_t = torch.from_numpy(idx).cuda()
        rows = moe.moe_max_rows(cfg)

        def outputs():
            return dict(slot=torch.full((w.T, w.k), -7, dtype=torch.int32, device="cuda"),
                        kept=torch.full((w.E,), -7, dtype=torch.int32, device="cuda"),
                        offsets=torch.full((w.E + 1,), -7, dtype=torch.int32, device="cuda"),
                        row_token=torch.full((rows,), -7, dtype=torch.int32, device="cuda"),
                        x_perm=torch.zeros(rows, w.d, dtype=torch.bfloat16, device="cuda"))

        ref = outputs()
        ws = torch.zeros(moe.moe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
        moe.moe_workspace_init(cfg, ws)
        moe.moe_dispatch(cfg, x, idx_t, ref["slot"], ref["kept"], ref["offsets"], ref["row_token"], ref["x_perm"],
                         ws)
        got = outputs()
        moe.moe_dispatch_noalloc(cfg, x, idx_t, got["slot"], got["kept"], got["offsets"], got["row_token"],
                                 got["x_perm"])
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
        n = int(ref["offsets"][-1].item())
        for key in ("slot", "kept", "offsets"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["row_token"][:n], ref["row_token"][:n])
        assert torch.equal(got["x_perm"][:n], ref["x_perm"][:n])
        assert (ref["slot"] >= 0).sum().item() == n > 0
