"""moe_permute_noalloc, the permute for callers that cannot allocate device
memory (for instance while a stream is being captured into a CUDA graph),
checked against moe_permute with a caller workspace.

The no-allocation variant keeps its scratch in one fixed device array that
all calls share, so this file runs last and calls it twice in a row with
different routing: the second call must not see anything the first left.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import mixture_experts_ffn_permute_gb300 as moe
from mixture_experts_ffn_permute_gb300 import _build

pytestmark = pytest.mark.gpu

DEV = "cuda"
KEYS = ("row_id_map", "permuted_token", "tokens_per_expert", "expert_offsets")


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.load()


def _outputs(T, E, k, H):
    R = T * k
    return {"row_id_map": torch.full((T, k), -7, dtype=torch.int32, device=DEV),
            "permuted_token": torch.full((R,), -7, dtype=torch.int32, device=DEV),
            "tokens_per_expert": torch.full((E,), -7, dtype=torch.int32, device=DEV),
            "expert_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
            "x_perm": torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=DEV)}


def _with_workspace(p, idx, x):
    o = _outputs(p.T, p.E, p.k, p.H)
    ws = moe.alloc_workspace(p)
    moe.permute(p, idx, x, o["x_perm"], o["row_id_map"], o["permuted_token"],
                o["tokens_per_expert"], o["expert_offsets"], ws)
    return o


def _without_workspace(p, idx, x):
    o = _outputs(p.T, p.E, p.k, p.H)
    moe.permute_noalloc(p, idx, x, o["x_perm"], o["row_id_map"], o["permuted_token"],
                        o["tokens_per_expert"], o["expert_offsets"])
    return o


def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    cases = [(1000, 64, 8, 0.1, 512, 1), (333, 16, 4, 0.0, 256, 2)]
    for T, E, k, mask, H, seed in cases:
        idx = mi.random_topk_idx(T, E, k, seed=seed, mask_frac=mask).to(DEV)
        x = mi.make_x(mi.MoEShape("x", T=T, H=H, F=128, E=E, k=k), seed=seed).to(DEV)
        p = moe.Problem.make(T, H, 128, E, k)
        want = _with_workspace(p, idx, x)
        # a one-launch call in between, so the count below is the no-alloc call's
        moe.unpermute_combine(p, want["x_perm"], want["row_id_map"],
                              torch.ones(T, k, dtype=torch.float32, device=DEV),
                              torch.empty(T, H, dtype=torch.bfloat16, device=DEV))
        assert moe.last_launch_count() == 1
        got = _without_workspace(p, idx, x)
        # histogram, scan, scatter and the row gather
        assert moe.last_launch_count() == 4
        torch.cuda.synchronize()
        for key in KEYS:  # integer outputs: bit for bit
            assert torch.equal(got[key], want[key]), (T, key)
        assert torch.equal(got["x_perm"].view(torch.int16), want["x_perm"].view(torch.int16))


def test_noalloc_permute_rejects_problems_beyond_its_scratch():
    # ceil(T/64) * E + E + 1 > 2**18 int32 entries
    p = moe.Problem.make(70000, 256, 128, 1024, 2)
    dummy = torch.empty(16, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoEError) as err:
        moe.permute_noalloc(p, dummy, None, None, dummy, dummy, dummy, dummy)
    assert err.value.status == 4  # MOE_ERR_WORKSPACE_TOO_SMALL
