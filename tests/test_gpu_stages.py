"""GPU parity of each C-ABI stage against the fp64 oracle on seeded inputs.

Sizes are small enough for the oracle to finish in seconds but span several
tiles (128 rows x 256 columns, K steps of 64) and ragged tails.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import mixture_experts_ffn_permute_gb300 as moe
from mixture_experts_ffn_permute_gb300 import _build
from parity import assert_bf16_close, assert_equal

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.load()


def _empty(*shape, dtype):
    return torch.empty(*shape, dtype=dtype, device=DEV)


# ------------------------------------------------------------------ routing

ROUTE_CASES = [
    (mi.TINY, True), (mi.TINY, False), (mi.MIXTRAL, True), (mi.SKEWED, True),
    (mi.DECODE, True), (mi.DECODE.with_T(1), True),
    (mi.MoEShape("e33", T=77, H=256, F=128, E=33, k=5), True),
    (mi.MoEShape("emax", T=40, H=256, F=128, E=1024, k=32), True),
    (mi.MoEShape("emax0", T=40, H=256, F=128, E=1024, k=32), False),
    (mi.MoEShape("e1", T=10, H=256, F=128, E=1, k=1), True),
]


@pytest.mark.parametrize("shape,renorm", ROUTE_CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_route_topk(shape, renorm):
    logits = mi.make_logits(shape, seed=3)
    idx_ref, w_ref = oracle.route_topk(logits, shape.k, renorm)
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, renorm)
    idx = _empty(shape.T, shape.k, dtype=torch.int32)
    w = _empty(shape.T, shape.k, dtype=torch.float32)
    moe.route_topk(p, logits.to(DEV), idx, w)
    torch.cuda.synchronize()
    assert_equal(idx, idx_ref, "topk_idx")
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=3e-6, atol=1e-7)


def test_route_topk_ties():
    g = torch.Generator().manual_seed(5)
    logits = torch.randint(-2, 3, (500, 64), generator=g).to(torch.float32)
    logits[::7] = 0.0
    logits[1::7] = -0.0
    idx_ref, w_ref = oracle.route_topk(logits, 8)
    p = moe.Problem.make(500, 256, 128, 64, 8)
    idx = _empty(500, 8, dtype=torch.int32)
    w = _empty(500, 8, dtype=torch.float32)
    moe.route_topk(p, logits.to(DEV), idx, w)
    torch.cuda.synchronize()
    assert_equal(idx, idx_ref, "topk_idx with ties")
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=3e-6, atol=1e-7)


# ------------------------------------------------------------------ permute

PERMUTE_CASES = [(64, 8, 2, 0.0, 256), (1, 8, 2, 0.0, 256), (65, 8, 2, 0.0, 256),
                 (1000, 33, 5, 0.0, 512), (700, 256, 8, 0.0, 256), (300, 16, 4, 0.3, 256),
                 (129, 1, 1, 0.0, 256), (50, 1024, 32, 0.1, 256), (8192, 256, 8, 0.0, 256)]


@pytest.mark.parametrize("T,E,k,mask,H", PERMUTE_CASES)
def test_permute(T, E, k, mask, H):
    idx = mi.random_topk_idx(T, E, k, seed=T + E + k, mask_frac=mask)
    x = mi.make_x(mi.MoEShape("x", T=T, H=H, F=128, E=E, k=k), seed=2)
    ref = oracle.permute(idx, E)
    ref_xp = oracle.gather_rows(x, ref["permuted_token"])
    p = moe.Problem.make(T, H, 128, E, k)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    R = T * k
    out = dict(row_id_map=_empty(T, k, dtype=torch.int32),
               permuted_token=torch.full((R,), 12345, dtype=torch.int32, device=DEV),
               tokens_per_expert=_empty(E, dtype=torch.int32),
               expert_offsets=_empty(E + 1, dtype=torch.int32))
    xp = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.permute(p, idx.to(DEV), x.to(DEV), xp, out["row_id_map"], out["permuted_token"],
                out["tokens_per_expert"], out["expert_offsets"], ws)
    assert moe.get_device_status(ws) == 0
    for key in ("row_id_map", "permuted_token", "tokens_per_expert", "expert_offsets"):
        assert_equal(out[key], ref[key], key)
    assert_equal(xp.view(torch.int16).cpu().numpy().view(np.uint16), ref_xp, "x_perm")


def test_permute_flags_bad_indices_without_faulting():
    T, E, k = 100, 8, 2
    idx = mi.random_topk_idx(T, E, k, seed=1)
    idx[3, 1] = 999
    idx[7, 0] = -5
    idx[9, 1] = idx[9, 0]  # duplicate expert in one token
    p = moe.Problem.make(T, 256, 128, E, k)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    rmap = _empty(T, k, dtype=torch.int32)
    ptok = _empty(T * k, dtype=torch.int32)
    tpe = _empty(E, dtype=torch.int32)
    off = _empty(E + 1, dtype=torch.int32)
    moe.permute(p, idx.to(DEV), None, None, rmap, ptok, tpe, off, ws)
    assert moe.get_device_status(ws) == 7  # MOE_ERR_DEVICE_INDEX
    # the bad routes were treated as masked: the rest matches the oracle
    clean = idx.clone()
    clean[3, 1] = -1
    clean[7, 0] = -1
    clean[9, 1] = -1
    ref = oracle.permute(clean, E)
    assert_equal(rmap, ref["row_id_map"], "row_id_map")
    assert_equal(tpe, ref["tokens_per_expert"], "tokens_per_expert")
    moe.clear_device_status(ws)
    assert moe.get_device_status(ws) == 0


# ------------------------------------------------------------------ grouped MLP

MLP_CASES = [
    mi.TINY,
    mi.MoEShape("ragged", T=300, H=512, F=384, E=5, k=2),
    mi.MoEShape("il32", T=200, H=256, F=256, E=4, k=2, glu_interleave=32, swiglu_clamp=7.0),
    mi.MoEShape("il64", T=150, H=256, F=384, E=3, k=2, glu_interleave=64),
    mi.MoEShape("il128", T=90, H=256, F=512, E=3, k=2, glu_interleave=128, swiglu_clamp=0.5),
    mi.MoEShape("sparse", T=20, H=256, F=128, E=16, k=1),
    mi.MoEShape("onexp", T=260, H=768, F=256, E=1, k=1),
]


def _routed_inputs(shape, seed=0, mask=0.0):
    inp = mi.make_inputs(shape, seed=seed)
    idx, w = oracle.route_topk(inp["logits"], shape.k)
    if mask > 0:
        g = np.random.default_rng(seed)
        idx = idx.copy()
        idx[g.random(idx.shape) < mask] = -1
    perm = oracle.permute(idx, shape.E)
    xp = oracle.gather_rows(inp["x"], perm["permuted_token"])
    return inp, idx, w, perm, xp


KERNELS = [moe.KERNEL_TOKEN_TILES, moe.KERNEL_WEIGHT_TILES, moe.KERNEL_WEIGHT_TILES_2CTA]


@pytest.mark.parametrize("kernel", KERNELS, ids=["token_tiles", "weight_tiles", "weight_tiles_2cta"])
@pytest.mark.parametrize("shape", MLP_CASES, ids=lambda s: s.name)
def test_grouped_swiglu_mlp(shape, kernel):
    inp, idx, w, perm, xp = _routed_inputs(shape, seed=1)
    h = oracle.gemm1_swiglu(xp, perm["expert_offsets"], inp["w1"], shape.F, shape.glu_interleave,
                            shape.swiglu_clamp)
    y_ref = oracle.gemm2(h, perm["expert_offsets"], inp["w2"], shape.H)
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, True, shape.glu_interleave,
                         shape.swiglu_clamp, kernel=kernel)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    R = shape.R
    y = torch.full((R, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    xp_d = torch.from_numpy(xp.view(np.int16)).view(torch.bfloat16).to(DEV)
    moe.grouped_swiglu_mlp(p, xp_d, torch.from_numpy(perm["expert_offsets"]).to(DEV),
                           inp["w1"].to(DEV), inp["w2"].to(DEV), y, ws)
    assert moe.get_device_status(ws) == 0
    assert_bf16_close(y, y_ref, f"y_perm[{shape.name}]")


@pytest.mark.parametrize("kernel", KERNELS, ids=["token_tiles", "weight_tiles", "weight_tiles_2cta"])
def test_grouped_mlp_masked_tail_rows_are_zero(kernel):
    shape = mi.MoEShape("masked", T=100, H=256, F=256, E=6, k=2)
    inp, idx, w, perm, xp = _routed_inputs(shape, seed=4, mask=0.25)
    n = int(perm["expert_offsets"][-1])
    assert n < shape.R
    h = oracle.gemm1_swiglu(xp, perm["expert_offsets"], inp["w1"], shape.F)
    y_ref = oracle.gemm2(h, perm["expert_offsets"], inp["w2"], shape.H)
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, kernel=kernel)
    ws = moe.alloc_workspace(p)
    y = torch.full((shape.R, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.grouped_swiglu_mlp(p, torch.from_numpy(xp.view(np.int16)).view(torch.bfloat16).to(DEV),
                           torch.from_numpy(perm["expert_offsets"]).to(DEV), inp["w1"].to(DEV),
                           inp["w2"].to(DEV), y, ws)
    torch.cuda.synchronize()
    assert_bf16_close(y, y_ref, "y_perm with masked tail")
    assert (y[n:] == 0).all()


def test_grouped_mlp_rejects_bad_offsets_on_device():
    shape = mi.MoEShape("bad", T=64, H=256, F=128, E=4, k=2)
    inp = mi.make_inputs(shape)
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    off = torch.tensor([0, 50, 40, 100, 128], dtype=torch.int32, device=DEV)  # decreasing
    y = torch.full((shape.R, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    xp = torch.zeros(shape.R, shape.H, dtype=torch.bfloat16, device=DEV)
    moe.grouped_swiglu_mlp(p, xp, off, inp["w1"].to(DEV), inp["w2"].to(DEV), y, ws)
    assert moe.get_device_status(ws) == 7


# ------------------------------------------------------------------ combine

@pytest.mark.parametrize("T,H,E,k,mask", [(64, 256, 8, 2, 0.0), (333, 768, 16, 8, 0.2),
                                          (5, 2048, 4, 4, 0.5), (1, 256, 1, 1, 0.0)])
def test_unpermute_combine(T, H, E, k, mask):
    idx = mi.random_topk_idx(T, E, k, seed=T, mask_frac=mask)
    perm = oracle.permute(idx, E)
    w = mi.random_weights(T, k, seed=T)
    R = T * k
    y = torch.randn(R, H, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16)
    ref = oracle.unpermute_combine(y.to(torch.float64).numpy(), perm["row_id_map"],
                                   w.to(torch.float64).numpy())
    p = moe.Problem.make(T, H, 128, E, k)
    out = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    moe.unpermute_combine(p, y.to(DEV), torch.from_numpy(perm["row_id_map"]).to(DEV), w.to(DEV),
                          out)
    torch.cuda.synchronize()
    assert_bf16_close(out, ref, "combine")
    # one rounding of an fp32 sum: within one bf16 ulp of the fp64 value
    g = out.to(torch.float64).cpu().numpy()
    assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30 + 1e-6)


def test_permute_then_unpermute_is_identity_on_gpu():
    T, E, k, H = 257, 8, 2, 512
    logits = mi.make_logits(mi.MoEShape("i", T=T, H=H, F=128, E=E, k=k), seed=8)
    x = mi.make_x(mi.MoEShape("i", T=T, H=H, F=128, E=E, k=k), seed=8).to(DEV)
    p = moe.Problem.make(T, H, 128, E, k)
    ws = moe.alloc_workspace(p)
    idx = _empty(T, k, dtype=torch.int32)
    wt = _empty(T, k, dtype=torch.float32)
    moe.route_topk(p, logits.to(DEV), idx, wt, ws)
    rmap = _empty(T, k, dtype=torch.int32)
    ptok = _empty(T * k, dtype=torch.int32)
    tpe = _empty(E, dtype=torch.int32)
    off = _empty(E + 1, dtype=torch.int32)
    xp = _empty(T * k, H, dtype=torch.bfloat16)
    moe.permute(p, idx, x, xp, rmap, ptok, tpe, off, ws)
    half = torch.full((T, k), 0.5, dtype=torch.float32, device=DEV)
    out = _empty(T, H, dtype=torch.bfloat16)
    moe.unpermute_combine(p, xp, rmap, half, out)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), x.view(torch.int16))
