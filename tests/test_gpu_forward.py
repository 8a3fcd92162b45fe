"""GPU parity of the fused moe_forward against the fp64 oracle.

Small shapes are compared element by element over the whole output.  The
full-size workloads (Mixtral-shaped, fine-grained skewed, decode) run the
GPU exactly as the benchmark does and are compared on sampled tokens, which
the oracle evaluates one by one; routing and counts are compared in full.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import mixture_experts_ffn_permute_gb300 as moe
from mixture_experts_ffn_permute_gb300 import _build
from parity import assert_bf16_close, assert_equal, tile_sample_tokens

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.load()


def run_forward(shape, inp, ws=None, renorm=True, fusion=0, kernel=0):
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, renorm, shape.glu_interleave,
                         shape.swiglu_clamp, fusion, kernel)
    if ws is None:
        ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    out = torch.full((shape.T, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(shape.T, shape.k, dtype=torch.int32, device=DEV)
    w = torch.empty(shape.T, shape.k, dtype=torch.float32, device=DEV)
    tpe = torch.empty(shape.E, dtype=torch.int32, device=DEV)
    moe.forward(p, inp["x"], inp["logits"], inp["w1"], inp["w2"], out, ws, idx, w, tpe)
    status = moe.get_device_status(ws)
    assert status == 0, moe.STATUS_NAMES[status]
    return {"out": out, "topk_idx": idx, "topk_w": w, "tokens_per_expert": tpe, "ws": ws}


def to_dev(inp):
    return {k: v.to(DEV) for k, v in inp.items()}


SMALL = [
    mi.TINY,
    mi.MoEShape("ragged", T=333, H=512, F=384, E=7, k=3),
    mi.MoEShape("il32clamp", T=128, H=256, F=256, E=8, k=2, glu_interleave=32, swiglu_clamp=7.0),
    # gate/up blocks 64 and 128 rows apart (the weight loads' block gap)
    mi.MoEShape("il64", T=200, H=256, F=256, E=6, k=2, glu_interleave=64, swiglu_clamp=3.0),
    mi.MoEShape("il128", T=150, H=512, F=256, E=5, k=3, glu_interleave=128),
    mi.MoEShape("skew-small", T=512, H=256, F=256, E=64, k=8, zipf_s=1.1),
    mi.MoEShape("t1", T=1, H=256, F=128, E=8, k=2),
]


KERNELS = [moe.KERNEL_TOKEN_TILES, moe.KERNEL_WEIGHT_TILES, moe.KERNEL_WEIGHT_TILES_2CTA,
           moe.KERNEL_DECODE_FUSED]
KERNEL_IDS = ["token_tiles", "weight_tiles", "weight_tiles_2cta", "decode_fused"]


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_forward_small(shape, kernel):
    inp = mi.make_inputs(shape, seed=0)
    ref = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], shape.k,
                             interleave=shape.glu_interleave, clamp=shape.swiglu_clamp)
    res = run_forward(shape, to_dev(inp), kernel=kernel)
    assert_equal(res["topk_idx"], ref["topk_idx"], "topk_idx")
    assert_equal(res["tokens_per_expert"], ref["tokens_per_expert"], "tokens_per_expert")
    np.testing.assert_allclose(res["topk_w"].cpu().numpy(), ref["topk_w"], rtol=3e-6, atol=1e-7)
    assert_bf16_close(res["out"], ref["out"], f"out[{shape.name}]")


FUSION_SHAPES = [mi.TINY, mi.MoEShape("ragged", T=333, H=512, F=384, E=7, k=3),
                 mi.MoEShape("skew-small", T=512, H=256, F=256, E=64, k=8, zipf_s=1.1)]


@pytest.mark.parametrize("fusion", [moe.FUSE_GATHER_A, moe.FUSE_COMBINE,
                                    moe.FUSE_GATHER_A | moe.FUSE_COMBINE])
@pytest.mark.parametrize("shape", FUSION_SHAPES, ids=lambda s: s.name)
def test_forward_fusion_variants(shape, fusion):
    inp = mi.make_inputs(shape, seed=3)
    ref = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], shape.k)
    d = to_dev(inp)
    tok = moe.KERNEL_TOKEN_TILES  # the fusions belong to the 1-CTA token-row tiling
    res = run_forward(shape, d, fusion=fusion, kernel=tok)
    assert_bf16_close(res["out"], ref["out"], f"out[{shape.name}, fusion={fusion}]")
    if not fusion & moe.FUSE_COMBINE:
        # gathering A from x instead of a permuted copy changes no arithmetic
        base = run_forward(shape, d, fusion=0, kernel=tok)
        assert torch.equal(res["out"].view(torch.int16), base["out"].view(torch.int16))
    again = run_forward(shape, d, ws=res["ws"], fusion=fusion, kernel=tok)
    assert torch.equal(res["out"].view(torch.int16), again["out"].view(torch.int16))


# Around the limits of the single-block routing + permutation (+ gather) used
# by the smallest decode steps: T <= 32, E <= 256, T*k <= 256, gather in the
# same block for T*k <= 64.
TINY_EDGE = [mi.MoEShape("tiny-t1-k1", T=1, H=256, F=256, E=16, k=1),
             mi.MoEShape("tiny-gather-edge", T=16, H=256, F=256, E=24, k=4),   # 64 routes
             mi.MoEShape("tiny-t17", T=17, H=256, F=256, E=24, k=4),           # 68 routes
             mi.MoEShape("tiny-t31", T=31, H=256, F=256, E=32, k=8),
             mi.MoEShape("tiny-t32", T=32, H=256, F=256, E=40, k=8),           # 256 routes
             mi.MoEShape("tiny-t33", T=33, H=256, F=256, E=40, k=8),           # other path
             mi.MoEShape("tiny-e256", T=8, H=256, F=256, E=256, k=8),
             mi.MoEShape("tiny-e257", T=8, H=256, F=256, E=257, k=8)]          # other path


@pytest.mark.parametrize("shape", TINY_EDGE, ids=lambda s: s.name)
def test_forward_tiny_decode_edges(shape):
    inp = mi.make_inputs(shape, seed=5)
    ref = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], shape.k)
    res = run_forward(shape, to_dev(inp))
    assert_equal(res["topk_idx"], ref["topk_idx"], "topk_idx")
    assert_equal(res["tokens_per_expert"], ref["tokens_per_expert"], "tokens_per_expert")
    np.testing.assert_allclose(res["topk_w"].cpu().numpy(), ref["topk_w"], rtol=3e-6, atol=1e-7)
    assert_bf16_close(res["out"], ref["out"], f"out[{shape.name}]")


def test_forward_unnormalised_weights():
    shape = mi.TINY
    inp = mi.make_inputs(shape, seed=2)
    ref = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], shape.k,
                             renormalize=False)
    res = run_forward(shape, to_dev(inp), renorm=False)
    assert_bf16_close(res["out"], ref["out"], "out (full-softmax weights)")


@pytest.mark.parametrize("kernel", KERNELS, ids=KERNEL_IDS)
@pytest.mark.parametrize("T", [1, 8, 32])
def test_forward_decode_full_dims(T, kernel):
    shape = mi.DECODE.with_T(T)
    inp = mi.make_inputs(shape, seed=0)
    ref = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], shape.k)
    res = run_forward(shape, to_dev(inp), kernel=kernel)
    assert_equal(res["topk_idx"], ref["topk_idx"], "topk_idx")
    assert_bf16_close(res["out"], ref["out"], f"out[decode T={T}]")


def test_forward_is_bitwise_deterministic_and_reuses_workspace():
    shape = mi.MoEShape("det", T=300, H=512, F=256, E=16, k=4)
    a = to_dev(mi.make_inputs(shape, seed=0))
    b = dict(a)
    b["logits"] = mi.make_logits(shape, seed=99).to(DEV)
    r1 = run_forward(shape, a)
    ws = r1["ws"]
    r2 = run_forward(shape, b, ws=ws)      # different routing on the same workspace
    r3 = run_forward(shape, a, ws=ws)
    assert torch.equal(r1["out"].view(torch.int16), r3["out"].view(torch.int16))
    fresh = run_forward(shape, b)
    assert torch.equal(r2["out"].view(torch.int16), fresh["out"].view(torch.int16))
    assert moe.last_launch_count() >= 5


# One launch for GEMM1, GEMM2 and the combine (decode sizes): the same MMA
# shapes, K order and epilogue arithmetic as the two-GEMM 32-token weight
# tiles followed by the separate combine kernel, so the outputs agree bit for
# bit.  Shapes cover the single-block routing path, the one-block permutation
# (E > 256), experts with several 32-token tiles, empty experts, and (T*k >
# 4096) the multi-kernel permutation with the counters cleared by a memset.
DECODE_FUSED_SHAPES = [mi.DECODE.with_T(1), mi.DECODE.with_T(8), mi.DECODE.with_T(32),
                       mi.MoEShape("fused-e257", T=8, H=256, F=256, E=257, k=8),
                       mi.MoEShape("fused-ragged", T=333, H=512, F=384, E=7, k=3),
                       mi.MoEShape("fused-il32clamp", T=20, H=512, F=256, E=64, k=4,
                                   glu_interleave=32, swiglu_clamp=7.0),
                       mi.MoEShape("fused-multikernel-permute", T=1100, H=256, F=256, E=16, k=4),
                       mi.MoEShape("fused-il64", T=6, H=256, F=256, E=32, k=4, glu_interleave=64),
                       mi.MoEShape("fused-il128", T=6, H=512, F=256, E=32, k=4,
                                   glu_interleave=128, swiglu_clamp=7.0),
                       mi.MoEShape("fused-e1024", T=4, H=256, F=128, E=1024, k=8),
                       mi.MoEShape("fused-t1-k1", T=1, H=256, F=128, E=64, k=1)]


@pytest.mark.parametrize("shape", DECODE_FUSED_SHAPES, ids=lambda s: s.name)
def test_decode_fused_matches_two_gemm_path_bitwise(shape):
    d = to_dev(mi.make_inputs(shape, seed=11))
    fused = run_forward(shape, d, kernel=moe.KERNEL_DECODE_FUSED)
    n_fused = moe.last_launch_count()
    two = run_forward(shape, d, kernel=moe.KERNEL_WEIGHT_TILES)
    assert n_fused < moe.last_launch_count()
    assert torch.equal(fused["topk_idx"], two["topk_idx"])
    assert torch.equal(fused["out"].view(torch.int16), two["out"].view(torch.int16)), \
        f"decode-fused output differs from the two-GEMM path [{shape.name}]"
    # the same workspace again, after a call with other routing: the counters
    # the one-launch kernel depends on start from zero on every call
    other = dict(d)
    other["logits"] = mi.make_logits(shape, seed=12).to(DEV)
    run_forward(shape, other, ws=fused["ws"], kernel=moe.KERNEL_DECODE_FUSED)
    again = run_forward(shape, d, ws=fused["ws"], kernel=moe.KERNEL_DECODE_FUSED)
    assert torch.equal(fused["out"].view(torch.int16), again["out"].view(torch.int16))


# ------------------------------------------------------------------ full size, sampled

def sampled_check(shape, seed=0, kernel=0):
    """Full-size layer: routing and counts of every token bit-exact; outputs
    element-wise for the tokens tile_sample_tokens picks from the oracle's own
    permutation (first and last row of every expert, last row of every token
    tile), evaluated by the oracle on those tokens only."""
    inp = mi.make_inputs(shape, seed=seed, device=DEV)
    res = run_forward(shape, inp, kernel=kernel)
    logits_h = inp["logits"].cpu()
    # routing of every token and the expert histogram: bit-exact
    idx_ref, w_ref = oracle.route_topk(logits_h, shape.k)
    assert_equal(res["topk_idx"], idx_ref, "topk_idx")
    perm = oracle.permute(idx_ref, shape.E)
    assert_equal(res["tokens_per_expert"], perm["tokens_per_expert"], "tokens_per_expert")
    toks = tile_sample_tokens(perm)
    used = sorted(set(idx_ref[toks].ravel().tolist()))
    w1 = [None] * shape.E
    w2 = [None] * shape.E
    for e in used:
        w1[e] = inp["w1"][e].cpu()
        w2[e] = inp["w2"][e].cpu()
    ti = torch.from_numpy(toks).to(DEV)
    ref = oracle.moe_forward(inp["x"][ti].cpu(), logits_h[toks], w1, w2, shape.k,
                             interleave=shape.glu_interleave, clamp=shape.swiglu_clamp)
    assert_bf16_close(res["out"][ti], ref["out"], f"out[{shape.name}] {len(toks)} sampled tokens")
    out = res["out"]
    assert torch.isfinite(out.float()).all()
    return len(toks)


@pytest.mark.slow
def test_forward_mixtral_full_size_sampled():
    n = sampled_check(mi.MIXTRAL)
    assert n >= 32


@pytest.mark.slow
@pytest.mark.parametrize("kernel", [moe.KERNEL_AUTO, moe.KERNEL_TOKEN_TILES],
                         ids=["auto", "token_tiles"])
def test_forward_skewed_full_size_sampled(kernel):
    n = sampled_check(mi.SKEWED, kernel=kernel)
    assert n >= 256


@pytest.mark.slow
@pytest.mark.parametrize("T", [1, 8, 32, 128, 256])
def test_forward_decode_full_size_sampled(T):
    sampled_check(mi.DECODE.with_T(T))


# ---------------------------------------------------------------- caller-supplied routing

ROUTED_SHAPES = [mi.MoEShape("routed-ragged", T=333, H=512, F=384, E=7, k=3),
                 mi.MoEShape("routed-many", T=200, H=256, F=256, E=64, k=8, glu_interleave=64)]
ROUTED_KERNELS = [moe.KERNEL_AUTO, moe.KERNEL_TOKEN_TILES, moe.KERNEL_WEIGHT_TILES,
                  moe.KERNEL_WEIGHT_TILES_2CTA]
ROUTED_IDS = ["auto", "token_tiles", "weight_tiles", "weight_tiles_2cta"]


def run_routed(shape, d, idx, w, kernel=0):
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, True, shape.glu_interleave,
                         shape.swiglu_clamp, kernel=kernel)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    out = torch.full((shape.T, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    tpe = torch.empty(shape.E, dtype=torch.int32, device=DEV)
    moe.forward_routed(p, d["x"], idx.to(DEV), w.to(DEV), d["w1"], d["w2"], out, ws, tpe)
    return out, tpe, moe.get_device_status(ws)


@pytest.mark.parametrize("kernel", ROUTED_KERNELS, ids=ROUTED_IDS)
@pytest.mark.parametrize("shape", ROUTED_SHAPES, ids=lambda s: s.name)
def test_forward_routed_matches_oracle(shape, kernel):
    """Masked slots are skipped, a token with every slot masked gets a zero row,
    and the weights are used as given."""
    inp = mi.make_inputs(shape, seed=6)
    idx = mi.random_topk_idx(shape.T, shape.E, shape.k, seed=6, mask_frac=0.25)
    idx[3] = -1
    w = mi.random_weights(shape.T, shape.k, seed=6)
    ref = oracle.moe_forward_routed(inp["x"], idx, w, inp["w1"], inp["w2"],
                                    interleave=shape.glu_interleave)
    out, tpe, st = run_routed(shape, to_dev(inp), idx, w, kernel)
    assert st == 0, moe.STATUS_NAMES[st]
    assert_equal(tpe, ref["tokens_per_expert"], "tokens_per_expert")
    assert_bf16_close(out, ref["out"], f"out[{shape.name}]")
    assert not out[3].float().abs().sum().item()


def test_forward_routed_invalid_indices_are_masked():
    """An index outside [-1, E) or an expert repeated in a later slot is
    treated as masked and reported as MOE_ERR_DEVICE_INDEX."""
    shape = ROUTED_SHAPES[0]
    inp = mi.make_inputs(shape, seed=7)
    idx = mi.random_topk_idx(shape.T, shape.E, shape.k, seed=7)
    w = mi.random_weights(shape.T, shape.k, seed=7)
    idx[10, 1] = shape.E          # out of range
    idx[11, 0] = -5               # out of range
    idx[12, 2] = idx[12, 0]       # repeated: the later slot is dropped
    clean = idx.clone()
    clean[10, 1] = -1
    clean[11, 0] = -1
    clean[12, 2] = -1
    ref = oracle.moe_forward_routed(inp["x"], clean, w, inp["w1"], inp["w2"])
    out, tpe, st = run_routed(shape, to_dev(inp), idx, w)
    assert moe.STATUS_NAMES[st] == "MOE_ERR_DEVICE_INDEX"
    assert_equal(tpe, ref["tokens_per_expert"], "tokens_per_expert")
    assert_bf16_close(out, ref["out"], "out (invalid routes masked)")


# ---------------------------------------------------------------- shared experts

SHARED_CASES = [(mi.MoEShape("shared-tiny-path", T=4, H=256, F=256, E=16, k=4), 2),
                (mi.MoEShape("shared-small-permute", T=100, H=256, F=256, E=16, k=2), 1),
                (mi.MoEShape("shared-multikernel", T=700, H=512, F=256, E=12, k=6), 2)]


@pytest.mark.parametrize("kernel", [moe.KERNEL_AUTO, moe.KERNEL_TOKEN_TILES,
                                    moe.KERNEL_WEIGHT_TILES_2CTA, moe.KERNEL_DECODE_FUSED],
                         ids=["auto", "token_tiles", "weight_tiles_2cta", "decode_fused"])
@pytest.mark.parametrize("case", SHARED_CASES, ids=lambda c: c[0].name)
def test_forward_shared_experts(case, kernel):
    """S shared experts (the last S of w1/w2) join every token with weight 1."""
    shape, S = case
    full = mi.MoEShape(shape.name, T=shape.T, H=shape.H, F=shape.F, E=shape.E + S, k=shape.k)
    inp = mi.make_inputs(full, seed=8)
    logits = mi.make_logits(shape, seed=8)
    ref = oracle.moe_forward_shared(inp["x"], logits, inp["w1"], inp["w2"], shape.k, S)
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, kernel=kernel,
                         shared_experts=S)
    ws = moe.alloc_workspace(p)
    moe.clear_device_status(ws)
    slots = shape.k + S
    out = torch.full((shape.T, shape.H), float("nan"), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(shape.T, slots, dtype=torch.int32, device=DEV)
    w = torch.empty(shape.T, slots, dtype=torch.float32, device=DEV)
    tpe = torch.empty(shape.E + S, dtype=torch.int32, device=DEV)
    d = to_dev(inp)
    moe.forward(p, d["x"], logits.to(DEV), d["w1"], d["w2"], out, ws, idx, w, tpe)
    st = moe.get_device_status(ws)
    assert st == 0, moe.STATUS_NAMES[st]
    assert_equal(idx, ref["topk_idx"], "topk_idx (routed + shared slots)")
    assert_equal(tpe, ref["tokens_per_expert"], "tokens_per_expert")
    np.testing.assert_allclose(w.cpu().numpy(), ref["topk_w"], rtol=3e-6, atol=1e-7)
    assert_bf16_close(out, ref["out"], f"out[{shape.name}, S={S}]")
