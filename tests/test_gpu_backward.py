"""GPU parity of the layer's backward (moe_backward through the C ABI) against
the fp64 oracle's gradients: dx, d_logits, dW1 and dW2.

Small shapes are compared element by element; they span several m-tiles,
n-tiles and K steps with ragged tails (F not a multiple of 256, expert row
counts not multiples of 64 or 128), empty experts, GLU interleave, the
SwiGLU clamp, both router weightings and shared experts.  The full-size
Mixtral-shaped and skewed layers run exactly as the benchmark runs them and
are compared on sampled token rows, dW1 rows and dW2 columns, each of which
the oracle evaluates on its own.  The oracle takes the clamp decisions on the
pre-activations rounded to fp32, the precision in which the backward keeps
them, and supplies for every element the magnitude of its terms that the
tolerance scales with (parity.assert_grad_bound).
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
import mixture_experts_ffn_permute_gb300 as moe
from mixture_experts_ffn_permute_gb300 import _build
from parity import assert_grad_bound

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    moe.load()


def run_backward(shape, inp, g, renorm=True, S=0, kernel=0):
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, renorm,
                         shape.glu_interleave, shape.swiglu_clamp, 0, kernel, shared_experts=S)
    ws = moe.alloc_backward_workspace(p)
    moe.clear_device_status(ws)
    nan = float("nan")
    dx = torch.full((shape.T, shape.H), nan, dtype=torch.bfloat16, device=DEV)
    dl = torch.full((shape.T, shape.E), nan, dtype=torch.float32, device=DEV)
    dw1 = torch.full_like(inp["w1"], nan)
    dw2 = torch.full_like(inp["w2"], nan)
    moe.backward(p, inp["x"], inp["logits"], inp["w1"], inp["w2"], g, dx, dw1, dw2, ws,
                 d_logits=dl)
    torch.cuda.synchronize()
    assert moe.get_device_status(ws) == moe.MOE_OK
    return {"dx": dx, "dlogits": dl, "dw1": dw1, "dw2": dw2, "ws": ws}


def small_inputs(shape, S=0, seed=0):
    full = mi.MoEShape(shape.name, T=shape.T, H=shape.H, F=shape.F, E=shape.E + S, k=shape.k)
    inp = mi.make_inputs(full, seed=seed)
    logits = mi.make_logits(shape, seed=seed)  # the routed experts' logits only
    return {"x": inp["x"], "logits": logits, "w1": inp["w1"], "w2": inp["w2"]}, \
        mi.make_grad_out(shape, seed=seed)


def check_small(shape, renorm=True, S=0, kernel=0, seed=0):
    inp, g = small_inputs(shape, S, seed)
    kw = dict(renormalize=renorm, interleave=shape.glu_interleave, clamp=shape.swiglu_clamp,
              shared_experts=S, mask_f32=True)
    ref = oracle.moe_backward(inp["x"], inp["logits"], inp["w1"], inp["w2"], g, shape.k, **kw)
    mag = oracle.moe_backward(inp["x"], inp["logits"], inp["w1"], inp["w2"], g, shape.k,
                              magnitude=True, **kw)
    res = run_backward(shape, {k: v.to(DEV) for k, v in inp.items()}, g.to(DEV), renorm, S,
                       kernel)
    tag = f"[{shape.name} renorm={renorm} S={S} kernel={kernel}]"
    for name in ("dx", "dw1", "dw2", "dlogits"):
        assert_grad_bound(res[name], ref[name], mag[name], name + tag)
    return res, ref


SMALL = [
    mi.TINY,
    mi.MoEShape("ragged", T=200, H=256, F=384, E=6, k=2, glu_interleave=32, swiglu_clamp=0.9),
    mi.MoEShape("il64", T=150, H=512, F=256, E=5, k=3, glu_interleave=64, swiglu_clamp=1.2),
    mi.MoEShape("il128", T=90, H=256, F=256, E=4, k=2, glu_interleave=128),
    mi.MoEShape("deep", T=700, H=256, F=256, E=2, k=1),
    # >= 512 rows per expert on average: the 4-stage weight-gradient variant
    mi.MoEShape("long", T=1100, H=256, F=384, E=2, k=1, glu_interleave=64, swiglu_clamp=1.0),
    mi.MoEShape("skew", T=160, H=256, F=256, E=16, k=2, zipf_s=1.5),
    mi.MoEShape("one", T=1, H=256, F=256, E=8, k=2),
]


@pytest.mark.parametrize("shape", SMALL, ids=[s.name for s in SMALL])
def test_backward_small(shape):
    check_small(shape)


def test_backward_ignores_the_forward_tiling_choice():
    shape = mi.MoEShape("tilings", T=96, H=256, F=384, E=4, k=2, glu_interleave=32,
                        swiglu_clamp=1.0)
    a, _ = check_small(shape)
    inp, g = small_inputs(shape)
    b = run_backward(shape, {k: v.to(DEV) for k, v in inp.items()}, g.to(DEV),
                     kernel=moe.KERNEL_WEIGHT_TILES_2CTA)
    for name in ("dx", "dw1", "dw2"):
        assert torch.equal(a[name].view(torch.int16), b[name].view(torch.int16)), name


def test_backward_full_softmax_weights():
    check_small(mi.MoEShape("full", T=120, H=256, F=256, E=8, k=3, swiglu_clamp=1.1),
                renorm=False)


@pytest.mark.parametrize("S", [1, 2])
def test_backward_shared_experts(S):
    check_small(mi.MoEShape("shared", T=80, H=256, F=256, E=6, k=2, glu_interleave=32), S=S)


def test_backward_empty_experts_get_exact_zero_gradients():
    shape = mi.MoEShape("empty", T=40, H=256, F=256, E=8, k=1)
    inp, g = small_inputs(shape)
    inp["logits"][:, 5] = -1e4  # expert 5 is never selected
    res = run_backward(shape, {k: v.to(DEV) for k, v in inp.items()}, g.to(DEV))
    assert torch.count_nonzero(res["dw1"][5]) == 0 and torch.count_nonzero(res["dw2"][5]) == 0
    assert torch.count_nonzero(res["dw1"][:5]) > 0


def test_backward_no_tokens_zeroes_the_weight_gradients():
    shape = mi.MoEShape("none", T=0, H=256, F=256, E=3, k=1)
    inp, g = small_inputs(mi.MoEShape("none", T=4, H=256, F=256, E=3, k=1))
    inp = {k: v.to(DEV) for k, v in inp.items()}
    p = moe.Problem.make(0, 256, 256, 3, 1)
    ws = moe.alloc_backward_workspace(moe.Problem.make(4, 256, 256, 3, 1))
    dw1 = torch.full_like(inp["w1"], float("nan"))
    dw2 = torch.full_like(inp["w2"], float("nan"))
    moe.backward(p, inp["x"][:0], inp["logits"][:0], inp["w1"], inp["w2"], g[:0].to(DEV),
                 inp["x"][:0], dw1, dw2, ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw1) == 0 and torch.count_nonzero(dw2) == 0


def test_backward_is_bitwise_deterministic():
    shape = mi.MoEShape("det", T=300, H=256, F=384, E=8, k=2, glu_interleave=32, swiglu_clamp=1.0)
    inp, g = small_inputs(shape)
    inp = {k: v.to(DEV) for k, v in inp.items()}
    a = run_backward(shape, inp, g.to(DEV))
    b = run_backward(shape, inp, g.to(DEV))
    for name in ("dx", "dw1", "dw2"):
        assert torch.equal(a[name].view(torch.int16), b[name].view(torch.int16)), name
    assert torch.equal(a["dlogits"], b["dlogits"])


# ------------------------------------------------------------------ full size, sampled

def sampled_backward(shape, n_tok=6, n_rows=6, seed=0):
    inp = mi.make_inputs(shape, seed=seed, device=DEV)
    g = mi.make_grad_out(shape, seed=seed, device=DEV)
    res = run_backward(shape, inp, g)
    logits_h = inp["logits"].cpu()
    idx, w = oracle.route_topk(logits_h, shape.k)
    x_h, g_h = inp["x"].cpu(), g.cpu()
    rng = np.random.default_rng(7)
    toks = np.sort(rng.choice(shape.T, size=n_tok, replace=False))
    counts = np.bincount(idx.ravel(), minlength=shape.E)
    busy = np.argsort(-counts, kind="stable")
    # W1 rows and W2 columns of the busiest expert, a median one and a light one
    light = busy[-1] if counts[busy[-1]] else busy[0]
    experts = [int(busy[0]), int(busy[shape.E // 2]), int(light)]
    used = sorted(set(idx[toks].ravel().tolist()) | set(experts))
    w1 = [None] * shape.E
    w2 = [None] * shape.E
    for e in used:
        w1[e] = inp["w1"][e].cpu()
        w2[e] = inp["w2"][e].cpu()
    kw = dict(interleave=shape.glu_interleave, clamp=shape.swiglu_clamp, mask_f32=True)
    dx_ref, dw_ref = oracle.backward_tokens(x_h, idx, w, w1, w2, g_h, toks, **kw)
    dx_mag, dw_mag = oracle.backward_tokens(x_h, idx, w, w1, w2, g_h, toks, magnitude=True,
                                            **kw)
    ti = torch.from_numpy(toks).to(DEV)
    assert_grad_bound(res["dx"][ti], dx_ref, dx_mag, f"dx[{shape.name}] sampled")
    dl_ref = oracle.router_backward(logits_h[toks], idx[toks], w[toks], dw_ref, shape.k)
    dl_mag = oracle.router_backward(logits_h[toks], idx[toks], w[toks], dw_mag, shape.k,
                                    magnitude=True)
    assert_grad_bound(res["dlogits"][ti], dl_ref, dl_mag, f"dlogits[{shape.name}] sampled")
    rows = rng.choice(2 * shape.F, size=n_rows, replace=False)
    pairs = [(experts[i % 3], int(r)) for i, r in enumerate(rows)]
    ref1 = oracle.backward_dw1_rows(x_h, idx, w, w1, w2, g_h, pairs, **kw)
    mag1 = oracle.backward_dw1_rows(x_h, idx, w, w1, w2, g_h, pairs, magnitude=True, **kw)
    got1 = torch.stack([res["dw1"][e, r] for e, r in pairs])
    assert_grad_bound(got1, ref1, mag1, f"dw1[{shape.name}] sampled rows")
    cols = rng.choice(shape.F, size=n_rows, replace=False)
    pairs = [(experts[i % 3], int(f)) for i, f in enumerate(cols)]
    ref2 = oracle.backward_dw2_cols(x_h, idx, w, w1, w2, g_h, pairs, **kw)
    mag2 = oracle.backward_dw2_cols(x_h, idx, w, w1, w2, g_h, pairs, magnitude=True, **kw)
    got2 = torch.stack([res["dw2"][e, :, f] for e, f in pairs])
    assert_grad_bound(got2, ref2, mag2, f"dw2[{shape.name}] sampled cols")


def test_backward_mixtral_full_size_sampled():
    sampled_backward(mi.MIXTRAL)


def test_backward_skewed_full_size_sampled():
    sampled_backward(mi.SKEWED, n_tok=4)


# ------------------------------------------------------------------ caller-supplied routing

def run_backward_routed(shape, inp, idx, w, g):
    p = moe.Problem.make(shape.T, shape.H, shape.F, shape.E, shape.k, True,
                         shape.glu_interleave, shape.swiglu_clamp)
    ws = moe.alloc_backward_workspace(p)
    moe.clear_device_status(ws)
    nan = float("nan")
    dx = torch.full((shape.T, shape.H), nan, dtype=torch.bfloat16, device=DEV)
    dtw = torch.full((shape.T, shape.k), nan, dtype=torch.float32, device=DEV)
    dw1 = torch.full_like(inp["w1"], nan)
    dw2 = torch.full_like(inp["w2"], nan)
    moe.backward_routed(p, inp["x"], idx.to(DEV), w.to(DEV), inp["w1"], inp["w2"], g, dx, dw1,
                        dw2, ws, d_topk_w=dtw)
    torch.cuda.synchronize()
    return {"dx": dx, "dw_route": dtw, "dw1": dw1, "dw2": dw2}, moe.get_device_status(ws)


ROUTED = [mi.MoEShape("routed", T=150, H=256, F=384, E=7, k=3, glu_interleave=32,
                      swiglu_clamp=1.0),
          mi.MoEShape("routed-big", T=900, H=512, F=256, E=4, k=2)]


@pytest.mark.parametrize("shape", ROUTED, ids=[s.name for s in ROUTED])
def test_backward_routed_matches_oracle(shape):
    """Masked slots contribute nothing and get a zero weight gradient; a token
    with every slot masked gets a zero dx row; the weights are used as given."""
    inp, g = small_inputs(shape, seed=9)
    idx = mi.random_topk_idx(shape.T, shape.E, shape.k, seed=9, mask_frac=0.25)
    idx[5] = -1
    w = mi.random_weights(shape.T, shape.k, seed=9)
    kw = dict(interleave=shape.glu_interleave, clamp=shape.swiglu_clamp, mask_f32=True)
    ref = oracle.expert_backward(inp["x"], idx, w, inp["w1"], inp["w2"], g, **kw)
    mag = oracle.expert_backward(inp["x"], idx, w, inp["w1"], inp["w2"], g, magnitude=True, **kw)
    res, st = run_backward_routed(shape, {k: v.to(DEV) for k, v in inp.items()}, idx, w,
                                  g.to(DEV))
    assert st == moe.MOE_OK, moe.STATUS_NAMES[st]
    for name in ("dx", "dw1", "dw2", "dw_route"):
        assert_grad_bound(res[name], ref[name], mag[name], f"{name}[{shape.name}]")
    assert (res["dw_route"].cpu()[idx < 0] == 0).all()
    assert not res["dx"][5].float().abs().sum().item()


def test_backward_routed_invalid_indices_are_masked():
    shape = ROUTED[0]
    inp, g = small_inputs(shape, seed=4)
    idx = mi.random_topk_idx(shape.T, shape.E, shape.k, seed=4)
    w = mi.random_weights(shape.T, shape.k, seed=4)
    idx[10, 1] = shape.E          # out of range
    idx[11, 0] = -5               # out of range
    idx[12, 2] = idx[12, 0]       # repeated: the later slot is dropped
    clean = idx.clone()
    clean[10, 1] = -1
    clean[11, 0] = -1
    clean[12, 2] = -1
    kw = dict(interleave=shape.glu_interleave, clamp=shape.swiglu_clamp, mask_f32=True)
    ref = oracle.expert_backward(inp["x"], clean, w, inp["w1"], inp["w2"], g, **kw)
    mag = oracle.expert_backward(inp["x"], clean, w, inp["w1"], inp["w2"], g, magnitude=True,
                                 **kw)
    res, st = run_backward_routed(shape, {k: v.to(DEV) for k, v in inp.items()}, idx, w,
                                  g.to(DEV))
    assert moe.STATUS_NAMES[st] == "MOE_ERR_DEVICE_INDEX"
    for name in ("dx", "dw1", "dw2", "dw_route"):
        assert_grad_bound(res[name], ref[name], mag[name], f"{name} (invalid routes masked)")
