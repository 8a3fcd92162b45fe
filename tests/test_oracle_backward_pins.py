"""Pins of the oracle's backward (gradients of sum(dOut * out) with respect to
x, the router logits, W1 and W2) against quantities it does not compute itself:

  * torch.autograd through a plain float64 forward of the layer written here
    (loops over tokens and slots, no permutation) -- the derivatives are taken
    mechanically from the forward's definition, not from the oracle's
    hand-derived formulas;
  * central finite differences of that forward along random directions;
  * invariants of the softmax router (gradients sum to zero per token and
    vanish off the selection when the weights are renormalised);
  * the sampled forms (single dx rows, dW1 rows, dW2 columns) against the
    whole backward.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle


def _rows(F, I):
    """W1 rows of gate and up column f (the layer's GLU interleave reading)."""
    f = np.arange(F)
    if I == 0:
        return f, f + F
    gate = (f // I) * 2 * I + f % I
    return gate, gate + I


def torch_layer(x, logits, w1, w2, idx, k, renormalize, I, c, S):
    """The layer in float64 torch ops with autograd.  ``idx`` [T, k+S] is the
    selection (piecewise constant, so it carries no gradient)."""
    T = x.shape[0]
    F = w2.shape[2]
    gate, up = (torch.as_tensor(r) for r in _rows(F, I))
    rows = []
    for t in range(T):
        sel = torch.as_tensor(idx[t, :k].astype(np.int64))
        if renormalize:
            w = torch.softmax(logits[t, sel], 0)
        else:
            w = torch.softmax(logits[t], 0)[sel]
        o = torch.zeros_like(x[t])
        for j in range(k + S):
            e = int(idx[t, j])
            a = w1[e] @ x[t]
            g, u = a[gate], a[up]
            if c > 0:
                g = torch.clamp(g, max=c)
                u = torch.clamp(u, -c, c)
            y = w2[e] @ (torch.nn.functional.silu(g) * u)
            o = o + (w[j] if j < k else 1.0) * y
        rows.append(o)
    return torch.stack(rows)


def _case(T=12, H=32, F=16, E=5, k=2, S=0, seed=3):
    s = mi.MoEShape("bwd", T=T, H=H, F=F, E=E + S, k=k)
    inp = mi.make_inputs(s, seed=seed)
    logits = inp["logits"][:, :E].contiguous()
    g = mi.make_grad_out(s, seed=seed)
    return inp["x"], logits, inp["w1"], inp["w2"], g


def _autograd(x, logits, w1, w2, g, k, renormalize, I, c, S):
    idx, _ = oracle.routes_with_shared(logits, k, S, renormalize)
    xt, lt, w1t, w2t = (t.to(torch.float64).clone().requires_grad_(True)
                        for t in (x, logits, w1, w2))
    out = torch_layer(xt, lt, w1t, w2t, idx, k, renormalize, I, c, S)
    (out * g.to(torch.float64)).sum().backward()
    return {"dx": xt.grad.numpy(), "dlogits": lt.grad.numpy(), "dw1": w1t.grad.numpy(),
            "dw2": w2t.grad.numpy(), "out": out.detach().numpy()}


@pytest.mark.parametrize("renormalize", [True, False])
@pytest.mark.parametrize("I,c,S", [(0, 0.0, 0), (8, 0.0, 0), (0, 0.8, 0), (4, 0.6, 0),
                                   (0, 0.0, 1), (8, 0.8, 2)])
def test_backward_matches_autograd_of_the_plain_forward(renormalize, I, c, S):
    k = 2
    x, logits, w1, w2, g = _case(S=S)
    ref = _autograd(x, logits, w1, w2, g, k, renormalize, I, c, S)
    res = oracle.moe_backward(x, logits, w1, w2, g, k, renormalize=renormalize, interleave=I,
                              clamp=c, shared_experts=S)
    for name in ("dx", "dlogits", "dw1", "dw2"):
        np.testing.assert_allclose(res[name], ref[name], rtol=1e-10, atol=1e-12, err_msg=name)
    # the autograd forward is the oracle's forward (with these routes)
    fwd = oracle.moe_forward_routed(x, res["topk_idx"], res["topk_w"], w1, w2, interleave=I,
                                    clamp=c)
    np.testing.assert_allclose(fwd["out"], ref["out"], rtol=1e-10, atol=1e-12)


def test_clamp_masks_actually_bite():
    # the clamped case must differ from the unclamped one, or the test above
    # would not see a dropped mask
    x, logits, w1, w2, g = _case()
    a = oracle.moe_backward(x, logits, w1, w2, g, 2, clamp=0.8)
    b = oracle.moe_backward(x, logits, w1, w2, g, 2, clamp=0.0)
    assert np.abs(a["dw1"] - b["dw1"]).max() > 1e-2


@pytest.mark.parametrize("renormalize", [True, False])
def test_directional_finite_differences(renormalize):
    k, I, c, S = 2, 8, 0.8, 1
    x, logits, w1, w2, g = _case(S=S, seed=11)
    res = oracle.moe_backward(x, logits, w1, w2, g, k, renormalize=renormalize, interleave=I,
                              clamp=c, shared_experts=S)
    idx = res["topk_idx"]
    base = [t.to(torch.float64) for t in (x, logits, w1, w2)]
    G = g.to(torch.float64)
    rng = np.random.default_rng(0)
    eps = 1e-6
    for i, name in enumerate(("dx", "dlogits", "dw1", "dw2")):
        D = torch.as_tensor(rng.standard_normal(base[i].shape))
        def loss(sign):
            args = list(base)
            args[i] = base[i] + sign * eps * D
            with torch.no_grad():
                return float((torch_layer(*args, idx, k, renormalize, I, c, S) * G).sum())
        fd = (loss(1) - loss(-1)) / (2 * eps)
        an = float((res[name] * D.numpy()).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


@pytest.mark.parametrize("renormalize", [True, False])
def test_router_gradient_invariants(renormalize):
    x, logits, w1, w2, g = _case(T=20, E=7, k=3, seed=5)
    res = oracle.moe_backward(x, logits, w1, w2, g, 3, renormalize=renormalize)
    dl = res["dlogits"]
    # softmax is invariant to adding a constant to a token's logits
    np.testing.assert_allclose(dl.sum(1), 0.0, atol=1e-12)
    if renormalize:
        mask = np.zeros_like(dl, dtype=bool)
        np.put_along_axis(mask, res["topk_idx"].astype(np.int64), True, axis=1)
        assert (dl[~mask] == 0.0).all()
    else:
        assert (dl != 0.0).all()


def test_gradients_are_linear_in_the_output_gradient():
    x, logits, w1, w2, g = _case(seed=8)
    a = oracle.moe_backward(x, logits, w1, w2, g, 2, clamp=0.8)
    b = oracle.moe_backward(x, logits, w1, w2, (g.float() * -2).to(torch.bfloat16), 2, clamp=0.8)
    for name in ("dx", "dlogits", "dw1", "dw2"):
        np.testing.assert_allclose(b[name], -2 * a[name], rtol=1e-12, atol=1e-14)


def test_expert_without_routes_gets_zero_weight_gradients():
    x, logits, w1, w2, g = _case(T=6, E=5, k=1, seed=1)
    logits = logits.clone()
    logits[:, 3] = -50.0  # expert 3 never selected
    res = oracle.moe_backward(x, logits, w1, w2, g, 1)
    assert (res["topk_idx"] != 3).all()
    assert (res["dw1"][3] == 0).all() and (res["dw2"][3] == 0).all()
    assert np.abs(res["dw1"]).sum() > 0


def test_masked_routes_contribute_nothing():
    # a masked slot is the same as the route never existing
    x, logits, w1, w2, g = _case(T=10, E=6, k=3, seed=6)
    idx, w = oracle.route_topk(logits, 3)
    idx_m = idx.copy()
    idx_m[::3, 1] = -1
    a = oracle.expert_backward(x, idx_m, w, w1, w2, g)
    keep = idx_m >= 0
    # drop the masked slot by giving it weight 0 and any valid expert: dy = 0,
    # so only dw_route of that slot could differ
    idx_z, w_z = idx.copy(), w.copy()
    w_z[~keep] = 0.0
    b = oracle.expert_backward(x, idx_z, w_z, w1, w2, g)
    np.testing.assert_allclose(a["dx"], b["dx"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a["dw1"], b["dw1"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a["dw2"], b["dw2"], rtol=1e-12, atol=1e-14)
    assert (a["dw_route"][~keep] == 0).all()


@pytest.mark.parametrize("magnitude", [False, True])
@pytest.mark.parametrize("I,c", [(0, 0.0), (8, 0.7)])
def test_sampled_forms_match_the_whole_backward(I, c, magnitude):
    x, logits, w1, w2, g = _case(T=16, E=4, k=2, seed=2)
    idx, w = oracle.route_topk(logits, 2)
    full = oracle.expert_backward(x, idx, w, w1, w2, g, interleave=I, clamp=c, mask_f32=True, magnitude=magnitude)
    toks = [0, 5, 15]
    dx, dw = oracle.backward_tokens(x, idx, w, w1, w2, g, toks, interleave=I, clamp=c,
                                    mask_f32=True, magnitude=magnitude)
    np.testing.assert_allclose(dx, full["dx"][toks], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dw, full["dw_route"][toks], rtol=1e-12, atol=1e-14)
    pairs = [(0, 0), (1, 17), (3, 31), (2, 8)]
    rows = oracle.backward_dw1_rows(x, idx, w, w1, w2, g, pairs, interleave=I, clamp=c,
                                    mask_f32=True, magnitude=magnitude)
    for i, (e, r) in enumerate(pairs):
        np.testing.assert_allclose(rows[i], full["dw1"][e, r], rtol=1e-12, atol=1e-14)
    pairs = [(0, 0), (1, 15), (3, 7)]
    cols = oracle.backward_dw2_cols(x, idx, w, w1, w2, g, pairs, interleave=I, clamp=c,
                                    mask_f32=True, magnitude=magnitude)
    for i, (e, f) in enumerate(pairs):
        np.testing.assert_allclose(cols[i], full["dw2"][e, :, f], rtol=1e-12, atol=1e-14)


def test_mask_precision_matters_only_with_a_clamp():
    x, logits, w1, w2, g = _case(seed=4)
    a = oracle.moe_backward(x, logits, w1, w2, g, 2, mask_f32=False)
    b = oracle.moe_backward(x, logits, w1, w2, g, 2, mask_f32=True)
    for name in ("dx", "dw1", "dw2"):
        np.testing.assert_array_equal(a[name], b[name])
    # with a clamp, values more than an fp32 rounding away from it decide alike
    a = oracle.moe_backward(x, logits, w1, w2, g, 2, clamp=0.8, mask_f32=False)
    b = oracle.moe_backward(x, logits, w1, w2, g, 2, clamp=0.8, mask_f32=True)
    for name in ("dx", "dw1", "dw2"):
        np.testing.assert_array_equal(a[name], b[name])


@pytest.mark.parametrize("renormalize", [True, False])
def test_magnitudes_bound_the_gradients(renormalize):
    x, logits, w1, w2, g = _case(T=14, E=5, k=2, S=1, seed=12)
    kw = dict(renormalize=renormalize, interleave=8, clamp=0.8, shared_experts=1)
    v = oracle.moe_backward(x, logits, w1, w2, g, 2, **kw)
    m = oracle.moe_backward(x, logits, w1, w2, g, 2, magnitude=True, **kw)
    for name in ("dx", "dlogits", "dw1", "dw2", "dw_route"):
        assert (m[name] >= np.abs(v[name]) * (1 - 1e-12)).all(), name
        assert (m[name] >= 0).all(), name
    # the magnitudes do not see the sign of the output gradient
    mneg = oracle.moe_backward(x, logits, w1, w2, (-g.float()).to(torch.bfloat16), 2,
                               magnitude=True, **kw)
    for name in ("dx", "dlogits", "dw1", "dw2"):
        np.testing.assert_allclose(mneg[name], m[name], rtol=1e-12, atol=0)


def test_magnitude_of_a_single_term_is_its_absolute_value():
    # one token, one expert: every dW element is a single product
    x, logits, w1, w2, g = _case(T=1, E=1, k=1, seed=13)
    v = oracle.moe_backward(x, logits, w1, w2, g, 1, clamp=0.8)
    m = oracle.moe_backward(x, logits, w1, w2, g, 1, clamp=0.8, magnitude=True)
    np.testing.assert_allclose(m["dw1"], np.abs(v["dw1"]), rtol=1e-12, atol=0)
    np.testing.assert_allclose(m["dw2"], np.abs(v["dw2"]), rtol=1e-12, atol=0)
