"""Pins of the fp64 CPU oracle against things other than itself.

Every check here compares the oracle with brute force on tiny inputs, a
library routine (numpy matmul, scipy's softmax/expit), a closed form, a
hand-derived golden fixture or an invariant -- never with a retyped copy of
the oracle's own formula.  Each is chosen so that a plausible slip (a swapped
gate/up, a transposed weight, a wrong tie-break, an unstable scatter, a
dropped slot) fails at least one test.
"""
import json
import os

import numpy as np
import pytest
import scipy.special as sps
import torch

import moe_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def _f64(t):
    return t.to(torch.float64).numpy()


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("T,E,k", [(50, 8, 2), (40, 16, 5), (30, 3, 3), (20, 33, 1)])
def test_route_matches_bruteforce_sort_with_ties(T, E, k):
    # small integer logits force many exact ties
    g = torch.Generator().manual_seed(T * 7 + E)
    logits = torch.randint(-3, 4, (T, E), generator=g).to(torch.float32)
    idx, w = oracle.route_topk(logits, k)
    lg = logits.numpy()
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))  # python's sort: independent
        assert list(idx[t]) == order[:k]
    # renormalised weights = library softmax over the selected logits
    sel = np.take_along_axis(lg.astype(np.float64), idx, axis=1)
    np.testing.assert_allclose(w, sps.softmax(sel, axis=1), rtol=1e-14, atol=0)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)


def test_route_all_equal_logits_picks_lowest_ids():
    logits = torch.zeros(4, 8)
    logits[1] = -0.0
    idx, w = oracle.route_topk(logits, 3)
    assert (idx == np.array([0, 1, 2])).all()
    np.testing.assert_allclose(w, 1.0 / 3.0, rtol=1e-15)


def test_route_k1_weight_is_one_and_k2_is_sigmoid():
    lg = mi.make_logits(mi.TINY)
    idx1, w1 = oracle.route_topk(lg, 1)
    assert (idx1[:, 0] == np.argmax(lg.numpy(), axis=1)).all()
    np.testing.assert_array_equal(w1, 1.0)
    idx2, w2 = oracle.route_topk(lg, 2)
    a = np.take_along_axis(lg.numpy().astype(np.float64), idx2, 1)
    np.testing.assert_allclose(w2[:, 0], sps.expit(a[:, 0] - a[:, 1]), rtol=1e-13)


def test_route_unnormalised_is_full_softmax():
    lg = mi.make_logits(mi.TINY)
    idx, w = oracle.route_topk(lg, 2, renormalize=False)
    p = sps.softmax(lg.numpy().astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(p, idx, 1), rtol=1e-13)
    # k = E with renormalisation is the full softmax too
    idxE, wE = oracle.route_topk(lg, 8)
    np.testing.assert_allclose(wE, np.take_along_axis(p, idxE, 1), rtol=1e-13)


def test_route_rejects_k_above_E():
    with pytest.raises(ValueError):
        oracle.route_topk(torch.zeros(2, 4), 5)


# ------------------------------------------------------------------ permute

def test_permute_golden_fixture():
    with open(os.path.join(GOLDEN, "permute_small.json")) as f:
        g = json.load(f)
    p = oracle.permute(np.array(g["topk_idx"], np.int32), g["E"])
    for key in ("tokens_per_expert", "expert_offsets", "row_id_map", "permuted_token"):
        np.testing.assert_array_equal(p[key], np.array(g[key]), err_msg=key)


@pytest.mark.parametrize("T,E,k,mask", [(64, 8, 2, 0.0), (37, 33, 5, 0.0), (50, 16, 4, 0.3),
                                         (1, 1, 1, 0.0), (0, 4, 2, 0.0)])
def test_permute_matches_stable_sort(T, E, k, mask):
    idx = mi.random_topk_idx(T, E, k, seed=T + E, mask_frac=mask).numpy()
    p = oracle.permute(idx, E)
    valid = idx >= 0
    # numpy's stable argsort on the key (expert, token) -- an independent ordering
    tt, jj = np.nonzero(valid)
    order = np.lexsort((tt, idx[tt, jj]))
    n = len(order)
    exp_rmap = -np.ones_like(idx)
    exp_rmap[tt[order], jj[order]] = np.arange(n)
    np.testing.assert_array_equal(p["row_id_map"], exp_rmap)
    exp_ptok = -np.ones(T * k, np.int32)
    exp_ptok[:n] = tt[order]
    np.testing.assert_array_equal(p["permuted_token"], exp_ptok)
    np.testing.assert_array_equal(p["tokens_per_expert"], np.bincount(idx[valid], minlength=E))
    # invariants
    assert p["tokens_per_expert"].sum() == valid.sum()
    assert p["expert_offsets"][0] == 0 and (np.diff(p["expert_offsets"]) >= 0).all()
    for t, j in zip(tt, jj):
        assert p["permuted_token"][p["row_id_map"][t, j]] == t


def test_permute_rejects_duplicates_and_out_of_range():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[1, 1]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, -2]], np.int32), 4)


def test_permute_then_unpermute_with_unit_weights_is_identity():
    T, E, k, H = 40, 8, 2, 24
    x = mi.make_x(mi.MoEShape("t", T=T, H=H, F=8, E=E, k=k))
    idx = mi.random_topk_idx(T, E, k, seed=3, mask_frac=0.2).numpy()
    p = oracle.permute(idx, E)
    xp = oracle.gather_rows(x, p["permuted_token"])
    y = torch.from_numpy(xp.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nvalid = (idx >= 0).sum(1, keepdims=True)
    w = np.where(idx >= 0, 1.0 / np.maximum(nvalid, 1), 0.0)
    out = oracle.unpermute_combine(y, p["row_id_map"], w)
    xf = _f64(x)
    exp = np.where(nvalid > 0, xf, 0.0)
    np.testing.assert_array_equal(out, exp)  # halves of a bf16 value add exactly in fp64


def test_combine_skips_masked_slots_and_is_linear():
    T, k, H = 6, 3, 5
    rng = np.random.default_rng(1)
    y = rng.standard_normal((T * k, H))
    rmap = np.arange(T * k, dtype=np.int32).reshape(T, k)
    rmap[2, 1] = -1
    w = rng.random((T, k))
    out = oracle.unpermute_combine(y, rmap, w)
    out2 = oracle.unpermute_combine(2.0 * y, rmap, w)
    np.testing.assert_allclose(out2, 2.0 * out, rtol=1e-15)
    np.testing.assert_allclose(out[2], w[2, 0] * y[6] + w[2, 2] * y[8], rtol=1e-15)
