"""Pins of the oracle's GEMM1 -> SwiGLU -> GEMM2 -> combine against library
routines and closed forms (numpy matmul, scipy.special.expit)."""
import numpy as np
import pytest
import scipy.special as sps
import torch

import moe_inputs as mi
import oracle


def _f64(t):
    return t.to(torch.float64).numpy()


def dense_mlp(x, w1, w2, F):
    """Textbook SwiGLU MLP with numpy matmul: (silu(x Wg^T) * (x Wu^T)) W2^T."""
    g = x @ w1[:F].T
    u = x @ w1[F:].T
    return ((g * sps.expit(g)) * u) @ w2.T


def test_single_expert_top1_is_dense_swiglu_mlp():
    s = mi.MoEShape("e1", T=9, H=64, F=96, E=1, k=1)
    inp = mi.make_inputs(s, seed=5)
    res = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], k=1)
    exp = dense_mlp(_f64(inp["x"]), _f64(inp["w1"][0]), _f64(inp["w2"][0]), s.F)
    np.testing.assert_allclose(res["out"], exp, rtol=1e-10, atol=1e-12)
    assert (res["topk_idx"] == 0).all() and (res["topk_w"] == 1.0).all()


def test_identical_experts_give_the_dense_mlp():
    # all experts equal and weights summing to one: routing cannot matter
    s = mi.MoEShape("same", T=20, H=64, F=64, E=6, k=3)
    inp = mi.make_inputs(s, seed=2)
    w1 = inp["w1"][:1].expand(s.E, -1, -1).contiguous()
    w2 = inp["w2"][:1].expand(s.E, -1, -1).contiguous()
    res = oracle.moe_forward(inp["x"], inp["logits"], w1, w2, k=s.k)
    exp = dense_mlp(_f64(inp["x"]), _f64(w1[0]), _f64(w2[0]), s.F)
    np.testing.assert_allclose(res["out"], exp, rtol=1e-10, atol=1e-12)


def test_power_of_two_expert_scaling_reaches_the_right_expert():
    # W2_e = 2^e * W2_0 (exact in bf16) -> out_t = sum_j w_tj 2^{e_tj} * MLP_0(x_t)
    s = mi.MoEShape("scaled", T=24, H=64, F=32, E=5, k=2)
    inp = mi.make_inputs(s, seed=9)
    w1 = inp["w1"][:1].expand(s.E, -1, -1).contiguous()
    w2 = torch.stack([inp["w2"][0] * (2.0 ** e) for e in range(s.E)]).contiguous()
    res = oracle.moe_forward(inp["x"], inp["logits"], w1, w2, k=s.k)
    idx, w = oracle.route_topk(inp["logits"], s.k)
    scale = (w * np.exp2(idx)).sum(1, keepdims=True)
    base = dense_mlp(_f64(inp["x"]), _f64(w1[0]), _f64(inp["w2"][0]), s.F)
    np.testing.assert_allclose(res["out"], scale * base, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("I", [1, 8, 32, 64])
def test_glu_interleave_is_a_row_reordering_of_gate_up(I):
    s = mi.MoEShape("il", T=16, H=64, F=64, E=4, k=2)
    inp = mi.make_inputs(s, seed=4)
    w1 = inp["w1"]
    gate, up = w1[:, :s.F], w1[:, s.F:]
    # blocks of I gate rows then I up rows, built by reshaping (no index formula)
    il = torch.stack([gate.reshape(s.E, s.F // I, I, s.H), up.reshape(s.E, s.F // I, I, s.H)],
                     dim=2).reshape(s.E, 2 * s.F, s.H).contiguous()
    a = oracle.moe_forward(inp["x"], inp["logits"], w1, inp["w2"], k=s.k)
    b = oracle.moe_forward(inp["x"], inp["logits"], il, inp["w2"], k=s.k, interleave=I)
    np.testing.assert_array_equal(a["out"], b["out"])
    if I < s.F:  # reading the interleaved layout as [gate|up] must change the answer
        c = oracle.moe_forward(inp["x"], inp["logits"], il, inp["w2"], k=s.k)
        assert np.abs(c["out"] - a["out"]).max() > 1e-3


def test_swiglu_clamp_closed_form():
    # one-hot x picks column 0 of W1, so g_f, u_f are the chosen numbers;
    # W2 = identity makes the output equal h.
    F = H = 8
    gs = np.array([10.0, -10.0, 3.0, 7.5, 0.0, -2.0, 100.0, 6.5], np.float32)
    us = np.array([10.0, -10.0, -9.0, 2.0, 5.0, 8.0, -100.0, -6.0], np.float32)
    w1 = np.zeros((1, 2 * F, H), np.float32)
    w1[0, :F, 0] = gs
    w1[0, F:, 0] = us
    w2 = np.eye(H, F, dtype=np.float32)[None]
    x = np.zeros((1, H), np.float32)
    x[0, 0] = 1.0
    tb = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    logits = torch.zeros(1, 1)
    silu = lambda z: z * sps.expit(z)
    for c in (7.0, 0.0, float("inf")):
        out = oracle.moe_forward(tb(x), logits, tb(w1), tb(w2), k=1, clamp=c)["out"][0]
        g = gs.astype(np.float64)
        u = us.astype(np.float64)
        if 0 < c < np.inf:
            g = np.minimum(g, c)
            u = np.clip(u, -c, c)
        np.testing.assert_allclose(out, silu(g) * u, rtol=1e-14, atol=1e-300)
    # spot values written out: silu(7)*7, silu(-10)*(-7), silu(3)*(-7)
    out = oracle.moe_forward(tb(x), logits, tb(w1), tb(w2), k=1, clamp=7.0)["out"][0]
    np.testing.assert_allclose(out[:3], [7 * 7 * sps.expit(7.0), -10 * sps.expit(-10.0) * -7,
                                         3 * sps.expit(3.0) * -7], rtol=1e-14)


def test_integer_operands_are_exact():
    # small-integer x and W: every GEMM1 dot product is an exact integer
    s = mi.MoEShape("int", T=12, H=32, F=16, E=3, k=2)
    g = torch.Generator().manual_seed(1)
    x = torch.randint(-3, 4, (s.T, s.H), generator=g).to(torch.bfloat16)
    w1 = torch.randint(-2, 3, (s.E, 2 * s.F, s.H), generator=g).to(torch.bfloat16)
    logits = torch.randn(s.T, s.E, generator=g)
    idx, _ = oracle.route_topk(logits, s.k)
    p = oracle.permute(idx, s.E)
    xp = oracle.gather_rows(x, p["permuted_token"])
    h = oracle.gemm1_swiglu(xp, p["expert_offsets"], w1, s.F)
    xf = x.to(torch.int64).numpy()
    for t in range(s.T):
        for j in range(s.k):
            e, r = idx[t, j], p["row_id_map"][t, j]
            gi = xf[t] @ w1[e, :s.F].to(torch.int64).numpy().T
            ui = xf[t] @ w1[e, s.F:].to(torch.int64).numpy().T
            np.testing.assert_allclose(h[r], gi * sps.expit(gi) * ui, rtol=1e-14, atol=1e-300)


def test_dense_bruteforce_agrees_with_permuted_form():
    s = mi.MoEShape("bf", T=33, H=64, F=64, E=8, k=3)
    inp = mi.make_inputs(s, seed=1)
    res = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], k=s.k, clamp=0.5)
    bf = oracle.dense_bruteforce(inp["x"], res["topk_idx"], res["topk_w"], inp["w1"], inp["w2"],
                                 clamp=0.5)
    np.testing.assert_allclose(res["out"], bf, rtol=1e-12, atol=1e-14)


def test_unused_experts_may_be_absent():
    s = mi.MoEShape("sparse", T=4, H=64, F=32, E=16, k=2)
    inp = mi.make_inputs(s, seed=6)
    full = oracle.moe_forward(inp["x"], inp["logits"], inp["w1"], inp["w2"], k=s.k)
    used = set(full["topk_idx"].ravel().tolist())
    w1l = [inp["w1"][e] if e in used else None for e in range(s.E)]
    w2l = [inp["w2"][e] if e in used else None for e in range(s.E)]
    part = oracle.moe_forward(inp["x"], inp["logits"], w1l, w2l, k=s.k)
    np.testing.assert_array_equal(full["out"], part["out"])


def test_routed_composition_matches_bruteforce_with_masks():
    """The staged oracle (permute -> gather -> GEMM1 -> GEMM2 -> combine) with
    caller routing that masks slots equals the per-token brute force, and a
    token with every slot masked gives a zero row."""
    shape = mi.MoEShape("routed", T=40, H=64, F=96, E=6, k=3)
    inp = mi.make_inputs(shape, seed=4)
    idx = mi.random_topk_idx(shape.T, shape.E, shape.k, seed=4, mask_frac=0.3)
    idx[5] = -1
    w = mi.random_weights(shape.T, shape.k, seed=4)
    got = oracle.moe_forward_routed(inp["x"], idx, w, inp["w1"], inp["w2"], interleave=32)
    ref = oracle.dense_bruteforce(inp["x"], idx, w, inp["w1"], inp["w2"], interleave=32)
    np.testing.assert_allclose(got["out"], ref, rtol=1e-12, atol=1e-12)
    assert not got["out"][5].any()
    assert int(got["tokens_per_expert"].sum()) == int((idx.numpy() >= 0).sum())


def test_shared_experts_add_their_dense_mlp():
    """With S shared experts the output is the routed layer's plus, for every
    token, each shared expert's textbook SwiGLU MLP (numpy matmul) with weight
    1; the routed slots are the plain routing's."""
    E, S, k = 6, 2, 2
    shape = mi.MoEShape("shared", T=30, H=64, F=96, E=E + S, k=k)
    inp = mi.make_inputs(shape, seed=9)
    logits = mi.make_logits(mi.MoEShape("routed-part", T=30, H=64, F=96, E=E, k=k), seed=9)
    res = oracle.moe_forward_shared(inp["x"], logits, inp["w1"], inp["w2"], k, S)
    base = oracle.moe_forward(inp["x"], logits, inp["w1"][:E], inp["w2"][:E], k)
    x = _f64(inp["x"])
    want = sum(dense_mlp(x, _f64(inp["w1"][E + s]), _f64(inp["w2"][E + s]), shape.F)
               for s in range(S))
    np.testing.assert_allclose(res["out"] - base["out"], want, rtol=1e-9, atol=1e-12)
    assert (res["topk_idx"][:, :k] == base["topk_idx"]).all()
    assert (res["topk_idx"][:, k:] == np.arange(E, E + S)).all()
    assert (res["tokens_per_expert"][E:] == shape.T).all()
