"""Pins of the oracle's low-precision arithmetic (FP8 E4M3, NVFP4 = E2M1 +
E4M3 block scales + an fp32 tensor scale) against torch's float8 casts and
the OCP format tables, and of its NVFP4 GEMM against the (already pinned)
bf16 oracle on weights whose dequantised values are exact in bf16."""
import math

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

# E2M1 code -> value, from the OCP Microscaling Formats specification
# (sign bit, 2 exponent bits with bias 1, 1 mantissa bit).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def torch_e4m3(codes):
    return torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)


def test_e4m3_decode_matches_torch_for_all_codes():
    ref = torch_e4m3(list(range(256))).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all() and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_e2m1_decode_matches_ocp_table():
    got = [oracle.e2m1_value(c) for c in range(16)]
    assert got == E2M1_TABLE
    assert [math.copysign(1, v) for v in got] == [math.copysign(1, v) for v in E2M1_TABLE]


def test_e4m3_encode_is_torch_rne_in_range_and_saturates():
    g = torch.Generator().manual_seed(0)
    mags = torch.exp2(torch.empty(4000).uniform_(-12, 8.8, generator=g))
    vals = (mags * torch.where(torch.rand(4000, generator=g) < 0.5, -1.0, 1.0)).float()
    vals = vals.clamp(-448, 448)
    # also every midpoint between adjacent finite codes (ties must go to even)
    pos = torch_e4m3(list(range(127))).float()
    mids = ((pos[1:].double() + pos[:-1].double()) / 2).float()
    allv = torch.cat([vals, mids, -mids])
    want = allv.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in allv])
    # torch keeps the sign of zero; compare decoded values
    np.testing.assert_array_equal(torch_e4m3(got.tolist()).numpy(), torch_e4m3(want.tolist()).numpy())
    assert oracle.e4m3_encode(500.0) == 0x7E and oracle.e4m3_encode(-1e9) == 0xFE
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(0.0) == 0


def test_requant_block_closed_form():
    # block whose maximum maps to 448 exactly; values that are E4M3 numbers
    # times the scale come back unchanged
    s = 0.125
    codes = list(range(0, 120, 1)) + [0x7E] * 8   # includes 448
    vals = torch_e4m3(codes).numpy() * s
    out = oracle.requant_fp8_block(vals)
    np.testing.assert_array_equal(out, vals)
    assert (oracle.requant_fp8_block(np.zeros(128)) == 0).all()
    # generic block: error at most half an E4M3 step of each value, scale amax/448
    rng = np.random.default_rng(0)
    h = rng.standard_normal(128) * 3
    out = oracle.requant_fp8_block(h)
    sc = np.float32(np.abs(h).astype(np.float32).max()) / np.float32(448)
    assert np.all(np.abs(out - h) <= np.abs(h) * 2.0 ** -4 + float(sc) * 2.0 ** -10)


def _dequant_nvfp4(q, s, g):
    """Dequantised NVFP4 values (exact in fp64) from packed codes: even index =
    low nibble, one E4M3 scale per 16 values, times g."""
    lo = (q & 15).to(torch.long)
    hi = (q >> 4).to(torch.long)
    codes = torch.stack([lo, hi], dim=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    table = torch.tensor(E2M1_TABLE, dtype=torch.float64)
    sv = s.view(torch.float8_e4m3fn).to(torch.float64)
    return table[codes] * sv.repeat_interleave(16, dim=-1) * g


@pytest.mark.parametrize("interleave", [0, 32])
def test_nvfp4_gemm1_matches_bf16_oracle_on_exact_values(interleave):
    # g a power of two and scales <= 2^-2: dequantised weights have <= 6
    # significant bits and are exact in bf16; FP8 activations with per-128
    # power-of-two scales are exact in bf16 too.
    s = mi.MoEShape("lp", T=20, H=256, F=128, E=3, k=2)
    g = torch.Generator().manual_seed(2)
    E, N, K = s.E, 2 * s.F, s.H
    q = torch.randint(0, 256, (E, N, K // 2), generator=g, dtype=torch.uint8)
    sc = torch.randint(0x10, 0x30, (E, N, K // 16), generator=g, dtype=torch.uint8)
    g1 = torch.tensor([2.0 ** -3, 1.0, 2.0 ** 2], dtype=torch.float32)
    xq = torch.randint(0, 256, (s.T, K), generator=g, dtype=torch.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x11  # no NaN codes
    xs = torch.exp2(torch.randint(-3, 3, (s.T, K // 128), generator=g).float())
    w_hat = torch.stack([_dequant_nvfp4(q[e], sc[e], float(g1[e])) for e in range(E)])
    x_hat = torch_e4m3(xq.flatten().tolist()).reshape(s.T, K) * xs.double().repeat_interleave(128, 1)
    logits = torch.randn(s.T, E, generator=g)
    idx, _ = oracle.route_topk(logits, s.k)
    p = oracle.permute(idx, E)
    pt = torch.from_numpy(p["permuted_token"]).long()
    h_lp = oracle.gemm1_swiglu_lowprec(xq[pt], xs[pt], p["expert_offsets"], q, sc, g1, s.F,
                                       interleave, 7.0, requant=False)
    w_b = w_hat.to(torch.bfloat16)
    assert torch.equal(w_b.double(), w_hat)
    x_b = x_hat.to(torch.bfloat16)
    assert torch.equal(x_b.double(), x_hat)
    xp = oracle.gather_rows(x_b, p["permuted_token"])
    h_ref = oracle.gemm1_swiglu(xp, p["expert_offsets"], w_b, s.F, interleave, 7.0)
    np.testing.assert_allclose(h_lp, h_ref, rtol=1e-12, atol=1e-12)


def test_nvfp4_gemm2_matches_bf16_oracle_on_exact_values():
    s = mi.MoEShape("lp2", T=12, H=256, F=128, E=2, k=1)
    g = torch.Generator().manual_seed(3)
    q = torch.randint(0, 256, (s.E, s.H, s.F // 2), generator=g, dtype=torch.uint8)
    sc = torch.randint(0x18, 0x30, (s.E, s.H, s.F // 16), generator=g, dtype=torch.uint8)
    g2 = torch.tensor([0.5, 2.0], dtype=torch.float32)
    w_hat = torch.stack([_dequant_nvfp4(q[e], sc[e], float(g2[e])) for e in range(s.E)])
    off = np.array([0, 5, 12], np.int32)
    h = torch.randn(12, s.F, generator=g, dtype=torch.float64)
    y_lp = oracle.gemm2_lowprec(h.numpy(), off, q, sc, g2, s.H)
    y_ref = np.concatenate([h[0:5].numpy() @ w_hat[0].numpy().T, h[5:12].numpy() @ w_hat[1].numpy().T])
    np.testing.assert_allclose(y_lp, y_ref, rtol=1e-12, atol=1e-12)


def test_lowprec_forward_is_composition_of_its_steps():
    s = mi.MoEShape("lpf", T=24, H=256, F=256, E=4, k=2, glu_interleave=32, swiglu_clamp=7.0,
                    lowprec=True)
    inp = mi.make_lowprec_inputs(s, seed=1)
    res = oracle.moe_forward_lowprec(inp["xq"], inp["xs"], inp["logits"], inp["w1q"], inp["w1s"],
                                     inp["w1g"], inp["w2q"], inp["w2s"], inp["w2g"], s.k,
                                     interleave=32, clamp=7.0)
    idx, w = oracle.route_topk(inp["logits"], s.k)
    p = oracle.permute(idx, s.E)
    pt = torch.from_numpy(p["permuted_token"]).long()
    h = oracle.gemm1_swiglu_lowprec(inp["xq"][pt], inp["xs"][pt], p["expert_offsets"], inp["w1q"],
                                    inp["w1s"], inp["w1g"], s.F, 32, 7.0, requant=True)
    # every 128-block of h is E4M3 values times one scale
    for r in range(h.shape[0]):
        for b in range(0, s.F, 128):
            blk = h[r, b:b + 128]
            np.testing.assert_array_equal(oracle.requant_fp8_block(blk), blk)
    y = oracle.gemm2_lowprec(h, p["expert_offsets"], inp["w2q"], inp["w2s"], inp["w2g"], s.H)
    out = oracle.unpermute_combine(y, p["row_id_map"], w)
    np.testing.assert_allclose(res["out"], out, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(res["topk_idx"], idx)


def test_quantised_inputs_approximate_the_normal_draws():
    s = mi.MoEShape("lpq", T=8, H=256, F=128, E=2, k=1, lowprec=True)
    w = torch.randn(2 * s.F, s.H, generator=torch.Generator().manual_seed(4)) / 16
    q, sc, g = mi.quantize_nvfp4(w)
    w_hat = _dequant_nvfp4(q, sc, float(g))
    rel = (w_hat - w.double()).norm() / w.double().norm()
    assert rel < 0.15  # NVFP4 keeps about 2 significant bits
    assert (sc.view(torch.float8_e4m3fn).float() * 6 <= 448).all()


# ---------------------------------------------------------------- MXFP4 weights

def test_e8m0_decode_is_a_power_of_two():
    assert [oracle.e8m0_value(e) for e in range(255)] == [math.ldexp(1.0, e - 127)
                                                         for e in range(255)]


def mx_dequant(q, s):
    """Test-side MXFP4 decode: OCP E2M1 table x 2^(scale - 127) per 32 values."""
    q, s = q.numpy(), s.numpy()
    codes = np.stack([q & 15, q >> 4], axis=-1).reshape(q.shape[0], -1)
    vals = np.array(E2M1_TABLE)[codes]
    return vals * np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, axis=1)


def test_mxfp4_gemm2_matches_numpy_on_decoded_weights():
    g = torch.Generator().manual_seed(3)
    E, H, F, R = 3, 64, 128, 20
    w2 = torch.randn(E, H, F, generator=g) / 10
    qs = [mi.quantize_mxfp4(w2[e]) for e in range(E)]
    h = torch.randn(R, F, generator=g, dtype=torch.float64).numpy()
    off = np.array([0, 7, 7, 20], np.int32)
    got = oracle.gemm2_lowprec(h, off, [q for q, _ in qs], [s for _, s in qs], np.ones(E),
                               H, wfmt=oracle.WFMT_MXFP4)
    want = np.concatenate([h[off[e]:off[e + 1]] @ mx_dequant(*qs[e]).T for e in range(E)])
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)


def e4m3_power_of_two(j):
    """E4M3 code of 2^j for j in [-9, 8] (subnormal below 2^-6)."""
    return (j + 7) << 3 if j >= -6 else 1 << (j + 9)


@pytest.mark.parametrize("interleave", [0, 32])
def test_mxfp4_equals_nvfp4_with_the_same_powers_of_two(interleave):
    """MXFP4 scales written (by hand) as E4M3 powers of two for both 16-value
    halves, expert scale 1, give the NVFP4 path's results exactly."""
    shape = mi.MoEShape("mx", T=24, H=256, F=128, E=3, k=2, glu_interleave=interleave,
                        swiglu_clamp=7.0, lowprec=True)
    inp = mi.make_lowprec_inputs(shape, seed=2, wfmt="mxfp4")
    assert int(inp["w1s"].min()) >= 127 - 9 and int(inp["w1s"].max()) <= 127 + 8
    nv = {}
    for n in ("w1", "w2"):
        j = inp[n + "s"].to(torch.int64) - 127
        codes = torch.tensor([e4m3_power_of_two(int(v)) for v in j.flatten()],
                             dtype=torch.uint8).reshape(j.shape)
        nv[n + "s"] = codes.repeat_interleave(2, dim=-1)
    ones = torch.ones(shape.E)
    mx = oracle.moe_forward_lowprec(inp["xq"], inp["xs"], inp["logits"], inp["w1q"], inp["w1s"],
                                    ones, inp["w2q"], inp["w2s"], ones, shape.k,
                                    interleave=interleave, clamp=7.0, wfmt=oracle.WFMT_MXFP4)
    ref = oracle.moe_forward_lowprec(inp["xq"], inp["xs"], inp["logits"], inp["w1q"], nv["w1s"],
                                     ones, inp["w2q"], nv["w2s"], ones, shape.k,
                                     interleave=interleave, clamp=7.0)
    np.testing.assert_array_equal(mx["out"], ref["out"])


def test_mxfp4_quantiser_error_bound():
    g = torch.Generator().manual_seed(5)
    w = torch.randn(64, 256, generator=g) / 16
    q, s = mi.quantize_mxfp4(w)
    deq = mx_dequant(q, s)
    scale = np.ldexp(1.0, s.numpy().astype(np.int64) - 127).repeat(32, axis=1)
    err = np.abs(deq - w.double().numpy())
    # rounding at most half the largest E2M1 step (1 at the top, times the scale),
    # plus the clipping of magnitudes between 6 and 8 scale units
    assert (err <= np.maximum(1.0, np.abs(w.double().numpy()) / scale - 6.0) * scale + 1e-12).all()
    assert np.sqrt((err ** 2).mean() / (w.double().numpy() ** 2).mean()) < 0.15
