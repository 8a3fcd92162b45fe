"""Comparison helpers shared by the GPU parity tests.

Floating-point contract (bf16 path): per element
    |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|
and over the whole tensor
    RMS relative error sqrt(sum (gpu - oracle)^2 / sum oracle^2) <= 5e-3.
Routing indices, row maps and counts are compared bit for bit.

Gradients (the backward): each output is a sum of products in which exactly
one factor was rounded to bf16 (relative error <= 2^-9) and the result is
rounded once more to bf16 (<= 2^-9 of its value); fp32 accumulation adds far
less.  So per element
    |gpu - oracle| <= 2^-7 * M
where M is the oracle's sum of the absolute values of that element's terms
(the dot-product error bound, with a factor 2 to spare), and over the whole
tensor the RMS relative error <= 5e-3.
"""
import numpy as np
import torch

ATOL = 1e-2
RTOL = 1e-2
RMS_BF16 = 5e-3


def to_f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to(torch.float64).cpu().numpy()
    return np.asarray(t, np.float64)


def rms_rel(gpu: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.sum(ref * ref))
    num = float(np.sum((gpu - ref) ** 2))
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return (num / den) ** 0.5


def assert_bf16_close(gpu, ref, what: str = "", rms: float = RMS_BF16):
    g = to_f64(gpu)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"gpu={g[i]!r} oracle={r[i]!r}")
    e = rms_rel(g, r)
    assert e <= rms, f"{what}: RMS relative error {e:.3e} > {rms:.1e}"
    return e


def assert_equal(gpu, ref, what: str = ""):
    g = gpu.detach().cpu().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu)
    r = np.asarray(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    if not np.array_equal(g, r):
        d = np.argwhere(g != r)
        raise AssertionError(f"{what}: {len(d)} mismatches, first at {tuple(d[0])}: "
                             f"gpu={g[tuple(d[0])]} oracle={r[tuple(d[0])]}")



TAU_GRAD = 2.0 ** -7


def assert_grad_bound(gpu, ref, mag, what: str = "", rms: float = RMS_BF16, tau: float = TAU_GRAD):
    """Gradient parity: per element within tau times the magnitude of its
    terms (``mag``, from the oracle), and RMS relative error <= rms."""
    g = to_f64(gpu)
    r = np.asarray(ref, np.float64)
    m = np.asarray(mag, np.float64)
    assert g.shape == r.shape == m.shape, (what, g.shape, r.shape, m.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - r)
    bound = tau * m
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"gpu={g[i]!r} oracle={r[i]!r} magnitude={m[i]!r}")
    e = rms_rel(g, r)
    assert e <= rms, f"{what}: RMS relative error {e:.3e} > {rms:.1e}"
    return e


def tile_sample_tokens(perm, tile_rows: int = 256) -> np.ndarray:
    """Tokens whose outputs a full-size parity test compares, chosen from the
    oracle's permutation (never from the GPU's) so that every tile kind the
    kernels run at full size is reached: for every expert with rows, the
    token at its first permuted row and at the last row of each of its
    tile_rows-row token tiles (the last one being the expert's ragged tail).
    Sorted, without repeats."""
    off = np.asarray(perm["expert_offsets"])
    ptok = np.asarray(perm["permuted_token"])
    rows = []
    for e in range(len(off) - 1):
        a, b = int(off[e]), int(off[e + 1])
        if b <= a:
            continue
        rows.append(a)
        for t0 in range(a, b, tile_rows):
            rows.append(min(b, t0 + tile_rows) - 1)
    toks = ptok[np.asarray(rows, np.int64)]
    return np.unique(toks[toks >= 0]).astype(np.int64)
