"""CPU checks of the C ABI: the library loads without a GPU, exports every
entry point include/moe_ffn.h declares, and rejects bad arguments on the
host before any CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import mixture_experts_ffn_permute_gb300 as moe
from mixture_experts_ffn_permute_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return moe.load()


def declared_symbols():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert "moe_forward" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code, name in moe.STATUS_NAMES.items():
        assert lib.moe_status_string(code).decode() == name


def fwd(lib, p, x, lg, w1, w2, out, ws, nbytes, x_scale=None, wscales=None):
    """moe_forward with no routing copies and the default stream."""
    return lib.moe_forward(p, x, x_scale, lg, w1, w2, wscales, out, None, None, None, ws, nbytes,
                           None)


def P(**kw):
    base = dict(T=64, H=256, F=512, E=8, k=2)
    base.update(kw)
    return moe.Problem.make(**base)


def test_workspace_size_grows_with_tokens(lib):
    a = moe.workspace_size(P(T=64))
    b = moe.workspace_size(P(T=128))
    assert 0 < a < b
    assert a % 256 == 0
    # at least the three permuted activations: x_perm, h, y (bf16)
    R = 64 * 2
    assert a >= 2 * R * (256 + 512 + 256)


@pytest.mark.parametrize("kw,code", [
    (dict(k=9), 1), (dict(k=0), 1), (dict(E=0), 1), (dict(T=-1), 1),
    (dict(H=200), 2), (dict(F=100), 2), (dict(E=2000, k=2), 2), (dict(k=33, E=64), 2),
    (dict(glu_interleave=48), 2), (dict(glu_interleave=-1), 1), (dict(glu_interleave=1024), 2),
])
def test_forward_rejects_bad_problems(lib, kw, code):
    p = P(**kw)
    fake = ctypes.c_void_p(1 << 20)
    rc = fwd(lib, ctypes.byref(p), fake, fake, fake, fake, fake, fake, 1 << 40)
    assert rc == code


def test_forward_rejects_bad_pointers_and_workspace(lib):
    p = P()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 8)
    big = 1 << 40
    ws_need = moe.workspace_size(p)
    assert fwd(lib, ctypes.byref(p), None, a, a, a, a, a, big) == 1
    assert fwd(lib, ctypes.byref(p), mis, a, a, a, a, a, big) == 3
    # workspace must be 256-byte aligned and large enough
    ws_mis = ctypes.c_void_p((1 << 20) + 16)
    assert fwd(lib, ctypes.byref(p), a, a, a, a, a, ws_mis, big) == 3
    assert fwd(lib, ctypes.byref(p), a, a, a, a, a, a, ws_need - 1) == 4
    assert fwd(lib, None, a, a, a, a, a, a, big) == 1


def test_other_entry_points_validate(lib):
    p = P()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    assert lib.moe_route_topk(ctypes.byref(P(k=9)), a, a, a, None, 0, None) == 1
    assert lib.moe_route_topk(ctypes.byref(p), mis, a, a, None, 0, None) == 3
    assert lib.moe_permute(ctypes.byref(p), a, None, None, a, a, None, a, a, 1 << 30, None) == 1
    assert lib.moe_grouped_swiglu_mlp(ctypes.byref(P(F=96)), a, None, a, a, a, None, a, a,
                                      1 << 40, None) == 2
    assert lib.moe_unpermute_combine(ctypes.byref(P(H=12)), a, a, a, a, None) == 2
    assert lib.moe_get_device_status(None, None) == 1


def test_binding_raises_without_library(tmp_path):
    with pytest.raises(ImportError):
        moe.load(str(tmp_path / "missing.so"))


def test_auto_tiling_selection():
    """Auto picks the one-launch decode MLP below 1 route per expert, the two-GEMM 32-token
    weight-row tiles up to 2, else 2-CTA weight-row tiles."""
    lib = moe.load()
    assert moe.selected_kernel(moe.Problem.make(T=1, H=2048, F=768, E=128, k=8)) == \
        moe.KERNEL_DECODE_FUSED
    assert moe.selected_kernel(moe.Problem.make(T=15, H=2048, F=768, E=128, k=8)) == \
        moe.KERNEL_DECODE_FUSED
    assert moe.selected_kernel(moe.Problem.make(T=16, H=2048, F=768, E=128, k=8)) == \
        moe.KERNEL_WEIGHT_TILES
    assert moe.selected_kernel(moe.Problem.make(T=32, H=2048, F=768, E=128, k=8)) == \
        moe.KERNEL_WEIGHT_TILES
    p = moe.Problem.make(T=8, H=2048, F=768, E=128, k=8, kernel=moe.KERNEL_WEIGHT_TILES)
    assert moe.selected_kernel(p) == moe.KERNEL_WEIGHT_TILES
    assert moe.selected_kernel(moe.Problem.make(T=64, H=2048, F=768, E=128, k=8)) == \
        moe.KERNEL_WEIGHT_TILES_2CTA
    assert moe.selected_kernel(moe.Problem.make(T=4096, H=4096, F=14336, E=8, k=2)) == \
        moe.KERNEL_WEIGHT_TILES_2CTA
    p = moe.Problem.make(T=4096, H=4096, F=14336, E=8, k=2, kernel=moe.KERNEL_TOKEN_TILES)
    assert moe.selected_kernel(p) == moe.KERNEL_TOKEN_TILES
    for dropped in (3, 4, 5, 8):  # tiling numbers that are not built
        p = moe.Problem.make(T=4096, H=4096, F=14336, E=8, k=2, kernel=dropped)
        assert moe.selected_kernel(p) == -1
    assert lib is not None


def test_lowprec_tiling_selection():
    """FP8/NVFP4: token-row tiles by default; 2-CTA weight-row tiles on request; no others."""
    moe.load()
    mk = lambda kernel: moe.Problem.make(T=4096, H=7168, F=2048, E=256, k=8, glu_interleave=32,  # noqa: E731
                                         swiglu_clamp=7.0, precision=moe.PREC_FP8_NVFP4,
                                         kernel=kernel)
    assert moe.selected_kernel(mk(moe.KERNEL_AUTO)) == moe.KERNEL_TOKEN_TILES
    assert moe.selected_kernel(mk(moe.KERNEL_WEIGHT_TILES_2CTA)) == moe.KERNEL_WEIGHT_TILES_2CTA
    assert moe.selected_kernel(mk(moe.KERNEL_TOKEN_TILES)) == moe.KERNEL_TOKEN_TILES
    for k in (moe.KERNEL_WEIGHT_TILES, 3, 4, 5, moe.KERNEL_DECODE_FUSED):
        assert moe.selected_kernel(mk(k)) == -1


def test_forward_routed_validates(lib):
    p = P()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    big = 1 << 40
    f = lib.moe_forward_routed
    assert f(ctypes.byref(p), a, None, a, a, a, a, None, a, big, None) == 1   # topk_idx
    assert f(ctypes.byref(p), a, a, None, a, a, a, None, a, big, None) == 1   # topk_w
    assert f(ctypes.byref(p), a, mis, a, a, a, a, None, a, big, None) == 3
    assert f(ctypes.byref(p), a, a, a, a, a, a, None, a, moe.workspace_size(p) - 1, None) == 4
    lp = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, precision=moe.PREC_FP8_NVFP4)
    assert f(ctypes.byref(lp), a, a, a, a, a, a, None, a, big, None) == 1    # bf16 only


def test_shared_experts_validation_and_workspace():
    """Shared experts: moe_forward only; k+S and E+S within the limits; the
    workspace grows with the k+S slots."""
    lib = moe.load()
    a = ctypes.c_void_p(1 << 20)
    big = 1 << 40
    p0 = moe.Problem.make(T=64, H=256, F=512, E=8, k=2)
    p1 = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, shared_experts=1)
    assert moe.workspace_size(p1) > moe.workspace_size(p0)
    assert lib.moe_route_topk(ctypes.byref(p1), a, a, a, a, big, None) == 1
    assert lib.moe_forward_routed(ctypes.byref(p1), a, a, a, a, a, a, None, a, big, None) == 1
    bad = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, shared_experts=-1)
    assert moe.workspace_size(bad) == 0
    too_many = moe.Problem.make(T=64, H=256, F=512, E=8, k=8, shared_experts=25)
    assert fwd(lib, ctypes.byref(too_many), a, a, a, a, a, a, big) == 2


def test_selftest_wait_timeout_validates(lib):
    a = ctypes.c_void_p(1 << 20)
    f = lib.moe_selftest_wait_timeout
    assert f(None, 1000, None) == 1
    assert f(a, 0, None) == 1
    assert f(a, 3 * 10**9, None) == 1   # above the library's own 2 s wait limit


def test_prepare_weights_mxfp4_validates(lib):
    a = ctypes.c_void_p(1 << 20)
    big = 1 << 40
    p = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, precision=moe.PREC_FP8_NVFP4)
    f = lib.moe_prepare_weights_mxfp4
    assert f(ctypes.byref(p), a, a, a, big, None, a, None) == 1
    assert f(ctypes.byref(p), a, a, a, moe.prepared_scales_size(p) - 1, a, a, None) == 4
    bf = moe.Problem.make(T=64, H=256, F=512, E=8, k=2)
    assert f(ctypes.byref(bf), a, a, a, big, a, a, None) == 1


def test_backward_validates(lib):
    """moe_backward's host checks (no GPU work is enqueued on any of these)."""
    p = P()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    big = 1 << 40
    f = lib.moe_backward
    need = moe.backward_workspace_size(p)
    assert need > moe.workspace_size(p)  # adds the pre-activations and router partials
    assert f(ctypes.byref(p), a, a, a, a, a, a, a, a, a, a, need - 1, None) == 4
    assert f(ctypes.byref(p), a, a, a, a, a, a, a, a, a, None, big, None) == 1      # ws
    assert f(ctypes.byref(p), a, a, a, a, a, a, a, None, a, a, big, None) == 1      # dw1
    assert f(ctypes.byref(p), a, a, a, a, a, a, a, a, mis, a, big, None) == 3      # dw2
    assert f(ctypes.byref(p), a, a, a, a, a, a, mis, a, a, a, big, None) == 3      # d_logits
    assert f(ctypes.byref(p), a, a, a, a, None, a, a, a, a, a, big, None) == 1     # d_out
    assert f(ctypes.byref(P(H=200)), a, a, a, a, a, a, a, a, a, a, big, None) == 2
    lp = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, precision=moe.PREC_FP8_NVFP4)
    assert f(ctypes.byref(lp), a, a, a, a, a, a, a, a, a, a, big, None) == 1        # bf16 only
    assert moe.backward_workspace_size(lp) == 0
    # shared experts widen the workspace like the forward's
    ps = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, shared_experts=1)
    assert moe.backward_workspace_size(ps) > need


def test_backward_routed_validates(lib):
    p = P()
    a = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 4)
    big = 1 << 40
    f = lib.moe_backward_routed
    need = moe.backward_workspace_size(p)
    assert f(ctypes.byref(p), a, None, a, a, a, a, a, a, a, a, a, big, None) == 1    # topk_idx
    assert f(ctypes.byref(p), a, a, None, a, a, a, a, a, a, a, a, big, None) == 1    # topk_w
    assert f(ctypes.byref(p), a, a, a, a, a, a, a, mis, a, a, a, big, None) == 3     # d_topk_w
    assert f(ctypes.byref(p), a, a, a, a, a, a, a, a, a, a, a, need - 1, None) == 4
    ps = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, shared_experts=1)
    assert f(ctypes.byref(ps), a, a, a, a, a, a, a, a, a, a, a, big, None) == 1      # no shared


def test_lowprec_stage_forms_validate(lib):
    """moe_grouped_swiglu_mlp and moe_forward take FP8/NVFP4 operands with their
    scales; bf16 calls must pass no scales; moe_permute_rows checks its width."""
    a = ctypes.c_void_p(1 << 20)
    big = 1 << 40
    lp = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, precision=moe.PREC_FP8_NVFP4)
    bf = P()
    sc = moe.FP4Scales(1 << 20, 1 << 20, 1 << 20)
    bad_sc = moe.FP4Scales(1 << 20, None, 1 << 20)
    mlp = lib.moe_grouped_swiglu_mlp
    # FP8: the scales struct is required and checked
    assert mlp(ctypes.byref(lp), a, a, a, a, a, None, a, a, big, None) == 1
    assert mlp(ctypes.byref(lp), a, a, a, a, a, ctypes.byref(bad_sc), a, a, big, None) == 1
    assert mlp(ctypes.byref(lp), a, None, a, a, a, ctypes.byref(sc), a, a, big, None) == 1
    ws_need = moe.workspace_size(lp)
    assert mlp(ctypes.byref(lp), a, a, a, a, a, ctypes.byref(sc), a, a, ws_need - 1, None) == 4
    # bf16: no scales
    assert mlp(ctypes.byref(bf), a, a, a, a, a, None, a, a, big, None) == 1
    assert mlp(ctypes.byref(bf), a, None, a, a, a, ctypes.byref(sc), a, a, big, None) == 1
    # the whole layer
    assert fwd(lib, ctypes.byref(lp), a, a, a, a, a, a, big) == 1           # no wscales
    assert fwd(lib, ctypes.byref(lp), a, a, a, a, a, a, big, None, ctypes.byref(sc)) == 1
    assert fwd(lib, ctypes.byref(bf), a, a, a, a, a, a, big, a) == 1        # bf16 with x_scale
    shared = moe.Problem.make(T=64, H=256, F=512, E=8, k=2, shared_experts=1,
                              precision=moe.PREC_FP8_NVFP4)
    assert fwd(lib, ctypes.byref(shared), a, a, a, a, a, a, big, a, ctypes.byref(sc)) == 1
    # row gather: a positive multiple of 4 bytes
    rows = lib.moe_permute_rows
    assert rows(ctypes.byref(bf), a, a, 6, a, None) == 2
    assert rows(ctypes.byref(bf), a, a, 0, a, None) == 2
    assert rows(ctypes.byref(bf), None, a, 8, a, None) == 1
    assert rows(ctypes.byref(bf), a, a, 8, ctypes.c_void_p((1 << 20) + 4), None) == 3
