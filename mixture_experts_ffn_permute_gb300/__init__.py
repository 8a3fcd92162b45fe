"""Python binding of libmoeffn.so, the GB300 (sm_103a) MoE expert-FFN library.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.  The
function names mirror the C entry points of ``include/moe_ffn.h``:

    route_topk            -> moe_route_topk
    permute               -> moe_permute
    permute_rows          -> moe_permute_rows
    grouped_swiglu_mlp    -> moe_grouped_swiglu_mlp
    unpermute_combine     -> moe_unpermute_combine
    forward               -> moe_forward
    forward_routed        -> moe_forward_routed

There is no CPU fallback: if the library is missing or a call returns an
error status, a ``MoEError`` is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Dict, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoeffn.so")

MOE_OK = 0
FUSE_GATHER_A = 1   # GEMM1 gathers A rows from x with TMA gather4
FUSE_COMBINE = 2    # weighted top-k reduction in GEMM2's epilogue
KERNEL_AUTO = 0
KERNEL_TOKEN_TILES = 1   # 128 token rows x 256 weight rows per tile
KERNEL_WEIGHT_TILES = 2  # 128 weight rows x up to 32 token rows per tile (decode sizes)
KERNEL_WEIGHT_TILES_2CTA = 6  # 256 weight rows x up to 256 tokens per CTA pair, N fitted
KERNEL_DECODE_FUSED = 7  # moe_forward: both GEMMs and the combine of 32-token tiles in one launch
STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
    3: "MOE_ERR_MISALIGNED", 4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_CUDA",
    6: "MOE_ERR_DEVICE_TIMEOUT", 7: "MOE_ERR_DEVICE_INDEX",
}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


class Problem(ctypes.Structure):
    """Mirror of ``moe_problem``."""
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("F", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("glu_interleave", ctypes.c_int32),
                ("swiglu_clamp", ctypes.c_float), ("precision", ctypes.c_int32),
                ("fusion", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("shared_experts", ctypes.c_int32)]

    @classmethod
    def make(cls, T, H, F, E, k, renormalize=True, glu_interleave=0, swiglu_clamp=0.0,
             fusion=0, kernel=0, precision=0, shared_experts=0):
        return cls(int(T), int(H), int(F), int(E), int(k), int(bool(renormalize)),
                   int(glu_interleave), float(swiglu_clamp), int(precision), int(fusion),
                   int(kernel), int(shared_experts))


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmoeffn.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pp = ctypes.POINTER(Problem)
    sigs = {
        "moe_status_string": ([ci], ctypes.c_char_p),
        "moe_workspace_size": ([pp], sz),
        "moe_route_topk": ([pp, vp, vp, vp, vp, sz, vp], ci),
        "moe_permute": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ci),
        "moe_grouped_swiglu_mlp": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ci),
        "moe_permute_rows": ([pp, vp, vp, ctypes.c_int32, vp, vp], ci),
        "moe_unpermute_combine": ([pp, vp, vp, vp, vp, vp], ci),
        "moe_forward": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ci),
        "moe_forward_routed": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ci),
        "moe_selftest_wait_timeout": ([vp, ctypes.c_uint64, vp], ci),
        "moe_backward_workspace_size": ([pp], sz),
        "moe_backward": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ci),
        "moe_backward_routed": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp], ci),
        "moe_get_device_status": ([vp, vp], ci),
        "moe_clear_device_status": ([vp, vp], ci),
        "moe_last_launch_count": ([], ci),
        "moe_selected_kernel": ([pp], ci),
        "moe_stage_timing_begin": ([ci], ci),
        "moe_stage_timing_end": ([ctypes.POINTER(ctypes.c_float), ci,
                                  ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)], ci),
        "moe_stage_name": ([ci], ctypes.c_char_p),
        "moe_permute_noalloc": ([pp, vp, vp, vp, vp, vp, vp, vp, vp], ci),
        "moe_prepared_scales_size": ([pp], sz),
        "moe_prepare_weights": ([pp, vp, vp, vp, sz, vp], ci),
        "moe_prepare_weights_mxfp4": ([pp, vp, vp, vp, sz, vp, vp, vp], ci),
        "moe_forward_fp8_nvfp4": ([pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz,
                                   vp], ci),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if path is None:
        _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _call(name: str, *args):
    rc = getattr(load(), name)(*args)
    if rc != MOE_OK:
        raise MoEError(name, rc)


def workspace_size(p: Problem) -> int:
    return int(load().moe_workspace_size(ctypes.byref(p)))


def alloc_workspace(p: Problem, device="cuda") -> torch.Tensor:
    """A uint8 device tensor sized by moe_workspace_size (256-byte aligned)."""
    n = workspace_size(p)
    if n == 0:
        raise MoEError("moe_workspace_size", 1)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def selected_kernel(p: Problem) -> int:
    """The GEMM tiling (KERNEL_*) moe_forward picks for this problem."""
    return int(load().moe_selected_kernel(ctypes.byref(p)))


def last_launch_count() -> int:
    return int(load().moe_last_launch_count())


def stage_timing_begin(n_calls: int) -> None:
    _call("moe_stage_timing_begin", int(n_calls))


def stage_timing_end() -> Dict[str, float]:
    """Average milliseconds per moe_forward stage over the recorded calls."""
    ms = (ctypes.c_float * 16)()
    ns, nc = ctypes.c_int(0), ctypes.c_int(0)
    _call("moe_stage_timing_end", ms, 16, ctypes.byref(ns), ctypes.byref(nc))
    lib = load()
    res = {lib.moe_stage_name(i).decode(): float(ms[i]) for i in range(ns.value)}
    res["_calls"] = nc.value
    return res


def get_device_status(ws: torch.Tensor, stream=None) -> int:
    return int(load().moe_get_device_status(_ptr(ws), _stream(stream)))


def clear_device_status(ws: torch.Tensor, stream=None) -> None:
    _call("moe_clear_device_status", _ptr(ws), _stream(stream))


def route_topk(p: Problem, logits, topk_idx, topk_w, ws=None, stream=None) -> None:
    _call("moe_route_topk", ctypes.byref(p), _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
          _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream))


def permute(p: Problem, topk_idx, x, x_perm, row_id_map, permuted_token, tokens_per_expert,
            expert_offsets, ws, stream=None) -> None:
    _call("moe_permute", ctypes.byref(p), _ptr(topk_idx), _ptr(x), _ptr(x_perm),
          _ptr(row_id_map), _ptr(permuted_token), _ptr(tokens_per_expert),
          _ptr(expert_offsets), _ptr(ws), ws.numel(), _stream(stream))


def permute_noalloc(p: Problem, topk_idx, x, x_perm, row_id_map, permuted_token,
                    tokens_per_expert, expert_offsets, stream=None) -> None:
    """moe_permute without a workspace, for callers that cannot allocate device
    memory (e.g. while a stream is being captured): the library uses its own
    fixed 1 MiB device scratch.  Calls that may overlap on the GPU race."""
    _call("moe_permute_noalloc", ctypes.byref(p), _ptr(topk_idx), _ptr(x), _ptr(x_perm),
          _ptr(row_id_map), _ptr(permuted_token), _ptr(tokens_per_expert),
          _ptr(expert_offsets), _stream(stream))


class FP4Scales(ctypes.Structure):
    """Mirror of ``moe_fp4_scales``: device pointers to the prepared block
    scales and the per-expert fp32 scales of W1 and W2."""
    _fields_ = [("prepared", ctypes.c_void_p), ("w1_gscale", ctypes.c_void_p),
                ("w2_gscale", ctypes.c_void_p)]

    @classmethod
    def of(cls, prepared, w1_gscale, w2_gscale):
        return cls(prepared.data_ptr(), w1_gscale.data_ptr(), w2_gscale.data_ptr())


def _scales_ref(wscales):
    if wscales is None:
        return None
    if isinstance(wscales, (tuple, list)):
        wscales = FP4Scales.of(*wscales)
    return ctypes.byref(wscales)


def grouped_swiglu_mlp(p: Problem, x_perm, expert_offsets, w1, w2, y_perm, ws,
                       stream=None, x_perm_scale=None, wscales=None) -> None:
    """Steps 3-5 on permuted rows.  bf16: x_perm [R, H] bf16, w1/w2 bf16.
    FP8/NVFP4 (p.precision = PREC_FP8_NVFP4): x_perm [R, H] E4M3 codes (uint8),
    x_perm_scale [R, H/128] fp32, w1/w2 packed E2M1 codes and wscales =
    (prepared, w1_gscale, w2_gscale) tensors or an FP4Scales."""
    _call("moe_grouped_swiglu_mlp", ctypes.byref(p), _ptr(x_perm), _ptr(x_perm_scale),
          _ptr(expert_offsets), _ptr(w1), _ptr(w2), _scales_ref(wscales), _ptr(y_perm), _ptr(ws),
          ws.numel(), _stream(stream))


def permute_rows(p: Problem, permuted_token, src, dst, stream=None) -> None:
    """dst[r] = src[permuted_token[r]] for rows of any width (a multiple of 4
    bytes); zero rows for -1.  src [T, ...], dst [T*k, ...] of one dtype."""
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else 0
    if dst.shape[0] != p.T * p.k or dst[0].numel() * dst.element_size() != row_bytes:
        raise ValueError("dst must hold T*k rows of src's row width")
    _call("moe_permute_rows", ctypes.byref(p), _ptr(permuted_token), _ptr(src),
          int(row_bytes), _ptr(dst), _stream(stream))


def unpermute_combine(p: Problem, y_perm, row_id_map, topk_w, out, stream=None) -> None:
    _call("moe_unpermute_combine", ctypes.byref(p), _ptr(y_perm), _ptr(row_id_map),
          _ptr(topk_w), _ptr(out), _stream(stream))


def forward(p: Problem, x, logits, w1, w2, out, ws, topk_idx=None, topk_w=None,
            tokens_per_expert=None, stream=None, x_scale=None, wscales=None) -> None:
    """The whole layer.  bf16: x bf16, w1/w2 bf16.  FP8/NVFP4 (p.precision =
    PREC_FP8_NVFP4): x E4M3 codes, x_scale [T, H/128] fp32, w1/w2 packed E2M1
    codes, wscales = (prepared, w1_gscale, w2_gscale) or an FP4Scales."""
    _call("moe_forward", ctypes.byref(p), _ptr(x), _ptr(x_scale), _ptr(logits), _ptr(w1),
          _ptr(w2), _scales_ref(wscales), _ptr(out), _ptr(topk_idx), _ptr(topk_w),
          _ptr(tokens_per_expert), _ptr(ws), ws.numel(), _stream(stream))


def forward_routed(p: Problem, x, topk_idx, topk_w, w1, w2, out, ws, tokens_per_expert=None,
                   stream=None) -> None:
    """The layer with caller-supplied routing (int32 [T, k], -1 = masked; fp32 [T, k])."""
    _call("moe_forward_routed", ctypes.byref(p), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(w1),
          _ptr(w2), _ptr(out), _ptr(tokens_per_expert), _ptr(ws), ws.numel(), _stream(stream))


def backward_workspace_size(p: Problem) -> int:
    return int(load().moe_backward_workspace_size(ctypes.byref(p)))


def alloc_backward_workspace(p: Problem, device="cuda") -> torch.Tensor:
    """A uint8 device tensor sized by moe_backward_workspace_size (256-byte aligned)."""
    n = backward_workspace_size(p)
    if n == 0:
        raise MoEError("moe_backward_workspace_size", 1)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    return ws[off:off + n]


def backward(p: Problem, x, logits, w1, w2, d_out, dx, dw1, dw2, ws, d_logits=None,
             stream=None) -> None:
    """Gradients of the layer given d_out = dL/d out: dx [T, H] bf16,
    d_logits [T, E] fp32 (optional), dw1 / dw2 bf16 in the weights' shapes."""
    _call("moe_backward", ctypes.byref(p), _ptr(x), _ptr(logits), _ptr(w1), _ptr(w2),
          _ptr(d_out), _ptr(dx), _ptr(d_logits), _ptr(dw1), _ptr(dw2), _ptr(ws), ws.numel(),
          _stream(stream))


def backward_routed(p: Problem, x, topk_idx, topk_w, w1, w2, d_out, dx, dw1, dw2, ws,
                    d_topk_w=None, stream=None) -> None:
    """Gradients of the layer with caller-supplied routing (int32 [T, k], -1 =
    masked; fp32 [T, k]): dx, dw1, dw2 and, optionally, d_topk_w [T, k] fp32."""
    _call("moe_backward_routed", ctypes.byref(p), _ptr(x), _ptr(topk_idx), _ptr(topk_w),
          _ptr(w1), _ptr(w2), _ptr(d_out), _ptr(dx), _ptr(d_topk_w), _ptr(dw1), _ptr(dw2),
          _ptr(ws), ws.numel(), _stream(stream))


def selftest_wait_timeout(ws, limit_ns: int, stream=None) -> None:
    """Run the bounded-wait self-test: a wait that runs out after limit_ns and
    records MOE_ERR_DEVICE_TIMEOUT in ws's status word."""
    _call("moe_selftest_wait_timeout", _ptr(ws), int(limit_ns), _stream(stream))


PREC_BF16 = 0
PREC_FP8_NVFP4 = 1


def prepared_scales_size(p: Problem) -> int:
    return int(load().moe_prepared_scales_size(ctypes.byref(p)))


def prepare_weights(p: Problem, w1_scale, w2_scale, prepared, stream=None) -> None:
    """Re-lay NVFP4 block scales into the order the low-precision kernels stream them."""
    _call("moe_prepare_weights", ctypes.byref(p), _ptr(w1_scale), _ptr(w2_scale), _ptr(prepared),
          prepared.numel() * prepared.element_size(), _stream(stream))


def prepare_weights_mxfp4(p: Problem, w1_scale, w2_scale, prepared, w1_gscale, w2_gscale,
                          stream=None) -> None:
    """Re-encode MXFP4 E8M0 scales for forward_fp8_nvfp4 (prepared scales and the
    per-expert fp32 scales w1_gscale / w2_gscale, both written)."""
    _call("moe_prepare_weights_mxfp4", ctypes.byref(p), _ptr(w1_scale), _ptr(w2_scale),
          _ptr(prepared), prepared.numel() * prepared.element_size(), _ptr(w1_gscale),
          _ptr(w2_gscale), _stream(stream))


def forward_fp8_nvfp4(p: Problem, xq, xs, logits, w1q, w1_gscale, w2q, w2_gscale, prepared,
                      out, ws, topk_idx=None, topk_w=None, tokens_per_expert=None,
                      stream=None) -> None:
    _call("moe_forward_fp8_nvfp4", ctypes.byref(p), _ptr(xq), _ptr(xs), _ptr(logits), _ptr(w1q),
          _ptr(w1_gscale), _ptr(w2q), _ptr(w2_gscale), _ptr(prepared), _ptr(out), _ptr(topk_idx),
          _ptr(topk_w), _ptr(tokens_per_expert), _ptr(ws), ws.numel(), _stream(stream))


class MoEFFN:
    """Convenience holder: weights + a reusable workspace for one problem size."""

    def __init__(self, w1: torch.Tensor, w2: torch.Tensor, k: int, renormalize=True,
                 glu_interleave=0, swiglu_clamp=0.0):
        E, twoF, H = w1.shape
        self.w1, self.w2 = w1, w2
        self.H, self.F, self.E, self.k = H, twoF // 2, E, k
        self.renormalize, self.glu_interleave, self.swiglu_clamp = (
            renormalize, glu_interleave, swiglu_clamp)
        self._ws = None
        self._ws_T = -1

    def problem(self, T: int) -> Problem:
        return Problem.make(T, self.H, self.F, self.E, self.k, self.renormalize,
                            self.glu_interleave, self.swiglu_clamp)

    def __call__(self, x: torch.Tensor, logits: torch.Tensor,
                 return_routing: bool = False) -> Dict[str, torch.Tensor]:
        T = x.shape[0]
        p = self.problem(T)
        if self._ws is None or T > self._ws_T:
            self._ws = alloc_workspace(p, device=x.device)
            self._ws_T = T
        out = torch.empty(T, self.H, dtype=torch.bfloat16, device=x.device)
        res = {"out": out}
        if return_routing:
            res["topk_idx"] = torch.empty(T, self.k, dtype=torch.int32, device=x.device)
            res["topk_w"] = torch.empty(T, self.k, dtype=torch.float32, device=x.device)
            res["tokens_per_expert"] = torch.empty(self.E, dtype=torch.int32, device=x.device)
        forward(p, x, logits, self.w1, self.w2, out, self._ws, res.get("topk_idx"),
                res.get("topk_w"), res.get("tokens_per_expert"))
        return res

    def backward(self, x: torch.Tensor, logits: torch.Tensor,
                 d_out: torch.Tensor) -> Dict[str, torch.Tensor]:
        """Gradients of the layer given d_out = dL/d out (moe_backward): dx, dlogits,
        dw1, dw2.  The forward's intermediates are recomputed from x and logits."""
        T = x.shape[0]
        p = self.problem(T)
        if getattr(self, "_bws", None) is None or T > self._bws_T:
            self._bws = alloc_backward_workspace(p, device=x.device)
            self._bws_T = T
        res = {"dx": torch.empty_like(x),
               "dlogits": torch.empty(T, self.E, dtype=torch.float32, device=x.device),
               "dw1": torch.empty_like(self.w1), "dw2": torch.empty_like(self.w2)}
        backward(p, x, logits, self.w1, self.w2, d_out, res["dx"], res["dw1"], res["dw2"],
                 self._bws, d_logits=res["dlogits"])
        return res


__all__ = ["Problem", "MoEError", "MoEFFN", "load", "workspace_size", "alloc_workspace",
           "route_topk", "permute", "permute_rows", "grouped_swiglu_mlp", "unpermute_combine",
           "forward", "FP4Scales",
           "get_device_status", "clear_device_status", "last_launch_count", "LIB_PATH",
           "stage_timing_begin", "stage_timing_end", "permute_noalloc",
           "prepared_scales_size", "prepare_weights", "forward_fp8_nvfp4", "selected_kernel",
           "forward_routed", "prepare_weights_mxfp4", "selftest_wait_timeout",
           "backward_workspace_size", "alloc_backward_workspace", "backward", "backward_routed"]
