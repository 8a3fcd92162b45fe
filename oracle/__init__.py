"""ctypes front-end of the fp64 CPU oracle (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and the oracle never imports the product.

Each wrapper below mirrors one C function of ``moe_oracle.cpp``; the C source
documents the definition it follows.  Inputs are torch tensors or numpy
arrays; bf16 tensors are passed as their raw bit patterns and widened exactly
inside the oracle.  Results are float64 / int32 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP, -O2, no fast-math) if needed."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["g++", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c++17",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp = ctypes.c_void_p
            ci, cl, cd = ctypes.c_int, ctypes.c_long, ctypes.c_double
            sig = {
                "oracle_num_threads": ([], ci),
                "oracle_set_num_threads": ([ci], ci),
                "oracle_bf16_value": ([ctypes.c_uint16], cd),
                "oracle_route_topk": ([ci, ci, ci, ci, vp, vp, vp], ci),
                "oracle_permute": ([ci, ci, ci, vp, vp, vp, vp, vp], ci),
                "oracle_gather_rows": ([cl, ci, vp, vp, vp], ci),
                "oracle_gemm1_swiglu": ([cl, ci, ci, ci, ci, cd, vp, vp, vp, vp], ci),
                "oracle_gemm2": ([cl, ci, ci, ci, vp, vp, vp, vp], ci),
                "oracle_unpermute_combine": ([ci, ci, ci, vp, vp, vp, vp], ci),
                "oracle_moe_forward": ([ci, ci, ci, ci, ci, ci, ci, cd, vp, vp, vp, vp,
                                        vp, vp, vp, vp], ci),
                "oracle_dense_bruteforce": ([ci, ci, ci, ci, ci, ci, cd, vp, vp, vp, vp,
                                             vp, vp], ci),
                "oracle_e4m3_value": ([ctypes.c_uint8], cd),
                "oracle_e2m1_value": ([ctypes.c_uint8], cd),
                "oracle_e8m0_value": ([ctypes.c_uint8], cd),
                "oracle_e4m3_encode": ([ctypes.c_float], ctypes.c_uint8),
                "oracle_requant_fp8_block": ([vp, ci, vp], None),
                "oracle_gemm1_swiglu_lowprec": ([cl, ci, ci, ci, ci, cd, vp, vp, vp, vp, vp, vp,
                                                 ci, ci, vp], ci),
                "oracle_gemm2_lowprec": ([cl, ci, ci, ci, vp, vp, vp, vp, vp, ci, vp], ci),
                "oracle_moe_forward_lowprec": ([ci, ci, ci, ci, ci, ci, ci, cd, vp, vp, vp, vp,
                                                vp, vp, vp, vp, vp, ci, vp, vp, vp], ci),
                "oracle_moe_backward": ([ci, ci, ci, ci, ci, ci, cd, ci, ci, vp, vp, vp, vp,
                                         vp, vp, vp, vp, vp, vp], ci),
                "oracle_backward_tokens": ([ci, ci, ci, ci, ci, ci, cd, ci, ci, vp, vp, vp, vp,
                                            vp, vp, ci, vp, vp, vp], ci),
                "oracle_backward_dw1_rows": ([ci, ci, ci, ci, ci, ci, cd, ci, ci, vp, vp, vp,
                                              vp, vp, vp, ci, vp, vp], ci),
                "oracle_backward_dw2_cols": ([ci, ci, ci, ci, ci, ci, cd, ci, ci, vp, vp, vp,
                                              vp, vp, ci, vp, vp], ci),
                "oracle_router_backward": ([ci, ci, ci, ci, ci, ci, vp, vp, vp, vp, vp], ci),
            }
            for name, (args, res) in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


# ---------------------------------------------------------------- helpers

def _np(a, dtype) -> np.ndarray:
    """Contiguous numpy copy/view of a torch tensor or array with ``dtype``."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu()
            if a.dtype == torch.bfloat16:
                a = a.contiguous().view(torch.int16).numpy().view(np.uint16)
            else:
                a = a.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        if np.dtype(dtype) == np.uint16:
            raise TypeError("bf16 operands must be passed as bf16 tensors or uint16 bits")
        a = np.ascontiguousarray(a.astype(dtype))
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _expert_ptrs(ws: Sequence[Optional[np.ndarray]]):
    arr = (ctypes.c_void_p * len(ws))()
    for i, w in enumerate(ws):
        arr[i] = None if w is None else w.ctypes.data
    return arr


def _experts(w, E: int):
    """Per-expert bf16 bit arrays from a [E, ...] tensor or a list (None = unused)."""
    if isinstance(w, (list, tuple)):
        assert len(w) == E
        return [None if m is None else _np(m, np.uint16) for m in w]
    a = _np(w, np.uint16)
    return [a[e] for e in range(E)]


def _check(rc: int, name: str):
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments (code {rc})")


# ---------------------------------------------------------------- API

def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> int:
    return _load().oracle_set_num_threads(int(n))


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(int(bits))


def route_topk(logits, k: int, renormalize: bool = True):
    lg = _np(logits, np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(_load().oracle_route_topk(T, E, k, int(renormalize), _p(lg), _p(idx), _p(w)),
           "oracle_route_topk")
    return idx, w


def permute(topk_idx, E: int) -> Dict[str, np.ndarray]:
    ix = _np(topk_idx, np.int32)
    T, k = ix.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    rmap = np.empty((T, k), np.int32)
    ptok = np.empty(T * k, np.int32)
    _check(_load().oracle_permute(T, E, k, _p(ix), _p(counts), _p(offsets), _p(rmap), _p(ptok)),
           "oracle_permute")
    return {"tokens_per_expert": counts, "expert_offsets": offsets,
            "row_id_map": rmap, "permuted_token": ptok}


def gather_rows(x, permuted_token) -> np.ndarray:
    xb = _np(x, np.uint16)
    pt = _np(permuted_token, np.int32)
    R, H = pt.shape[0], xb.shape[1]
    out = np.empty((R, H), np.uint16)
    _load().oracle_gather_rows(R, H, _p(xb), _p(pt), _p(out))
    return out


def gemm1_swiglu(x_perm, expert_offsets, w1, F: int, interleave: int = 0,
                 clamp: float = 0.0) -> np.ndarray:
    xp = _np(x_perm, np.uint16)
    off = _np(expert_offsets, np.int32)
    E = off.shape[0] - 1
    R, H = xp.shape
    ws = _experts(w1, E)
    ptrs = _expert_ptrs(ws)
    h = np.empty((R, F), np.float64)
    _check(_load().oracle_gemm1_swiglu(R, H, F, E, interleave, float(clamp), _p(off), _p(xp),
                                       ptrs, _p(h)), "oracle_gemm1_swiglu")
    return h


def gemm2(h, expert_offsets, w2, H: int) -> np.ndarray:
    hh = _np(h, np.float64)
    off = _np(expert_offsets, np.int32)
    E = off.shape[0] - 1
    R, F = hh.shape
    ws = _experts(w2, E)
    ptrs = _expert_ptrs(ws)
    y = np.empty((R, H), np.float64)
    _check(_load().oracle_gemm2(R, H, F, E, _p(off), _p(hh), ptrs, _p(y)), "oracle_gemm2")
    return y


def unpermute_combine(y, row_id_map, topk_w) -> np.ndarray:
    yy = _np(y, np.float64)
    rm = _np(row_id_map, np.int32)
    ww = _np(topk_w, np.float64)
    T, k = rm.shape
    H = yy.shape[1]
    out = np.empty((T, H), np.float64)
    _load().oracle_unpermute_combine(T, H, k, _p(yy), _p(rm), _p(ww), _p(out))
    return out


def moe_forward(x, logits, w1, w2, k: int, renormalize: bool = True, interleave: int = 0,
                clamp: float = 0.0) -> Dict[str, np.ndarray]:
    """The whole layer on the given tokens.  ``w1``/``w2`` are [E, ...] tensors or
    per-expert lists where unused experts may be None."""
    xb = _np(x, np.uint16)
    lg = _np(logits, np.float32)
    T, H = xb.shape
    E = lg.shape[1]
    w1s, w2s = _experts(w1, E), _experts(w2, E)
    F = next(m for m in w2s if m is not None).shape[1]
    out = np.empty((T, H), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    counts = np.empty(E, np.int32)
    _check(_load().oracle_moe_forward(T, H, F, E, k, int(renormalize), interleave, float(clamp),
                                      _p(lg), _p(xb), _expert_ptrs(w1s), _expert_ptrs(w2s),
                                      _p(out), _p(idx), _p(w), _p(counts)),
           "oracle_moe_forward")
    return {"out": out, "topk_idx": idx, "topk_w": w, "tokens_per_expert": counts}


def moe_forward_routed(x, topk_idx, topk_w, w1, w2, interleave: int = 0, clamp: float = 0.0):
    """The layer with the routing given (steps 2-6 of the MegaMoE page's
    Usage: staged top-k indices with -1 for a masked route and FP32 weights),
    composed from the stage functions above in their order.  Returns out
    (fp64) and the permutation."""
    idx = _np(topk_idx, np.int32)
    if isinstance(w1, (list, tuple)):  # per-expert arrays, None for experts never routed to
        E = len(w1)
        F = next(w for w in w1 if w is not None).shape[0] // 2
    else:
        E, F = int(w1.shape[0]), int(w1.shape[1]) // 2
    perm = permute(idx, E)
    xp = gather_rows(x, perm["permuted_token"])
    h = gemm1_swiglu(xp, perm["expert_offsets"], w1, F, interleave=interleave, clamp=clamp)
    H = xp.shape[1]
    y = gemm2(h, perm["expert_offsets"], w2, H)
    out = unpermute_combine(y, perm["row_id_map"], topk_w)
    return {"out": out, **perm}


def moe_forward_shared(x, logits, w1, w2, k: int, S: int, renormalize: bool = True,
                       interleave: int = 0, clamp: float = 0.0):
    """The layer with S shared experts: the last S experts of w1/w2, used by
    every token with weight 1 after its k routed slots (this build's reading
    of "Fuse shared expert MLP with grouped GEMM", a commit title in the
    Megatron-LM change log on the pages; no formula is given there).  The
    routing over the first E = logits.shape[1] experts is route_topk's."""
    idx, w = route_topk(logits, k, renormalize)
    T, E = idx.shape[0], _np(logits, np.float32).shape[1]
    idx_all = np.concatenate([idx, np.tile(np.arange(E, E + S, dtype=np.int32), (T, 1))], axis=1)
    w_all = np.concatenate([w, np.ones((T, S), np.float64)], axis=1)
    res = moe_forward_routed(x, idx_all, w_all, w1, w2, interleave=interleave, clamp=clamp)
    return {**res, "topk_idx": idx_all, "topk_w": w_all}


def dense_bruteforce(x, topk_idx, topk_w, w1, w2, interleave: int = 0,
                     clamp: float = 0.0) -> np.ndarray:
    xb = _np(x, np.uint16)
    ix = _np(topk_idx, np.int32)
    ww = _np(topk_w, np.float64)
    T, H = xb.shape
    k = ix.shape[1]
    w2a = _np(w2, np.uint16)
    E, _, F = w2a.shape
    w1s, w2s = _experts(w1, E), [w2a[e] for e in range(E)]
    out = np.empty((T, H), np.float64)
    _check(_load().oracle_dense_bruteforce(T, H, F, E, k, interleave, float(clamp), _p(ix),
                                           _p(ww), _p(xb), _expert_ptrs(w1s),
                                           _expert_ptrs(w2s), _p(out)),
           "oracle_dense_bruteforce")
    return out


# ---------------------------------------------------------------- low precision

def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e8m0_value(code: int) -> float:
    return _load().oracle_e8m0_value(int(code))


# weight formats of the low-precision functions
WFMT_NVFP4 = 0  # E2M1 codes, E4M3 scale per 16 values, fp32 scale per expert tensor
WFMT_MXFP4 = 1  # E2M1 codes, E8M0 scale per 32 values (the expert scales are unused)


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def requant_fp8_block(h) -> np.ndarray:
    hh = _np(h, np.float64)
    out = np.empty_like(hh)
    _load().oracle_requant_fp8_block(_p(hh), hh.shape[0], _p(out))
    return out


def _bytes_experts(w, E: int):
    if isinstance(w, (list, tuple)):
        return [None if m is None else _np(m, np.uint8) for m in w]
    a = _np(w, np.uint8)
    return [a[e] for e in range(E)]


def _byte_ptrs(ws):
    arr = (ctypes.c_void_p * len(ws))()
    for i, w in enumerate(ws):
        arr[i] = None if w is None else w.ctypes.data
    return arr


def gemm1_swiglu_lowprec(xq_perm, xs_perm, expert_offsets, w1q, w1s, g1, F: int,
                         interleave: int = 0, clamp: float = 0.0, requant: bool = True,
                         wfmt: int = WFMT_NVFP4):
    xq = _np(xq_perm, np.uint8)
    xs = _np(xs_perm, np.float32)
    off = _np(expert_offsets, np.int32)
    E = off.shape[0] - 1
    R, H = xq.shape
    q, sc = _bytes_experts(w1q, E), _bytes_experts(w1s, E)
    g = _np(g1, np.float32)
    h = np.empty((R, F), np.float64)
    _check(_load().oracle_gemm1_swiglu_lowprec(R, H, F, E, interleave, float(clamp), _p(off),
                                               _p(xq), _p(xs), _byte_ptrs(q), _byte_ptrs(sc),
                                               _p(g), int(requant), int(wfmt), _p(h)),
           "oracle_gemm1_swiglu_lowprec")
    return h


def gemm2_lowprec(h, expert_offsets, w2q, w2s, g2, H: int, wfmt: int = WFMT_NVFP4):
    hh = _np(h, np.float64)
    off = _np(expert_offsets, np.int32)
    E = off.shape[0] - 1
    R, F = hh.shape
    q, sc = _bytes_experts(w2q, E), _bytes_experts(w2s, E)
    g = _np(g2, np.float32)
    y = np.empty((R, H), np.float64)
    _check(_load().oracle_gemm2_lowprec(R, H, F, E, _p(off), _p(hh), _byte_ptrs(q),
                                        _byte_ptrs(sc), _p(g), int(wfmt), _p(y)),
           "oracle_gemm2_lowprec")
    return y


def moe_forward_lowprec(xq, xs, logits, w1q, w1s, g1, w2q, w2s, g2, k: int,
                        renormalize: bool = True, interleave: int = 0, clamp: float = 0.0,
                        wfmt: int = WFMT_NVFP4):
    """The FP8-activation / FP4-weight layer on the given tokens (NVFP4 or,
    with wfmt=WFMT_MXFP4, MXFP4 weights; g1/g2 are then ignored).  Weight
    arguments are [E, ...] byte tensors or per-expert lists (None = unused)."""
    xqa = _np(xq, np.uint8)
    xsa = _np(xs, np.float32)
    lg = _np(logits, np.float32)
    T, H = xqa.shape
    E = lg.shape[1]
    q1, s1 = _bytes_experts(w1q, E), _bytes_experts(w1s, E)
    q2, s2 = _bytes_experts(w2q, E), _bytes_experts(w2s, E)
    F = 2 * next(m for m in q2 if m is not None).shape[1]
    out = np.empty((T, H), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _check(_load().oracle_moe_forward_lowprec(
        T, H, F, E, k, int(renormalize), interleave, float(clamp), _p(lg), _p(xqa), _p(xsa),
        _byte_ptrs(q1), _byte_ptrs(s1), _p(_np(g1, np.float32)), _byte_ptrs(q2), _byte_ptrs(s2),
        _p(_np(g2, np.float32)), int(wfmt), _p(out), _p(idx), _p(w)),
        "oracle_moe_forward_lowprec")
    return {"out": out, "topk_idx": idx, "topk_w": w}


# ---------------------------------------------------------------- backward

def routes_with_shared(logits, k: int, S: int = 0, renormalize: bool = True):
    """route_topk's routes plus S shared-expert slots (experts E .. E+S-1,
    weight 1) after the k routed ones, as [T, k+S] arrays."""
    idx, w = route_topk(logits, k, renormalize)
    if S:
        T, E = idx.shape[0], _np(logits, np.float32).shape[1]
        idx = np.concatenate([idx, np.tile(np.arange(E, E + S, dtype=np.int32), (T, 1))], axis=1)
        w = np.concatenate([w, np.ones((T, S), np.float64)], axis=1)
    return np.ascontiguousarray(idx), np.ascontiguousarray(w)


def _bwd_args(x, topk_idx, topk_w, w1, w2, d_out):
    xb = _np(x, np.uint16)
    gb = _np(d_out, np.uint16)
    ix = _np(topk_idx, np.int32)
    ww = _np(topk_w, np.float64)
    if isinstance(w1, (list, tuple)):
        E = len(w1)
    else:
        E = int(w1.shape[0])
    w1s, w2s = _experts(w1, E), _experts(w2, E)
    F = next(m for m in w2s if m is not None).shape[1]
    return xb, gb, ix, ww, w1s, w2s, E, F


def expert_backward(x, topk_idx, topk_w, w1, w2, d_out, interleave: int = 0,
                    clamp: float = 0.0, mask_f32: bool = False,
                    magnitude: bool = False) -> Dict[str, np.ndarray]:
    """Gradients of sum(d_out * out) through the expert MLPs for the given
    routes ([T, slots] indices, -1 masked, and weights): dx [T, H],
    dw_route [T, slots] (d loss / d weight of each route), dw1 [E, 2F, H] and
    dw2 [E, H, F], all fp64.  ``mask_f32`` takes the clamp decisions on the
    pre-activations rounded to fp32; ``magnitude`` returns for every output
    the sum of the absolute values of its terms instead."""
    xb, gb, ix, ww, w1s, w2s, E, F = _bwd_args(x, topk_idx, topk_w, w1, w2, d_out)
    T, H = xb.shape
    slots = ix.shape[1]
    dx = np.empty((T, H), np.float64)
    dwr = np.empty((T, slots), np.float64)
    dw1 = np.empty((E, 2 * F, H), np.float64)
    dw2 = np.empty((E, H, F), np.float64)
    _check(_load().oracle_moe_backward(T, H, F, E, slots, interleave, float(clamp),
                                       int(mask_f32), int(magnitude), _p(ix), _p(ww), _p(xb),
                                       _expert_ptrs(w1s), _expert_ptrs(w2s), _p(gb), _p(dx),
                                       _p(dwr), _p(dw1), _p(dw2)), "oracle_moe_backward")
    return {"dx": dx, "dw_route": dwr, "dw1": dw1, "dw2": dw2}


def router_backward(logits, topk_idx, topk_w, dw_route, k: int,
                    renormalize: bool = True, magnitude: bool = False) -> np.ndarray:
    """d loss / d logits [T, E] from the per-route weight gradients (the
    first k slots are the routed ones; later slots are shared experts).  With
    ``magnitude`` dw_route holds magnitudes and so does the result."""
    lg = _np(logits, np.float32)
    ix = _np(topk_idx, np.int32)
    ww = _np(topk_w, np.float64)
    dw = _np(dw_route, np.float64)
    T, E = lg.shape
    slots = ix.shape[1]
    dl = np.empty((T, E), np.float64)
    _check(_load().oracle_router_backward(T, E, k, slots, int(renormalize), int(magnitude),
                                          _p(lg), _p(ix),
                                          _p(ww), _p(dw), _p(dl)), "oracle_router_backward")
    return dl


def moe_backward(x, logits, w1, w2, d_out, k: int, renormalize: bool = True,
                 interleave: int = 0, clamp: float = 0.0, shared_experts: int = 0,
                 mask_f32: bool = False, magnitude: bool = False) -> Dict[str, np.ndarray]:
    """Gradients of sum(d_out * out) for the whole layer (route_topk's
    routing, optional shared experts): dx, dlogits, dw1, dw2 plus the
    routes."""
    idx, w = routes_with_shared(logits, k, shared_experts, renormalize)
    res = expert_backward(x, idx, w, w1, w2, d_out, interleave, clamp, mask_f32, magnitude)
    res["dlogits"] = router_backward(logits, idx, w, res["dw_route"], k, renormalize, magnitude)
    res["topk_idx"], res["topk_w"] = idx, w
    return res


def backward_tokens(x, topk_idx, topk_w, w1, w2, d_out, tokens, interleave: int = 0,
                    clamp: float = 0.0, mask_f32: bool = False, magnitude: bool = False):
    """dx rows [n, H] and per-route weight gradients [n, slots] of the listed
    tokens (expert_backward's definitions, only those rows)."""
    xb, gb, ix, ww, w1s, w2s, E, F = _bwd_args(x, topk_idx, topk_w, w1, w2, d_out)
    T, H = xb.shape
    slots = ix.shape[1]
    tk = np.ascontiguousarray(np.asarray(tokens, np.int32))
    dx = np.empty((tk.shape[0], H), np.float64)
    dw = np.empty((tk.shape[0], slots), np.float64)
    _check(_load().oracle_backward_tokens(T, H, F, E, slots, interleave, float(clamp),
                                          int(mask_f32), int(magnitude), _p(ix), _p(ww), _p(xb),
                                          _expert_ptrs(w1s), _expert_ptrs(w2s), _p(gb),
                                          tk.shape[0], _p(tk), _p(dx), _p(dw)),
           "oracle_backward_tokens")
    return dx, dw


def backward_dw1_rows(x, topk_idx, topk_w, w1, w2, d_out, pairs, interleave: int = 0,
                      clamp: float = 0.0, mask_f32: bool = False,
                      magnitude: bool = False) -> np.ndarray:
    """Rows dw1[e, row, :] for the listed (e, row) pairs, [n, H]."""
    xb, gb, ix, ww, w1s, w2s, E, F = _bwd_args(x, topk_idx, topk_w, w1, w2, d_out)
    T, H = xb.shape
    pr = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    rows = np.empty((pr.shape[0], H), np.float64)
    _check(_load().oracle_backward_dw1_rows(T, H, F, E, ix.shape[1], interleave, float(clamp),
                                            int(mask_f32), int(magnitude), _p(ix), _p(ww), _p(xb),
                                            _expert_ptrs(w1s), _expert_ptrs(w2s), _p(gb),
                                            pr.shape[0], _p(pr), _p(rows)),
           "oracle_backward_dw1_rows")
    return rows


def backward_dw2_cols(x, topk_idx, topk_w, w1, w2, d_out, pairs, interleave: int = 0,
                      clamp: float = 0.0, mask_f32: bool = False,
                      magnitude: bool = False) -> np.ndarray:
    """Columns dw2[e, :, f] for the listed (e, f) pairs, [n, H]."""
    xb, gb, ix, ww, w1s, w2s, E, F = _bwd_args(x, topk_idx, topk_w, w1, w2, d_out)
    T, H = xb.shape
    pr = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    cols = np.empty((pr.shape[0], H), np.float64)
    _check(_load().oracle_backward_dw2_cols(T, H, F, E, ix.shape[1], interleave, float(clamp),
                                            int(mask_f32), int(magnitude), _p(ix), _p(ww), _p(xb),
                                            _expert_ptrs(w1s), _p(gb), pr.shape[0], _p(pr),
                                            _p(cols)),
           "oracle_backward_dw2_cols")
    return cols
