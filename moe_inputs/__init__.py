"""Seeded synthetic inputs for the MoE expert-FFN layer.

This module only draws random numbers and shapes them into the tensors the
layer consumes; it holds none of the layer's arithmetic (no routing, no
permutation, no GEMM, no activation).  Both the CUDA path and the CPU oracle
receive the very same tensors from here, so neither side's inputs ever come
from the other.

Workloads (the five shapes the pages' MoE discussion revolves around; see the
"[SM90] Add W4A8 MegaMoE support" page, Usage section, for the problem
statement: hidden width H, intermediate width F, E experts, top-k routes):

  tiny      T=64   H=256  F=512   E=8   k=2
  mixtral   T=4096 H=4096 F=14336 E=8   k=2
  skewed    T=8192 H=7168 F=2048  E=256 k=8   (Zipf-law per-expert logit bias)
  decode    T in {1,8,32,128,256}, H=2048 F=768 E=128 k=8
  lowprec   T=4096 H=7168 F=2048  E=256 k=8   (FP8 activations, NVFP4 weights,
                                               GLU interleave 32, clamp 7.0)

Recipe (all from one ``torch.Generator`` seeded with ``seed``; draws happen
in the fixed order logits, x, w1, w2 so a tensor never depends on another's
size):
  * X      ~ N(0, 1), rounded to bf16 (round-to-nearest-even, torch's cast)
  * logits ~ N(0, 1) fp32; for ``skewed`` a per-expert bias
    b_e = -s * ln(rank_e) is added, rank = a seeded random permutation of
    1..E and s = 1.1 (Zipf-law expert popularity)
  * W1 [E, 2F, H] ~ N(0, 1/H), W2 [E, H, F] ~ N(0, 1/F), rounded to bf16.
  * backward: the output gradient dOut [T, H] ~ N(0, 1), rounded to bf16,
    from its own generator (seed + 4).

Full-size weights are drawn directly on the device given (``device='cuda'``)
because they are gigabytes; the oracle is then handed host copies of exactly
those bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    zipf_s: float = 0.0          # > 0: add the Zipf-law per-expert bias
    glu_interleave: int = 0      # 0: W1 rows are [gate(F) | up(F)]
    swiglu_clamp: float = 0.0    # <= 0: no clamp
    lowprec: bool = False        # FP8 activations / NVFP4 weights

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops(self) -> float:
        """Algorithmic FLOPs of one forward: GEMM1 4*R*H*F + GEMM2 2*R*H*F."""
        return 6.0 * self.T * self.k * self.H * self.F

    def with_T(self, T: int) -> "MoEShape":
        return dataclasses.replace(self, T=T)


TINY = MoEShape("tiny", T=64, H=256, F=512, E=8, k=2)
MIXTRAL = MoEShape("mixtral", T=4096, H=4096, F=14336, E=8, k=2)
SKEWED = MoEShape("skewed", T=8192, H=7168, F=2048, E=256, k=8, zipf_s=1.1)
DECODE_TS = (1, 8, 32, 128, 256)
DECODE = MoEShape("decode", T=256, H=2048, F=768, E=128, k=8)
LOWPREC = MoEShape("lowprec", T=4096, H=7168, F=2048, E=256, k=8,
                   glu_interleave=32, swiglu_clamp=7.0, lowprec=True)

SHAPES = {s.name: s for s in (TINY, MIXTRAL, SKEWED, DECODE, LOWPREC)}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zipf_bias(E: int, s: float, seed: int) -> torch.Tensor:
    """Per-expert logit bias b_e = -s * ln(rank_e), rank a seeded permutation of 1..E."""
    g = _gen(seed + 7919, "cpu")
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-s * torch.log(rank)).to(torch.float32)


def make_logits(shape: MoEShape, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    logits = torch.randn(shape.T, shape.E, generator=g, device=device, dtype=torch.float32)
    if shape.zipf_s > 0:
        logits = logits + zipf_bias(shape.E, shape.zipf_s, seed).to(device)
    return logits


def make_x(shape: MoEShape, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed + 1, device)
    return torch.randn(shape.T, shape.H, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def _randn_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    # Draw per expert so peak fp32 scratch stays one expert's worth.
    for e in range(shape[0]):
        out[e].copy_(torch.randn(shape[1:], generator=g, device=device,
                                 dtype=torch.float32).mul_(std))
    return out


def make_w1(shape: MoEShape, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed + 2, device)
    return _randn_bf16((shape.E, 2 * shape.F, shape.H), 1.0 / math.sqrt(shape.H), g, device)


def make_w2(shape: MoEShape, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed + 3, device)
    return _randn_bf16((shape.E, shape.H, shape.F), 1.0 / math.sqrt(shape.F), g, device)


def make_inputs(shape: MoEShape, seed: int = 0, device="cpu",
                weights: bool = True) -> Dict[str, Optional[torch.Tensor]]:
    """All bf16-path inputs of one layer call, drawn on ``device``."""
    out = {
        "logits": make_logits(shape, seed, device),
        "x": make_x(shape, seed, device),
        "w1": make_w1(shape, seed, device) if weights else None,
        "w2": make_w2(shape, seed, device) if weights else None,
    }
    return out


def make_grad_out(shape: MoEShape, seed: int = 0, device="cpu") -> torch.Tensor:
    """The gradient of the loss with respect to the layer's output, [T, H] bf16."""
    g = _gen(seed + 4, device)
    return torch.randn(shape.T, shape.H, generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor as a contiguous numpy array."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def random_topk_idx(T: int, E: int, k: int, seed: int = 0, mask_frac: float = 0.0):
    """Seeded routing table with k distinct experts per token (int32 [T, k]).

    Used to exercise the permute/combine stages on their own; ``mask_frac`` of
    the routes are set to -1 (a masked route).
    """
    g = _gen(seed + 11, "cpu")
    scores = torch.rand(T, E, generator=g)
    idx = torch.argsort(scores, dim=1)[:, :k].to(torch.int32)
    if mask_frac > 0:
        m = torch.rand(T, k, generator=g) < mask_frac
        idx[m] = -1
    return idx.contiguous()


def random_weights(T: int, k: int, seed: int = 0) -> torch.Tensor:
    """Seeded positive routing weights (fp32 [T, k]) for combine-only tests."""
    g = _gen(seed + 13, "cpu")
    return torch.rand(T, k, generator=g, dtype=torch.float32).add_(0.05).contiguous()


# ------------------------------------------------------------------ low precision inputs
#
# The low-precision workload's tensors are quantised from the same seeded
# normal draws (this is how its inputs are made, not part of the layer):
#   activations: per 1x128 block, s = amax / 448, code = E4M3(x / s) (torch's
#     round-to-nearest-even cast after clamping to +-448)
#   weights (per expert tensor): g = amax / 448; per 16 values along K,
#     s_b = E4M3(amax_b / (6 g)); q = E2M1(w / (s_b g)) round-to-nearest-even,
#     saturating at 6; two codes per byte, the even index in the low nibble.
#     (6 * s_b <= 448, the decoder-range rule for NVFP4 scales.)

def quantize_fp8_rows(x: torch.Tensor, block: int = 128):
    """x [T, H] float -> (codes uint8 [T, H], scales fp32 [T, H/block])."""
    T, H = x.shape
    xb = x.float().reshape(T, H // block, block)
    amax = xb.abs().amax(-1)
    s = amax / 448.0
    s = torch.where(amax > 0, s, torch.ones_like(s))
    q = (xb / s[..., None]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).reshape(T, H).contiguous(), s.contiguous()


def _e2m1_code(a: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even E2M1 code (0..7) of magnitudes a >= 0, saturating."""
    code = torch.zeros_like(a, dtype=torch.uint8)
    # boundaries between codes; equality goes to the even code
    for c, lo, incl in ((1, 0.25, False), (2, 0.75, True), (3, 1.25, False), (4, 1.75, True),
                        (5, 2.5, False), (6, 3.5, True), (7, 5.0, False)):
        above = a >= lo if incl else a > lo
        code = torch.where(above, torch.full_like(code, c), code)
    return code


def quantize_nvfp4(w: torch.Tensor):
    """w [N, K] float -> (packed uint8 [N, K/2], scales uint8 [N, K/16], g fp32 scalar)."""
    N, K = w.shape
    wf = w.float()
    amax = wf.abs().max()
    g = (amax / 448.0) if amax > 0 else torch.ones((), device=w.device)
    blocks = wf.reshape(N, K // 16, 16)
    bmax = blocks.abs().amax(-1)
    s8 = (bmax / (6.0 * g)).clamp_(max=448.0).to(torch.float8_e4m3fn)
    sv = s8.float()
    denom = (sv * g)[..., None]
    ratio = torch.where(denom > 0, blocks / torch.where(denom > 0, denom, torch.ones_like(denom)),
                        torch.zeros_like(blocks))
    code = _e2m1_code(ratio.abs()) | (ratio < 0).to(torch.uint8) << 3
    code = code.reshape(N, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, s8.view(torch.uint8).contiguous(), g.float().reshape(())


def quantize_mxfp4(w: torch.Tensor):
    """w [N, K] float -> (packed uint8 [N, K/2], E8M0 scale bytes uint8 [N, K/32]).

    Per 32 values (the OCP microscaling recipe): shared exponent
    s = floor(log2(amax)) - 2 (2 = the largest E2M1 exponent), scale byte
    s + 127 (0 for an all-zero block); q = E2M1(w / 2^s) round-to-nearest-even,
    saturating at 6.  Two codes per byte, the even index in the low nibble."""
    N, K = w.shape
    blocks = w.float().reshape(N, K // 32, 32)
    amax = blocks.abs().amax(-1)
    exp = torch.floor(torch.log2(torch.where(amax > 0, amax, torch.ones_like(amax)))) - 2
    exp = torch.where(amax > 0, exp.clamp_(-127, 127), torch.full_like(exp, -127))
    ratio = blocks / torch.exp2(exp)[..., None]
    code = _e2m1_code(ratio.abs()) | (ratio < 0).to(torch.uint8) << 3
    code = code.reshape(N, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, (exp + 127).to(torch.uint8).contiguous()


def make_lowprec_inputs(shape: MoEShape, seed: int = 0, device="cpu",
                        weights: bool = True, wfmt: str = "nvfp4"
                        ) -> Dict[str, Optional[torch.Tensor]]:
    """FP8 activations (+ fp32 scales), fp32 logits and FP4 weights: NVFP4
    (codes w?q, E4M3 scales per 16 w?s, fp32 expert scales w?g) or, with
    wfmt="mxfp4", MXFP4 (codes w?q, E8M0 scales per 32 w?s) from the same
    normal draws."""
    g = _gen(seed + 1, device)
    x = torch.randn(shape.T, shape.H, generator=g, device=device, dtype=torch.float32)
    xq, xs = quantize_fp8_rows(x)
    out = {"logits": make_logits(shape, seed, device), "xq": xq, "xs": xs}
    if weights:
        blk = 32 if wfmt == "mxfp4" else 16
        for name, rows, cols, sd in (("w1", 2 * shape.F, shape.H, seed + 2),
                                     ("w2", shape.H, shape.F, seed + 3)):
            gw = _gen(sd, device)
            q = torch.empty(shape.E, rows, cols // 2, dtype=torch.uint8, device=device)
            sc = torch.empty(shape.E, rows, cols // blk, dtype=torch.uint8, device=device)
            gs = torch.empty(shape.E, dtype=torch.float32, device=device)
            for e in range(shape.E):
                wf = torch.randn(rows, cols, generator=gw, device=device,
                                 dtype=torch.float32).mul_(1.0 / math.sqrt(cols))
                if wfmt == "mxfp4":
                    q[e], sc[e] = quantize_mxfp4(wf)
                    gs[e] = 1.0
                else:
                    q[e], sc[e], gs[e] = quantize_nvfp4(wf)
            out[name + "q"], out[name + "s"] = q, sc
            if wfmt != "mxfp4":
                out[name + "g"] = gs
    return out
