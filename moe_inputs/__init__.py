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
