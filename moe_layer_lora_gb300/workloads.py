"""Seeded synthetic inputs for the fused MoE-LoRA layer.

This module only draws numbers: it holds none of the layer's arithmetic, and
both the CUDA path and the fp64 oracle read the very same tensors it
returns.  Every draw comes from a ``torch.Generator`` seeded per tensor, so one
tensor can be regenerated without the others.  Router logits, the expert
bias, x and the adapter ids come from CPU generators; the weight tensors
come from a generator on ``device`` (a CUDA device draws gigabytes in
milliseconds), so the same spec gives different weights on CPU and GPU,
and both sides of a comparison always read the tensors of one draw.  Floating-point samples
are drawn in fp32 and rounded to bf16 (round-to-nearest-even); router logits
and the expert bias stay fp32.

Distributions ("N(0, v)" means variance v):
  x ~ N(0,1); logits ~ N(0,1); w13 ~ N(0, 1/H); w2 ~ N(0, 1/I);
  A13 ~ N(0, 1/H); A2 ~ N(0, 1/I); B13, B2 ~ N(0, 0.01); bias ~ N(0, 0.5).

Workloads (sizes from the five layer configurations this library is measured
on; the pages name GPT-OSS 20B and MiniMax-M3 as the models behind them):
  tiny     M=16,  H=256,  I=128,  E=8,   k=2 softmax, L=4  r=8,  idx uniform {-1..3}
  decode   M=64,  H=I=2880,       E=32,  k=4 softmax, L=8  r=16, idx uniform {-1..7}
  prefill  M=8192 (16 sequences x 512 rows), H=I=2880, E=32, k=4 softmax over
           logits + per-expert bias (load skew), L=8 r=32, one adapter per
           sequence drawn uniformly, two sequences with no adapter
  shared   M in {1,32,128}, H=3072, I=1536, E=128 + 1 shared expert,
           sigmoid+bias k=8, routed_scaling_factor 2.5, no adapters
  stress   M=512, H=I=2880, E=32, k=4 softmax, L=64 r=64, exactly 25% of
           tokens without adapter, the rest Zipf(1.1) over the adapters
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

SCORE_SOFTMAX = 0
SCORE_SIGMOID_BIAS = 1

WORKLOADS = ("tiny", "decode", "prefill", "shared", "stress")
_SEED_BASE = {"tiny": 20261, "decode": 20262, "prefill": 20263, "shared": 20264, "stress": 20265}


@dataclasses.dataclass
class Spec:
    name: str
    M: int
    H: int
    I: int
    E: int
    top_k: int
    scoring: int = SCORE_SOFTMAX
    renormalize: int = 1
    n_shared: int = 0
    routed_scaling_factor: float = 1.0
    L: int = 0
    r: int = 0
    scaling: float = 2.0
    lora_mode: str = "uniform"      # uniform | sequences | zipf | none | all_none
    logit_bias: bool = False        # add a per-expert bias to the logits (load skew)
    seq_len: int = 512
    seqs_without_adapter: int = 2
    frac_without_adapter: float = 0.25
    zipf_s: float = 1.1
    seed: int = 0

    @property
    def E_tot(self) -> int:
        return self.E + self.n_shared

    @property
    def K_total(self) -> int:
        return self.top_k + self.n_shared

    @property
    def out_scale(self) -> float:
        # shared-fusion mode scales the combined sum back by the routed
        # scaling factor; otherwise the combine is unscaled
        return self.routed_scaling_factor if self.n_shared > 0 else 1.0

    @property
    def has_lora(self) -> bool:
        return self.L > 0 and self.r > 0


def spec(name: str, **overrides) -> Spec:
    """The named workload, with optional field overrides (smaller M, ...)."""
    base = {
        "tiny": dict(M=16, H=256, I=128, E=8, top_k=2, L=4, r=8, lora_mode="uniform"),
        "decode": dict(M=64, H=2880, I=2880, E=32, top_k=4, L=8, r=16, lora_mode="uniform"),
        "prefill": dict(M=8192, H=2880, I=2880, E=32, top_k=4, L=8, r=32,
                        lora_mode="sequences", logit_bias=True),
        "shared": dict(M=128, H=3072, I=1536, E=128, top_k=8, scoring=SCORE_SIGMOID_BIAS,
                       n_shared=1, routed_scaling_factor=2.5, L=0, r=0, lora_mode="none"),
        "stress": dict(M=512, H=2880, I=2880, E=32, top_k=4, L=64, r=64, lora_mode="zipf"),
    }[name]
    base.update(overrides)
    base.setdefault("seed", _SEED_BASE[name])
    return Spec(name=name, **base)


def _gen(seed: int, slot: int, device="cpu") -> torch.Generator:
    return torch.Generator(device=device).manual_seed(seed * 64 + slot)


def _normal_bf16(shape, std: float, seed: int, slot: int, device="cpu") -> torch.Tensor:
    t = torch.randn(*shape, generator=_gen(seed, slot, device), dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


@dataclasses.dataclass
class Inputs:
    spec: Spec
    logits: torch.Tensor            # [M, E] fp32
    bias: Optional[torch.Tensor]    # [E] fp32 (sigmoid+bias routing), else None
    x: torch.Tensor                 # [M, H] bf16
    w13: torch.Tensor               # [E_tot, 2I, H] bf16
    w2: torch.Tensor                # [E_tot, H, I] bf16
    A13: Optional[torch.Tensor]     # [L, E_tot, r, H] bf16
    B13: Optional[torch.Tensor]     # [L, E_tot, 2I, r] bf16
    A2: Optional[torch.Tensor]      # [L, E_tot, r, I] bf16
    B2: Optional[torch.Tensor]      # [L, E_tot, H, r] bf16
    token_lora_idx: Optional[torch.Tensor]  # [M] int32, -1 = no adapter


def token_adapters(s: Spec) -> Optional[torch.Tensor]:
    """Per-token adapter index in [-1, L) following the workload's mode."""
    if not s.has_lora or s.lora_mode == "none":
        return None
    g = _gen(s.seed, 9)
    if s.lora_mode == "uniform":
        idx = torch.randint(-1, s.L, (s.M,), generator=g)
    elif s.lora_mode == "all_none":
        idx = torch.full((s.M,), -1)
    elif s.lora_mode == "sequences":
        nseq = max(1, math.ceil(s.M / s.seq_len))
        per_seq = torch.randint(0, s.L, (nseq,), generator=g)
        none = torch.randperm(nseq, generator=g)[: min(s.seqs_without_adapter, nseq)]
        per_seq[none] = -1
        idx = per_seq.repeat_interleave(s.seq_len)[: s.M]
    elif s.lora_mode == "zipf":
        p = torch.tensor([(l + 1.0) ** (-s.zipf_s) for l in range(s.L)], dtype=torch.float64)
        idx = torch.multinomial(p, s.M, replacement=True, generator=g)
        n_none = int(round(s.frac_without_adapter * s.M))
        none = torch.randperm(s.M, generator=g)[:n_none]
        idx[none] = -1
    else:
        raise ValueError(s.lora_mode)
    return idx.to(torch.int32).contiguous()


def make(s: Spec, with_weights: bool = True, device="cpu") -> Inputs:
    """Draw every input of one layer call (weights on ``device``)."""
    Et, H, I = s.E_tot, s.H, s.I
    logits = torch.randn(s.M, s.E, generator=_gen(s.seed, 0), dtype=torch.float32)
    bias = None
    if s.logit_bias or s.scoring == SCORE_SIGMOID_BIAS:
        b = torch.randn(s.E, generator=_gen(s.seed, 1), dtype=torch.float32) * math.sqrt(0.5)
        if s.scoring == SCORE_SIGMOID_BIAS:
            bias = b.contiguous()
        else:
            logits = (logits + b[None, :]).contiguous()
    x = _normal_bf16((s.M, H), 1.0, s.seed, 2)
    w13 = w2 = A13 = B13 = A2 = B2 = None
    if with_weights:
        w13 = _normal_bf16((Et, 2 * I, H), H ** -0.5, s.seed, 3, device)
        w2 = _normal_bf16((Et, H, I), I ** -0.5, s.seed, 4, device)
        if s.has_lora:
            A13 = _normal_bf16((s.L, Et, s.r, H), H ** -0.5, s.seed, 5, device)
            B13 = _normal_bf16((s.L, Et, 2 * I, s.r), 0.1, s.seed, 6, device)
            A2 = _normal_bf16((s.L, Et, s.r, I), I ** -0.5, s.seed, 7, device)
            B2 = _normal_bf16((s.L, Et, H, s.r), 0.1, s.seed, 8, device)
    return Inputs(s, logits.contiguous(), bias, x, w13, w2, A13, B13, A2, B2, token_adapters(s))


def bits(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Raw bf16 bit patterns of a CPU bf16 tensor as a numpy uint16 array."""
    if t is None:
        return None
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray) -> torch.Tensor:
    """Inverse of ``bits``: a numpy uint16 array as a CPU bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 (or fp32) tensor to float64 numpy."""
    return t.detach().cpu().to(torch.float64).numpy()
