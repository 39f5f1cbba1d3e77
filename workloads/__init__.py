"""Seeded synthetic inputs for the dropless MoE layer forward.

This module is shared by the tests, ``bench.py`` and ``smoke()``.  It holds no
arithmetic of the method itself: it only draws random tensors with the shapes
and distributions of the five workload shapes below and rounds them to the
storage precisions the layer takes (bf16 activations and expert weights, fp32
router weights and bias).

Shapes (T tokens, d model dim, E experts, K experts per token, f expert FFN
dim).  The layer is a SwiGLU FFN per expert: W1 maps d -> 2f (gate rows
0..f-1, up rows f..2f-1), W2 maps f -> d.

Distributions (std unless stated):
  x  ~ N(0, 1)                -> bf16 (round to nearest even)
  Wr ~ N(0, 1/d)   [d, E]     fp32
  W1 ~ N(0, 1/d)   [E, 2f, d] -> bf16
  W2 ~ N(0, 1/f)   [E, d, f]  -> bf16
  bias [E] fp32, per workload:
    tiny, qwen : 0
    mixtral    : N(0, 0.5^2)  (std 0.5, mild load skew)
    dsv3       : -1.1 * ln(e + 1)  (log of a Zipf(s=1.1) popularity; some
                 experts then receive no token)
    skew       : +3 on expert 0 (chosen by nearly every token, which is the
                 most one expert can receive with K distinct experts per
                 token, and about half of the combine weight), -30 on experts
                 E-16..E-1 (they receive no token), 0 elsewhere

Generators: on a CPU device, numpy PCG64(seed) (identical on every host);
on a CUDA device, torch's Philox generator seeded with ``seed`` (identical on
the same GPU model and torch build).  Token activations and weights take
separate seeds so that a caller can re-draw x (and with it the routing) while
keeping the weights resident.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

CONFIGS = {
    "tiny": dict(T=256, d=128, E=8, K=2, f=256, bias="zero"),
    "mixtral": dict(T=8192, d=4096, E=8, K=2, f=14336, bias="normal_0.5"),
    "dsv3": dict(T=4096, d=7168, E=256, K=8, f=2048, bias="zipf_1.1"),
    "qwen": dict(T=16384, d=2048, E=128, K=8, f=768, bias="zero"),
    "skew": dict(T=32768, d=4096, E=64, K=6, f=1536, bias="skew"),
    # profiling-size stand-in for dsv3: the same d, f, K and rows per expert
    # (T*K/E = 128) with 32 experts, so a full ncu capture holds ~3 GB
    "dsv3_e32": dict(T=512, d=7168, E=32, K=8, f=2048, bias="zipf_1.1"),
    # profiling-size stand-in for the Mixtral-shaped GEMMs: the same d and f
    # (so the same tile shapes and K lengths) with 2 experts and 2048 rows
    # each, about 1 GB of weights
    "mixtral_e2": dict(T=2048, d=4096, E=2, K=1, f=14336, bias="zero"),
    # profiling-size stand-in for the skew layer: the same d, f, E, K and bias
    # rule with an eighth of the tokens (the same GEMM kernels and tile
    # shapes), about 3 GB on the device
    "skew_t4096": dict(T=4096, d=4096, E=64, K=6, f=1536, bias="skew"),
}

DESCRIPTIONS = {
    "tiny": "Tiny dropless MoE fwd T=256 d=128 E=8 K=2 f=256",
    "mixtral": "Mixtral-8x7B-shaped MoE layer fwd T=8192 d=4096 E=8 K=2 f=14336",
    "dsv3": "DeepSeek-V3-shaped routed-expert layer fwd T=4096 d=7168 E=256 K=8 f=2048",
    "qwen": "Qwen-MoE-shaped layer fwd T=16384 d=2048 E=128 K=8 f=768",
    "skew": "Extreme-skew MoE layer fwd T=32768 d=4096 E=64 K=6 f=1536",
    "dsv3_e32": "DeepSeek-V3-shaped layer, 32 experts (profiling size) T=512 d=7168 E=32 K=8 f=2048",
    "mixtral_e2": "Mixtral-shaped expert GEMMs, 2 experts (profiling size) T=2048 d=4096 E=2 K=1 f=14336",
    "skew_t4096": "Extreme-skew MoE layer, 4096 tokens (profiling size) T=4096 d=4096 E=64 K=6 f=1536",
}


@dataclass
class Shape:
    T: int
    d: int
    E: int
    K: int
    f: int
    bias: str = "zero"

    @property
    def TK(self) -> int:
        return self.T * self.K

    @property
    def useful_flops(self) -> int:
        """Two grouped GEMMs over the T*K valid rows: 2*TK*d*(2f) + 2*TK*f*d."""
        return 6 * self.TK * self.d * self.f


def shape(name_or_shape) -> Shape:
    if isinstance(name_or_shape, Shape):
        return name_or_shape
    if isinstance(name_or_shape, dict):
        return Shape(**name_or_shape)
    return Shape(**CONFIGS[name_or_shape])


@dataclass
class LayerWeights:
    Wr: torch.Tensor    # [d, E] fp32
    bias: torch.Tensor  # [E]    fp32
    W1: torch.Tensor    # [E, 2f, d] bf16
    W2: torch.Tensor    # [E, d, f]  bf16


class _Draw:
    """Standard-normal fp32 draws from one seeded stream on one device."""

    def __init__(self, seed: int, device):
        self.device = torch.device(device)
        if self.device.type == "cpu":
            self.np = np.random.Generator(np.random.PCG64(seed))
            self.g = None
        else:
            self.np = None
            self.g = torch.Generator(device=self.device)
            self.g.manual_seed(seed)

    def normal(self, shape_, std: float = 1.0) -> torch.Tensor:
        if self.np is not None:
            a = self.np.standard_normal(size=shape_, dtype=np.float32)
            if std != 1.0:
                a *= np.float32(std)
            return torch.from_numpy(a)
        t = torch.randn(shape_, generator=self.g, device=self.device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t


def _bias(s: Shape, draw: _Draw) -> torch.Tensor:
    E = s.E
    if s.bias == "zero":
        b = torch.zeros(E, dtype=torch.float32)
    elif s.bias == "normal_0.5":
        b = draw.normal((E,), 0.5).cpu()
    elif s.bias == "zipf_1.1":
        b = torch.tensor([-1.1 * math.log(e + 1) for e in range(E)], dtype=torch.float32)
    elif s.bias == "skew":
        b = torch.zeros(E, dtype=torch.float32)
        b[0] = 3.0
        if E > 16:
            b[E - 16:] = -30.0
    else:
        raise ValueError(f"unknown bias rule {s.bias!r}")
    return b.to(draw.device)


def make_weights(cfg, seed: int = 0, device="cpu") -> LayerWeights:
    """Router and expert weights of one layer, drawn from ``seed`` on ``device``."""
    s = shape(cfg)
    draw = _Draw(seed, device)
    Wr = draw.normal((s.d, s.E), 1.0 / math.sqrt(s.d))
    bias = _bias(s, draw)
    W1 = torch.empty((s.E, 2 * s.f, s.d), dtype=torch.bfloat16, device=draw.device)
    W2 = torch.empty((s.E, s.d, s.f), dtype=torch.bfloat16, device=draw.device)
    for e in range(s.E):  # one expert at a time keeps the fp32 temporaries small
        W1[e].copy_(draw.normal((2 * s.f, s.d), 1.0 / math.sqrt(s.d)))
        W2[e].copy_(draw.normal((s.d, s.f), 1.0 / math.sqrt(s.f)))
    return LayerWeights(Wr=Wr.contiguous(), bias=bias.contiguous(), W1=W1, W2=W2)


def make_tokens(cfg, seed: int = 0, device="cpu") -> torch.Tensor:
    """Token activations x [T, d] bf16 ~ N(0, 1), drawn from ``seed`` on ``device``."""
    s = shape(cfg)
    draw = _Draw(seed + 1_000_003, device)
    return draw.normal((s.T, s.d)).to(torch.bfloat16)


def random_shape_cases():
    """Small ragged shapes for parity tests: they span several GEMM tiles and
    leave ragged tails in T, in the per-expert groups and in d and f."""
    return [
        Shape(T=1, d=64, E=1, K=1, f=64),
        Shape(T=7, d=64, E=3, K=2, f=128),
        Shape(T=33, d=192, E=8, K=2, f=192),
        Shape(T=300, d=256, E=64, K=8, f=128),
        Shape(T=129, d=128, E=256, K=8, f=64),
        Shape(T=1000, d=512, E=8, K=1, f=320),
        Shape(T=517, d=320, E=16, K=4, f=448),
        Shape(T=333, d=320, E=16, K=8, f=192),   # K = 8 with a ragged 256-column round of the combine
        # average group >= 384 rows: the grouped GEMMs take their CTA-pair
        # (256-row tile) path; ragged tails inside the pair tiles
        Shape(T=2048, d=256, E=4, K=1, f=256),
        Shape(T=1500, d=192, E=2, K=2, f=192),
        Shape(T=777, d=320, E=3, K=2, f=448),
    ]
