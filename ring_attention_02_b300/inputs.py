"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws random tensors and
names problem sizes, so both the CUDA path and the CPU oracle's tests can use
it.  It imports neither of them.

Inputs are fp32 samples of N(0, 1) rounded to bf16 (round to nearest even),
drawn from ``torch.Generator`` streams seeded ``seed + 0`` for Q, ``+1`` for
K, ``+2`` for V and ``+3`` for dO.  A CUDA generator and a CPU generator give
different streams; every comparison copies the very tensors the GPU used to
the host for the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch

LAYOUT_IDS = {"contiguous": 0, "striped": 1, "zigzag": 2}


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, shard count, layout and mask."""
    name: str
    B: int
    H: int
    Hkv: int
    S: int
    D: int
    P: int
    layout: str
    causal: bool
    out_f32: bool = False
    backward: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / (self.D ** 0.5)

    def with_layout(self, layout: str) -> "Workload":
        return Workload(**{**asdict(self), "layout": layout,
                           "name": f"{self.name}-{layout}"})

    def counted_flops(self) -> float:
        """4*B*H*S^2*D, halved for a causal mask (forward only)."""
        f = 4.0 * self.B * self.H * self.S * self.S * self.D
        return f / 2 if self.causal else f

    def step_flops(self) -> float:
        """Counted flops of one step: the forward, plus 2.5x the forward for
        the backward (five matrix products against the forward's two)."""
        return self.counted_flops() * (3.5 if self.backward else 1.0)


# The five problems the library is measured and checked on.
TINY = Workload("tiny-noncausal-B1H2S256D64P4", 1, 2, 2, 256, 64, 4, "contiguous", False,
                out_f32=True)
CAUSAL_8K = Workload("causal-B1H8S8192D128P8", 1, 8, 8, 8192, 128, 8, "zigzag", True)
GQA_128K = Workload("causal-gqa-B1H32Hkv8S131072D128P16", 1, 32, 8, 131072, 128, 16,
                    "striped", True)
MILLION = Workload("causal-B1H8Hkv1S1048576D128P32", 1, 8, 1, 1048576, 128, 32, "zigzag",
                   True)
TRAIN_32K = Workload("train-B2H16S32768D128P8", 2, 16, 16, 32768, 128, 8, "zigzag", True,
                     backward=True)
WORKLOADS = [TINY, CAUSAL_8K, GQA_128K, MILLION, TRAIN_32K]
# A mid-size causal forward for profiler captures: 192 MiB of q/k/v (larger
# than the 126 MB L2) and a few milliseconds per launch.
PROFILE_32K = Workload("causal-B1H8S32768D128P8", 1, 8, 8, 32768, 128, 8, "zigzag", True)
# A smaller training step for profiler captures of the backward kernels.
PROFILE_TRAIN_16K = Workload("train-B1H16S16384D128P8", 1, 16, 16, 16384, 128, 8, "zigzag",
                             True, backward=True)
# The headline forward: the 128k GQA shapes with the zig-zag layout.
HEADLINE = GQA_128K.with_layout("zigzag")


def by_name(name: str) -> Workload:
    for w in WORKLOADS + [HEADLINE, PROFILE_32K, PROFILE_TRAIN_16K]:
        if w.name == name:
            return w
    raise KeyError(name)


def _randn_bf16(shape, seed: int, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_qkv(B, H, Hkv, S, D, seed: int = 0, device="cpu"):
    """Q [B,S,H,D], K and V [B,S,Hkv,D], bf16, natural token order."""
    q = _randn_bf16((B, S, H, D), seed + 0, device)
    k = _randn_bf16((B, S, Hkv, D), seed + 1, device)
    v = _randn_bf16((B, S, Hkv, D), seed + 2, device)
    return q, k, v


def make_dout(B, H, S, D, seed: int = 0, device="cpu") -> torch.Tensor:
    """dO [B,S,H,D] bf16 for the backward pass."""
    return _randn_bf16((B, S, H, D), seed + 3, device)


def make_for(w: Workload, seed: int = 0, device="cpu"):
    return make_qkv(w.B, w.H, w.Hkv, w.S, w.D, seed=seed, device=device)


def pack_lengths(count: int, lo: int, hi: int, multiple: int, seed: int = 0):
    """Seeded document lengths for a packed batch: log-uniform in [lo, hi],
    rounded down to a multiple of `multiple` (so every sequence splits evenly
    over the ranks), at least `multiple`."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 4)
    u = torch.rand(count, generator=g, dtype=torch.float64)
    L = torch.exp(torch.log(torch.tensor(float(lo))) + u * (torch.log(torch.tensor(float(hi)))
                                                          - torch.log(torch.tensor(float(lo)))))
    return [max(multiple, int(x) // multiple * multiple) for x in L.tolist()]

