"""Seeded synthetic inputs for attention backward workloads.

This module holds no attention arithmetic: it only draws random numbers and
names the workloads.  Both the CUDA path's tests/benchmark and the CPU oracle's
tests take their inputs from here, so the two sides see identical bits.

Recipe: ``torch.Generator().manual_seed(seed)``, then ``torch.randn`` in
float32 on the CPU in the order Q, K, V, dO, each of shape [B, H, S, d], then
rounding to bfloat16.  Workloads that keep softmax peaked but finite scale Q
and K by 0.5 after rounding (a power of two, so exact in bfloat16).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    d: int
    seed: int
    masks: tuple = ("full",)
    qk_scale: float = 1.0  # multiplier applied to Q and K after bf16 rounding

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d)."""
        return 1.0 / math.sqrt(self.d)

    def flops(self, mask: str) -> float:
        """Algorithmic backward FLOPs: 10*B*H*S^2*d for full, half for causal."""
        f = 10.0 * self.B * self.H * self.S * self.S * self.d
        return f if mask == "full" else f / 2.0


# The workloads of the benchmark plan.
PR1_REF = Workload("pr1_ref_b1h2s256d64", 1, 2, 256, 64, 0, ("causal", "full"))
MID_D64 = Workload("b4h16s2048d64_full", 4, 16, 2048, 64, 1, ("full",))
HEADLINE = Workload("b2h16s8192d128", 2, 16, 8192, 128, 2, ("causal", "full"), 0.5)
LONG = Workload("b1h32s16384d128", 1, 32, 16384, 128, 3, ("full", "causal"))


def sweep(d: int) -> list:
    """B*S fixed at 32768 tokens, H=16, S from 1k to 32k, both masks, seed 4."""
    out = []
    for S in (1024, 2048, 4096, 8192, 16384, 32768):
        out.append(Workload(f"sweep_s{S}_d{d}", 32768 // S, 16, S, d, 4,
                            ("causal", "full")))
    return out


WORKLOADS = {w.name: w for w in (PR1_REF, MID_D64, HEADLINE, LONG,
                                 *sweep(64), *sweep(128))}


def make_qkvdo(B: int, H: int, S: int, d: int, seed: int, qk_scale: float = 1.0):
    """Return (q, k, v, dout) as contiguous CPU bfloat16 tensors [B, H, S, d]."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, S, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32).bfloat16()
    k = torch.randn(shape, generator=g, dtype=torch.float32).bfloat16()
    v = torch.randn(shape, generator=g, dtype=torch.float32).bfloat16()
    do = torch.randn(shape, generator=g, dtype=torch.float32).bfloat16()
    if qk_scale != 1.0:
        q = q * qk_scale
        k = k * qk_scale
    return q.contiguous(), k.contiguous(), v.contiguous(), do.contiguous()


def make_workload(w: Workload):
    return make_qkvdo(w.B, w.H, w.S, w.d, w.seed, w.qk_scale)
