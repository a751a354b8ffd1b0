"""Helpers shared by the GPU tests: seeded inputs, oracle cache, error metric."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from deterministic_attn_backward_gb300 import inputs

TOL = 1e-2  # max|gpu - ref| / max|ref| per gradient tensor (float64 oracle)


def relerr(got, ref) -> float:
    g = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else got
    r = ref
    den = float(np.max(np.abs(r)))
    return float(np.max(np.abs(g - r))) / max(den, 1e-30)


@functools.lru_cache(maxsize=32)
def case(B, H, S, d, seed, qk_scale=1.0):
    return inputs.make_qkvdo(B, H, S, d, seed, qk_scale)


@functools.lru_cache(maxsize=32)
def oracle_ref(B, H, S, d, seed, causal, qk_scale=1.0):
    q, k, v, do = case(B, H, S, d, seed, qk_scale)
    return oracle.attn_fwd_bwd(q, k, v, do, 1.0 / d ** 0.5, causal)


def oracle_heads(q, k, v, do, heads, causal):
    """Oracle on selected (b, h) heads only; returns dict of [len(heads), S, d]."""
    sel = lambda t: torch.stack([t[b, h] for b, h in heads])
    d = q.shape[-1]
    return oracle.attn_fwd_bwd(sel(q), sel(k), sel(v), sel(do), 1.0 / d ** 0.5, causal)
