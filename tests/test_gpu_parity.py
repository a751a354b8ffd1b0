"""CUDA forward/backward against the float64 oracle, element by element."""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import TOL, case, oracle_ref, relerr

SCHEDS = ["serial", "descending_q", "shift", "atomic"]
# (B, H, S, d): one and several tiles, both head dims, an odd tile count.
SHAPES = [(1, 2, 256, 64), (1, 2, 256, 128), (2, 3, 640, 64), (1, 2, 768, 128), (1, 1, 128, 128)]


def _run(B, H, S, d, seed, mask, sched):
    q, k, v, do = case(B, H, S, d, seed)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = dab.attn_fwd(qd, kd, vd, mask)
    ws = dab.new_workspace(B, H, S, d, mask, sched)
    dq, dk, dv = dab.attn_bwd(qd, kd, vd, o, lse, dod, mask, sched, workspace=ws)
    assert dab.check_status(ws) == 0
    return o, lse, dq, dk, dv


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%dh%ds%dd%d" % s)
@pytest.mark.parametrize("mask", ["full", "causal"])
def test_forward_matches_oracle(shape, mask):
    B, H, S, d = shape
    q, k, v, _ = case(B, H, S, d, 0)
    o, lse = dab.attn_fwd(q.cuda(), k.cuda(), v.cuda(), mask)
    ref = oracle_ref(B, H, S, d, 0, mask == "causal")
    assert relerr(o, ref["o"]) < TOL
    assert (lse.cpu().double().numpy() - ref["lse"]).__abs__().max() < 1e-3


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b%dh%ds%dd%d" % s)
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", SCHEDS)
def test_backward_matches_oracle(shape, mask, sched):
    B, H, S, d = shape
    if sched == "shift" and mask == "causal" and (S // 128) % 2:
        pytest.skip("causal shift needs an even tile count")
    _, _, dq, dk, dv = _run(B, H, S, d, 0, mask, sched)
    ref = oracle_ref(B, H, S, d, 0, mask == "causal")
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        err = relerr(got, ref[name])
        assert err < TOL, f"{name}: {err:.3e}"
