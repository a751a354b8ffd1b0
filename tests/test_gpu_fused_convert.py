"""dQ finalised in the main kernel's tail (the default for the ordered
schedules) against the separate convert pass (DAB_BWD_SEPARATE_CONVERT): the
same additions in the same order, so the same bits, whatever the schedule,
mask, head dimension, sequence length (whole or partial last tile) or number
of CTAs; and the fused result stays within tolerance of the oracle."""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import TOL, case, oracle_ref, relerr

SEPARATE = dab.BwdOpts(spin_timeout_ns=0, flags=dab.DAB_BWD_SEPARATE_CONVERT, grid=0)


def _same_bits(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", ["serial", "descending_q", "shift"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [1024, 768, 1000])
def test_fused_convert_gives_the_separate_bits(mask, sched, d, S):
    B, H = 2, 3
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 17))
    o, lse = dab.attn_fwd(q, k, v, mask)
    ws = dab.new_workspace(B, H, S, d, mask, sched)
    fused = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws)
    assert dab.check_status(ws) == 0
    sep = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, opts=SEPARATE)
    _same_bits(fused, sep)


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("S", [200, 1000])
def test_fused_convert_partial_last_tile(mask, S):
    """A partial last Q tile: rows past S are neither read nor written (the
    next head's rows follow in the accumulator and in dQ)."""
    B, H, d = 2, 2, 64
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 5))
    o, lse = dab.attn_fwd(q, k, v, mask)
    for sched in ("serial", "descending_q"):
        fused = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
        sep = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, opts=SEPARATE)
        _same_bits(fused, sep)
    ref = oracle_ref(B, H, S, d, 5, mask == "causal")
    assert relerr(fused[0], ref["dq"]) < TOL


@pytest.mark.gpu
@pytest.mark.parametrize("grid", [1, 3, 37])
def test_fused_convert_with_few_ctas(grid):
    """Fewer CTAs than units: CTAs enter the tail at different times and
    claim tiles of heads still in progress (their waits end when the
    contributions are in); with one CTA every tile is final when claimed."""
    B, H, S, d, mask = 2, 2, 1024, 128, "causal"
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 9))
    o, lse = dab.attn_fwd(q, k, v, mask)
    for sched in ("serial", "descending_q"):
        base = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, opts=SEPARATE)
        ws = dab.new_workspace(B, H, S, d, mask, sched)
        got = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws,
                           opts=dab.BwdOpts(spin_timeout_ns=0, flags=0, grid=grid))
        assert dab.check_status(ws) == 0
        _same_bits(got, base)
        if sched == "serial":
            dq_serial = got[0]
    # serial and descending share the ranks of dQ (not the order along a
    # chain, so dK and dV may differ in the last bits)
    _same_bits((dq_serial,), (got[0],))


@pytest.mark.gpu
def test_fused_convert_parity_and_repeatability():
    B, H, S, d, mask = 1, 4, 2048, 128, "causal"
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 21))
    o, lse = dab.attn_fwd(q, k, v, mask)
    ref = oracle_ref(B, H, S, d, 21, True)
    runs = [dab.attn_bwd(q, k, v, o, lse, do, mask, "shift") for _ in range(5)]
    for r in runs[1:]:
        _same_bits(r, runs[0])
    for name, g in zip(("dq", "dk", "dv"), runs[0]):
        assert relerr(g, ref[name]) < TOL, name
