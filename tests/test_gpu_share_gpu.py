"""DAB_BWD_SHARE_GPU: the main kernel launched without the cooperative
attribute where the schedule hands out units dynamically.  Same bits as the
default launch for every schedule (SHIFT keeps the cooperative launch), and
two backward calls on two streams run concurrently to completion with the
bits each gives alone."""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import case

SHARE = dab.BwdOpts(spin_timeout_ns=0, flags=dab.DAB_BWD_SHARE_GPU, grid=0)


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", ["serial", "descending_q", "shift"])
def test_share_gpu_gives_the_same_bits(mask, sched):
    B, H, S, d = 2, 4, 1024, 128
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 41))
    o, lse = dab.attn_fwd(q, k, v, mask)
    want = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
    ws = dab.new_workspace(B, H, S, d, mask, sched)
    got = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws, opts=SHARE)
    assert dab.check_status(ws) == 0
    _same(got, want)


@pytest.mark.gpu
def test_two_concurrent_calls_on_two_streams():
    """Each call's CTAs take SMs as the other's release them; the waits of
    the ticket-dispatched schedules only point at claimed units, so both
    finish, each with its own solo bits."""
    shapes = [((2, 8, 2048, 128), "full", "descending_q", 51), ((4, 4, 1024, 64), "causal", "serial", 52)]
    runs = []
    for (B, H, S, d), mask, sched, seed in shapes:
        q, k, v, do = (t.cuda() for t in case(B, H, S, d, seed))
        o, lse = dab.attn_fwd(q, k, v, mask)
        solo = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
        ws = dab.new_workspace(B, H, S, d, mask, sched)
        out = tuple(torch.empty_like(q) for _ in range(3))
        runs.append((q, k, v, o, lse, do, mask, sched, ws, out, solo))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in runs]
    for _ in range(3):
        for st, (q, k, v, o, lse, do, mask, sched, ws, out, _) in zip(streams, runs):
            with torch.cuda.stream(st):
                dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws, out=out, opts=SHARE)
        torch.cuda.synchronize()
        for *_, ws, out, solo in runs:
            assert dab.check_status(ws) == 0
            _same(out, solo)
