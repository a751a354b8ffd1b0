"""Bitwise run-to-run reproducibility of the deterministic schedules."""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import case

RUNS = 20


def _grads(B, H, S, d, mask, sched, runs):
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 11))
    o, lse = dab.attn_fwd(q, k, v, mask)
    ws = dab.new_workspace(B, H, S, d, mask, sched)
    out = []
    for _ in range(runs):
        g = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws)
        out.append(tuple(t.clone() for t in g))
    assert dab.check_status(ws) == 0
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", ["serial", "descending_q", "shift"])
@pytest.mark.parametrize("d", [64, 128])
def test_bitwise_repeatable(mask, sched, d):
    runs = _grads(2, 4, 1024, d, mask, sched, RUNS)
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("d", [64, 128])
def test_descending_keeps_serial_dq_bits(mask, d):
    """Descending Q-tile iteration keeps the serial schedule's dQ reduction
    order, so dQ is bitwise equal.  dK and dV accumulate on chip along the
    chain, whose Q-tile order descending reverses: equal within tolerance."""
    a = _grads(2, 4, 1024, d, mask, "serial", 1)[0]
    b = _grads(2, 4, 1024, d, mask, "descending_q", 1)[0]
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    for x, y in zip(a[1:], b[1:]):
        err = (x.double() - y.double()).abs().max() / y.double().abs().max()
        assert err < 1e-2


@pytest.mark.gpu
@pytest.mark.parametrize("shape,mask", [((2, 4, 1024, 64), "full"), ((2, 4, 1024, 128), "causal"),
                                        ((1, 3, 2048, 128), "full")])
def test_auto_runs_the_selected_schedule(shape, mask):
    """DAB_SCHED_AUTO runs the schedule dab_sched_select picks for this
    device's SM count: the same bits as asking for it by name, every time."""
    B, H, S, d = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pick = dab.sched_select(mask, B, H, S, sms)
    auto = _grads(B, H, S, d, mask, "auto", 2)
    named = _grads(B, H, S, d, mask, pick, 1)[0]
    for run in auto:
        for a, b in zip(run, named):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", ["serial", "descending_q", "shift"])
@pytest.mark.parametrize("d", [64, 128])
def test_plain_adds_give_the_red_bits(mask, sched, d):
    """The ordered reduction adds each partial with red.add.f32 in the L2.
    Done instead as load + add + store (DAB_BWD_PLAIN_ADD), the same IEEE
    additions in the same order: the same bits."""
    B, H, S = 2, 4, 1024
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 13))
    o, lse = dab.attn_fwd(q, k, v, mask)
    red = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
    plain = dab.attn_bwd(q, k, v, o, lse, do, mask, sched,
                         opts=dab.BwdOpts(spin_timeout_ns=0, flags=dab.DAB_BWD_PLAIN_ADD, grid=0))
    for a, b in zip(red, plain):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", ["serial", "descending_q", "shift"])
def test_bits_do_not_depend_on_the_grid(mask, sched):
    """The reduction order is fixed by the schedule's ranks alone, never by
    how many CTAs run or which CTA takes which unit."""
    B, H, S, d = 2, 3, 2048, 128          # N = 16: shift gangs of 16 (full) / 8 (causal)
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 12))
    o, lse = dab.attn_fwd(q, k, v, mask)
    base = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
    for grid in (64, 37, 16):
        ws = dab.new_workspace(B, H, S, d, mask, sched)
        got = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws,
                           opts=dab.BwdOpts(spin_timeout_ns=0, flags=0, grid=grid))
        assert dab.check_status(ws) == 0
        for a, b in zip(got, base):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), grid
