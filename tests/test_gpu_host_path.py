"""dab_attn_bwd_host: the backward on host buffers, copies overlapped with the
computation in groups of heads (consecutive groups on two streams, so their
kernels overlap).  Each group is an ordinary backward on that range of heads,
so for an explicit deterministic schedule the gradients are bitwise those of
the device path, whatever the group count and whether the host buffers are
pinned or not; the workspace's status header reports the first device error
of any group (none here)."""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import case


@pytest.mark.gpu
@pytest.mark.parametrize("shape,mask,sched", [
    ((2, 3, 640, 128), "full", "serial"),
    ((1, 5, 768, 64), "causal", "shift"),
    ((3, 2, 512, 128), "causal", "descending_q"),
])
@pytest.mark.parametrize("chunks", [0, 1, 2, 4, 64])
def test_host_path_matches_device_path(shape, mask, sched, chunks):
    B, H, S, d = shape
    q, k, v, do = case(B, H, S, d, 21)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = dab.attn_fwd(qd, kd, vd, mask)
    want = dab.attn_bwd(qd, kd, vd, o, lse, dod, mask, sched)
    pinned = chunks % 2 == 0   # both pinned and pageable host buffers
    host = [t.cpu() for t in (q, k, v, o, lse, do)]
    if pinned:
        host = [t.pin_memory() for t in host]
    ws = dab.new_host_workspace(B, H, S, d, mask, sched, chunks)
    ws.fill_(0xFF)  # the status header must be written by the call itself
    got = dab.attn_bwd(*host, mask=mask, sched=sched, workspace=ws, chunks=chunks)
    assert dab.check_status(ws) == 0
    for g, w in zip(got, want):
        assert not g.is_cuda
        assert torch.equal(g.view(torch.int16), w.cpu().view(torch.int16))


@pytest.mark.gpu
def test_host_path_atomic_within_tolerance_and_workspace_reuse():
    B, H, S, d = 2, 2, 384, 64
    q, k, v, do = case(B, H, S, d, 22)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = dab.attn_fwd(qd, kd, vd, "full")
    want = dab.attn_bwd(qd, kd, vd, o, lse, dod, "full", "serial")
    ws = dab.new_host_workspace(B, H, S, d, "full", "atomic", 3)
    host = [t.cpu().pin_memory() for t in (q, k, v, o, lse, do)]
    out = tuple(torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(3))
    for _ in range(2):  # the same device workspace twice in a row
        got = dab.attn_bwd(*host, mask="full", sched="atomic", workspace=ws, out=out, chunks=3)
        assert dab.check_status(ws) == 0
        for g, w in zip(got, want):
            err = (g.double() - w.cpu().double()).abs().max() / w.cpu().double().abs().max()
            assert err < 1e-2
