"""Device-side failure detection, injected from the host (no GPU fault).

A semaphore of the workspace is set to a value its waiters never see; the
bounded wait must run out, the kernel must return, and dab_check_status must
report DAB_ERR_TIMEOUT.  The context must stay usable afterwards.
"""
import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import TOL, case, oracle_ref, relerr


@pytest.mark.gpu
@pytest.mark.parametrize("sched", ["serial", "shift"])
def test_poisoned_semaphore_times_out(sched):
    B, H, S, d, mask = 1, 2, 256, 64, "full"
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 0))
    o, lse = dab.attn_fwd(q, k, v, mask)
    ws = dab.new_workspace(B, H, S, d, mask, sched)
    L = dab.workspace_layout(B, H, S, d, mask, sched)
    dab.bwd_preprocess(o, lse, do, mask, sched, ws)
    sem = ws[L.sem:L.D].view(torch.int32)  # [head][Q tile][8 sub-tiles][4 buffers]
    sem[32:64] = 1000  # every semaphore of Q tile 1 of head 0: nobody waits for 1000
    opts = dab.BwdOpts(spin_timeout_ns=50_000_000, flags=dab.DAB_BWD_SKIP_PREPROCESS, grid=0)
    dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws, opts=opts)
    assert dab.check_status(ws) == 5  # DAB_ERR_TIMEOUT
    # the context is still usable and a clean call is correct
    ws2 = dab.new_workspace(B, H, S, d, mask, sched)
    dq, dk, dv = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws2)
    assert dab.check_status(ws2) == 0
    ref = oracle_ref(B, H, S, d, 0, False)
    assert relerr(dq, ref["dq"]) < TOL


@pytest.mark.gpu
def test_bad_arguments_are_rejected_synchronously():
    q, k, v, do = (t.cuda() for t in case(1, 1, 256, 64, 0))
    o, lse = dab.attn_fwd(q, k, v, "full")
    with pytest.raises(dab.DabError) as e:
        dab.attn_bwd(q, k, v, o, lse, do, "full", "serial",
                     workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == 3  # DAB_ERR_WORKSPACE
