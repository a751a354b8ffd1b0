"""dab_attn_bwd_noalloc: the backward for callers that cannot allocate.

Callers such as a plugin inside a framework that owns all device memory, or a
latency-critical loop that must not call cudaMalloc (it can synchronise the
device), cannot hand the library a workspace.  This entry point takes its
workspace from a fixed array inside the library instead.  The test calls it
through the C ABI twice in a row and checks both results against the
ordinary, workspace-taking entry point, within the tolerance of the parity
tests; it also checks that a problem too large for the array is refused.

The entry point's status word lives in the library's array, and
dab_noalloc_check_status() must report each call as clean.  A further test
checks the one promise of the entry point itself: after a warm-up call, a
call changes the device's free memory by nothing.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import deterministic_attn_backward_gb300 as dab
from gpu_common import TOL, case

MASKS = {"full": 0, "causal": 1}
SCHEDS = {"serial": 0, "descending_q": 1, "shift": 2, "atomic": 3}


def _noalloc(q, k, v, o, lse, do, mask, sched, out):
    lib = dab.load_library()
    B, H, S, d = q.shape
    dq, dk, dv = out
    stream = torch.cuda.current_stream().cuda_stream
    return lib.dab_attn_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), do.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, d, ctypes.c_float(d ** -0.5),
        MASKS[mask], SCHEDS[sched], ctypes.c_void_p(stream))


def _status():
    lib = dab.load_library()
    return lib.dab_noalloc_check_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _rel(a, b):
    a, b = a.double(), b.double()
    return ((a - b).abs().max() / b.abs().max()).item()


@pytest.mark.gpu
@pytest.mark.parametrize("shape,mask,sched", [
    ((1, 2, 256, 64), "full", "serial"),
    ((2, 3, 640, 128), "full", "shift"),
    ((1, 2, 768, 128), "causal", "shift"),
    ((2, 2, 512, 64), "causal", "descending_q"),
    ((1, 3, 384, 128), "full", "atomic"),
])
def test_noalloc_matches_workspace_entry_point(shape, mask, sched):
    B, H, S, d = shape
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 5))
    o, lse = dab.attn_fwd(q, k, v, mask)
    want = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
    results = []
    for _ in range(2):  # two calls in a row share the library's scratch array
        out = tuple(torch.full_like(q, float("nan")) for _ in range(3))
        rc = _noalloc(q, k, v, o, lse, do, mask, sched, out)
        assert rc == 0, dab.STATUS.get(rc, rc)
        st = _status()
        assert st == 0, dab.STATUS.get(st, st)
        results.append(out)
    for out in results:
        for got, ref in zip(out, want):
            assert torch.isfinite(got).all()
            assert _rel(got, ref) < TOL
    if sched != "atomic":  # same kernels, same reduction order: same bits
        for got, ref in zip(results[1], want):
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = dab.load_library()
    B, H, S, d = 4, 16, 8192, 128  # needs far more than the built-in array
    assert dab.workspace_size(B, H, S, d) > 32 << 20
    p = ctypes.c_void_p(256)  # never dereferenced: the size check comes first
    rc = lib.dab_attn_bwd_noalloc(p, p, p, p, p, p, p, p, p, B, H, S, d, ctypes.c_float(0.088),
                                  0, 0, None)
    assert rc == 3  # DAB_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_call_leaves_free_device_memory_unchanged():
    B, H, S, d = 1, 2, 512, 128
    q, k, v, do = (t.cuda() for t in case(B, H, S, d, 6))
    o, lse = dab.attn_fwd(q, k, v, "causal")
    out = tuple(torch.empty_like(q) for _ in range(3))
    # warm-up: loads the kernels and looks up the array's address
    assert _noalloc(q, k, v, o, lse, do, "causal", "descending_q", out) == 0
    assert _status() == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    assert _noalloc(q, k, v, o, lse, do, "causal", "descending_q", out) == 0
    assert _status() == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
