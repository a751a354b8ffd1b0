"""Block masks (128 x 128 tiles, optionally with the causal mask): the GPU
forward and backward against the float64 oracle's block mode, their edge
cases, and the schedules' bit-level properties under a mask."""
import numpy as np
import pytest
import torch

import oracle
import deterministic_attn_backward_gb300 as dab
from gpu_common import TOL, case, relerr


def pattern(name, N, seed=0):
    i, j = np.meshgrid(np.arange(N), np.arange(N))   # j: query tile (row), i: key tile (column)
    if name == "band":                               # sliding window of three tiles
        return (np.abs(i - j) <= 1).astype(np.uint8)
    if name == "documents":                          # block diagonal: documents of whole tiles
        doc = np.minimum(np.arange(N) // 2, 2)
        return (doc[j] == doc[i]).astype(np.uint8)
    if name == "random":
        return (np.random.default_rng(seed).random((N, N)) < 0.5).astype(np.uint8)
    if name == "empty":                              # an empty query tile and an empty key tile
        t = np.ones((N, N), np.uint8)
        t[1, :] = 0
        t[:, 2] = 0
        return t
    raise ValueError(name)


def _check_outputs(o, lse, grads, ref):
    lse_g = lse.double().cpu().numpy()
    neg = np.isneginf(ref["lse"])
    assert np.array_equal(np.isneginf(lse_g), neg)
    assert np.max(np.abs(lse_g[~neg] - ref["lse"][~neg])) < 1e-3
    assert relerr(o, ref["o"]) < TOL
    for name, g in zip(("dq", "dk", "dv"), grads):
        assert relerr(g, ref[name]) < TOL, name


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1, 2, 640, 64), (2, 2, 768, 128)])
@pytest.mark.parametrize("name", ["band", "documents", "random", "empty"])
@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_parity(shape, name, causal):
    B, H, S, d = shape
    N = S // 128
    t = pattern(name, N, seed=S + d)
    q, k, v, do = case(B, H, S, d, 31)
    ref = oracle.attn_fwd_bwd(q, k, v, do, d ** -0.5, causal, tiles=t)
    mask = "causal" if causal else "full"
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = dab.attn_fwd(qd, kd, vd, mask, tiles=t)
    for sched in ("serial", "descending_q", "atomic"):
        grads = dab.attn_bwd(qd, kd, vd, o, lse, dod, mask, sched, tiles=t)
        _check_outputs(o, lse, grads, ref)


@pytest.mark.gpu
@pytest.mark.parametrize("mask", ["full", "causal"])
@pytest.mark.parametrize("sched", ["serial", "descending_q"])
@pytest.mark.parametrize("d", [64, 128])
def test_all_visible_block_mask_gives_the_unmasked_bits(mask, sched, d):
    """Every tile visible: the same visit order and ranks as without a mask,
    hence the same bits (forward and backward)."""
    B, H, S = 2, 3, 768
    q, k, v, do = (x.cuda() for x in case(B, H, S, d, 32))
    t = np.ones((S // 128, S // 128), np.uint8)
    o, lse = dab.attn_fwd(q, k, v, mask)
    ob, lseb = dab.attn_fwd(q, k, v, mask, tiles=t)
    assert torch.equal(o.view(torch.int16), ob.view(torch.int16)) and torch.equal(lse, lseb)
    plain = dab.attn_bwd(q, k, v, o, lse, do, mask, sched)
    block = dab.attn_bwd(q, k, v, o, lse, do, mask, sched, tiles=t)
    for a, b in zip(plain, block):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.gpu
def test_block_mask_bitwise_repeatable_and_serial_descending_share_dq():
    B, H, S, d = 2, 4, 1024, 128
    q, k, v, do = (x.cuda() for x in case(B, H, S, d, 33))
    t = pattern("random", S // 128, seed=5)
    o, lse = dab.attn_fwd(q, k, v, "causal", tiles=t)
    runs = [dab.attn_bwd(q, k, v, o, lse, do, "causal", "descending_q", tiles=t) for _ in range(5)]
    for r in runs[1:]:
        for a, b in zip(runs[0], r):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ser = dab.attn_bwd(q, k, v, o, lse, do, "causal", "serial", tiles=t)
    assert torch.equal(ser[0].view(torch.int16), runs[0][0].view(torch.int16))


@pytest.mark.gpu
def test_block_mask_rejects_shift_and_nulls():
    lib = dab.load_library()
    B, H, S, d = 1, 1, 256, 64
    q, k, v, do = (x.cuda() for x in case(B, H, S, d, 34))
    t = np.ones((2, 2), np.uint8)
    o, lse = dab.attn_fwd(q, k, v, "full", tiles=t)
    with pytest.raises(dab.DabError) as e:
        dab.attn_bwd(q, k, v, o, lse, do, "full", "shift", tiles=t,
                     workspace=dab.new_workspace(B, H, S, d, sched="serial", block=True))
    assert e.value.code == 2
    assert lib.dab_bwd_block_workspace_size(B, H, S, d, 2) == 0
