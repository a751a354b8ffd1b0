"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments synchronously (no GPU needed: no compute call is made)."""
import ctypes
import os
import re

import pytest

import deterministic_attn_backward_gb300 as dab

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = set()
    for fn in os.listdir(INCLUDE):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(INCLUDE, fn)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(dab_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from deterministic_attn_backward_gb300 import build
    build.build()
    return dab.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dab.EXPORTED)


def test_status_strings(lib):
    for code, name in dab.STATUS.items():
        assert lib.dab_status_string(code).decode() == name


def test_auto_schedule_workspace_is_the_ordered_one(lib):
    for B, H, S, d in ((1, 1, 128, 64), (2, 16, 8192, 128)):
        for mask in (0, 1):
            assert lib.dab_bwd_workspace_size(B, H, S, d, mask, 4) == lib.dab_bwd_workspace_size(
                B, H, S, d, mask, 1) > 0


def test_workspace_layout(lib):
    B, H, S, d = 2, 16, 8192, 128
    L = dab.workspace_layout(B, H, S, d, "causal", "descending_q")
    rows = B * H * S
    assert L.status == 0 and L.sem == 256
    ways = 4  # ordered schedules: four interleaved accumulation buffers
    assert L.D >= L.sem + 4 * 8 * ways * B * H * (S // 128)
    assert L.lse2 >= L.D + 4 * rows and L.dqacc >= L.lse2 + 4 * rows
    assert L.total >= L.dqacc + ways * 4 * rows * d
    La = dab.workspace_layout(B, H, S, d, "causal", "atomic")  # one buffer
    assert La.total >= La.dqacc + 4 * rows * d and La.total < L.total
    for off in (L.sem, L.D, L.lse2, L.dqacc, L.total):
        assert off % 256 == 0
    assert dab.workspace_size(B, H, S, d, "causal", "descending_q") == L.total
    # any S: a partial last tile pads D and LSE2 to whole tiles per head
    Lr = dab.workspace_layout(B, H, 200, d, "full", "serial")
    assert Lr.lse2 >= Lr.D + 4 * B * H * 256 and Lr.dqacc >= Lr.lse2 + 4 * B * H * 256
    assert Lr.total >= Lr.dqacc + 4 * 4 * B * H * 200 * d
    assert lib.dab_bwd_workspace_size(B, H, 0, d, 0, 0) > 0            # empty problem
    assert lib.dab_bwd_workspace_size(B, H, -1, d, 0, 0) == 0          # negative length
    assert lib.dab_bwd_workspace_size(B, H, S, 96, 0, 0) == 0       # d not 64/128
    assert lib.dab_bwd_workspace_size(B, H, S, d, 2, 0) == 0        # bad mask


def test_bad_arguments_rejected_without_touching_the_device(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    nul = None
    big = 1 << 30
    call = lambda *a: lib.dab_attn_bwd(*a)
    # null / misaligned pointers
    assert call(nul, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, p, big, None) == 1
    assert call(ctypes.c_void_p(17), p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, p, big,
                None) == 1
    # bad shape / enum / scale
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, -128, 64, 0.125, 0, 0, p, big, None) == 1
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 128, 80, 0.125, 0, 0, p, big, None) == 1
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 7, p, big, None) == 1
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, -1.0, 0, 0, p, big, None) == 1
    # causal shift with an odd tile count
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 384, 64, 0.125, 1, 2, p, big, None) == 2
    # workspace missing or too small
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, nul, 0, None) == 3
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, p, 64, None) == 3
    # forward
    assert lib.dab_attn_fwd(nul, p, p, p, p, 1, 1, 128, 64, 0.125, 0, nul, 0, None) == 1
    assert lib.dab_attn_fwd(p, p, p, p, p, 1, 1, 128, 64, 0.125, 3, nul, 0, None) == 1
    assert lib.dab_check_status(nul, None) == 1
    # DAB_SCHED_AUTO (4): accepted by the backward entry points, not by the
    # schedule introspection functions
    assert lib.dab_sched_units_per_head(4, 0, 8) == -1
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, -128, 64, 0.125, 0, 4, p, big, None) == 1
    assert call(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 5, p, big, None) == 1
    # host-buffer path: sizes, null pointers and workspace checked before any CUDA call
    assert lib.dab_bwd_host_workspace_size(2, 3, 640, 128, 0, 0, 2) > lib.dab_bwd_workspace_size(
        1, 3, 640, 128, 0, 0)
    assert lib.dab_bwd_host_workspace_size(2, 3, -600, 128, 0, 0, 2) == 0
    assert lib.dab_bwd_host_workspace_size(2, 3, 640, 80, 0, 0, 2) == 0
    hcall = lambda *a: lib.dab_attn_bwd_host(*a)
    assert hcall(nul, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, p, big, 0, None) == 1
    assert hcall(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, nul, big, 0, None) == 3
    assert hcall(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, p, 64, 0, None) == 3
    assert hcall(p, p, p, p, p, p, p, p, p, 1, 1, 128, 64, 0.125, 0, 0, ctypes.c_void_p(16 + 256), big,
                 0, None) == 3
    # block masks: null tile table, causal flag, SHIFT
    assert lib.dab_attn_fwd_block(p, p, p, p, p, 1, 1, 256, 64, 0.125, nul, 0, nul, 0, None) == 1
    assert lib.dab_attn_fwd_block(p, p, p, p, p, 1, 1, 256, 64, 0.125, p, 2, nul, 0, None) == 1
    assert lib.dab_attn_bwd_block(p, p, p, p, p, p, p, p, p, 1, 1, 256, 64, 0.125, nul, 0, 0, p, big,
                                  None) == 1
    assert lib.dab_attn_bwd_block(p, p, p, p, p, p, p, p, p, 1, 1, 256, 64, 0.125, p, 0, 2, p, big,
                                  None) == 2
    assert lib.dab_bwd_block_workspace_size(1, 1, 256, 64, 2) == 0
    assert lib.dab_bwd_block_workspace_size(1, 1, 256, 64, 1) > lib.dab_bwd_workspace_size(
        1, 1, 256, 64, 0, 1)
    assert lib.dab_bwd_block_workspace_size(1, 1, 256, 64, 4) == lib.dab_bwd_block_workspace_size(
        1, 1, 256, 64, 1)
    # tensor-peak measurement: iteration count and status buffer are checked first
    assert lib.dab_mma_peak(0, p, None) == 1
    assert lib.dab_mma_peak(1 << 23, p, None) == 1
    assert lib.dab_mma_peak(1000, ctypes.c_void_p(17), None) == 1


def test_host_workspace_holds_two_group_workspaces(lib):
    """The host-buffer path: a status header and per-group slots, device
    copies of the nine tensors, and one backward workspace per compute
    stream (two once there are at least two groups)."""
    rnd = lambda x: (x + 255) // 256 * 256
    B, H, S, d = 2, 3, 640, 128
    bh = B * H
    copies = 8 * rnd(bh * S * d * 2) + rnd(bh * S * 4)
    for chunks, per in ((1, 6), (2, 3), (6, 1)):
        group_ws = rnd(lib.dab_bwd_workspace_size(1, per, S, d, 0, 1))
        size = lib.dab_bwd_host_workspace_size(B, H, S, d, 0, 1, chunks)
        want = 256 + rnd(8 * chunks) + copies + (2 if chunks > 1 else 1) * group_ws
        assert size == want, (chunks, size, want)
