"""Deterministic attention backward for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libdab.so`` (``include/dab.h``):
argument marshalling only.  Every step of the forward and backward runs in the
library's CUDA kernels; if the library is missing this module raises instead of
falling back to anything else.  PyTorch is used for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import inputs  # noqa: F401  (seeded input generators)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdab.so")

MASKS = {"full": 0, "causal": 1}
SCHEDS = {"serial": 0, "descending": 1, "descending_q": 1, "shift": 2, "atomic": 3, "auto": 4}
SCHED_NAMES = ("serial", "descending_q", "shift", "atomic")
STATUS = {0: "DAB_OK", 1: "DAB_ERR_INVALID_ARG", 2: "DAB_ERR_UNSUPPORTED", 3: "DAB_ERR_WORKSPACE",
          4: "DAB_ERR_CUDA", 5: "DAB_ERR_TIMEOUT", 6: "DAB_ERR_DEVICE_BOUNDS"}
DAB_BWD_SKIP_PREPROCESS = 0x1
DAB_BWD_SKIP_CONVERT = 0x2
DAB_BWD_SKIP_MAIN = 0x4
DAB_BWD_PLAIN_ADD = 0x8
DAB_BWD_SEPARATE_CONVERT = 0x10
DAB_BWD_SHARE_GPU = 0x20

EXPORTED = (
    "dab_attn_fwd", "dab_bwd_workspace_size", "dab_attn_bwd", "dab_check_status",
    "dab_status_string", "dab_attn_bwd_ex", "dab_bwd_preprocess", "dab_bwd_workspace_layout",
    "dab_sched_units_per_head", "dab_sched_unit_steps", "dab_sched_step", "dab_sched_rank",
    "dab_sched_contributors", "dab_sched_gang_size", "dab_dag_simulate", "dab_dag_critical_path",
    "dab_dag_simulate_ways", "dab_sched_select", "dab_attn_bwd_host", "dab_bwd_host_workspace_size",
    "dab_attn_fwd_block", "dab_attn_bwd_block", "dab_bwd_block_workspace_size",
    "dab_selftest_mma", "dab_last_error_string", "dab_attn_bwd_noalloc", "dab_mma_peak",
    "dab_mma_peak_grid", "dab_noalloc_check_status",
)


class DabError(RuntimeError):
    def __init__(self, code: int, what: str):
        detail = ""
        if code == 4 and _lib is not None:
            detail = " (" + _lib.dab_last_error_string().decode() + ")"
        super().__init__(f"{what}: {STATUS.get(code, code)}{detail}")
        self.code = code


class BwdOpts(ctypes.Structure):
    _fields_ = [("spin_timeout_ns", ctypes.c_uint64), ("flags", ctypes.c_uint32),
                ("grid", ctypes.c_int32)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("status", "sem", "D", "lse2", "dqacc", "total")]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libdab.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise OSError(f"{path} is missing: build it with "
                      "`python -m deterministic_attn_backward_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.dab_attn_fwd.argtypes = [vp] * 5 + [i] * 4 + [f, i, vp, sz, vp]
    lib.dab_attn_fwd.restype = i
    lib.dab_bwd_workspace_size.argtypes = [i] * 6
    lib.dab_bwd_workspace_size.restype = sz
    lib.dab_attn_bwd.argtypes = [vp] * 9 + [i] * 4 + [f, i, i, vp, sz, vp]
    lib.dab_attn_bwd.restype = i
    lib.dab_attn_bwd_ex.argtypes = [vp] * 9 + [i] * 4 + [f, i, i, vp, sz, vp, ctypes.POINTER(BwdOpts)]
    lib.dab_attn_bwd_ex.restype = i
    lib.dab_bwd_preprocess.argtypes = [vp] * 3 + [i] * 6 + [vp, sz, vp]
    lib.dab_bwd_preprocess.restype = i
    lib.dab_bwd_workspace_layout.argtypes = [i] * 6 + [ctypes.POINTER(WsLayout)]
    lib.dab_bwd_workspace_layout.restype = i
    lib.dab_check_status.argtypes = [vp, vp]
    lib.dab_check_status.restype = i
    lib.dab_status_string.argtypes = [i]
    lib.dab_status_string.restype = ctypes.c_char_p
    lib.dab_last_error_string.argtypes = []
    lib.dab_last_error_string.restype = ctypes.c_char_p
    lib.dab_sched_units_per_head.argtypes = [i, i, i]
    lib.dab_sched_units_per_head.restype = i
    lib.dab_sched_unit_steps.argtypes = [i, i, i, i]
    lib.dab_sched_unit_steps.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    lib.dab_sched_step.argtypes = [i, i, i, i, i, ip, ip]
    lib.dab_sched_step.restype = i
    lib.dab_sched_rank.argtypes = [i, i, i, i, i]
    lib.dab_sched_rank.restype = i
    lib.dab_sched_contributors.argtypes = [i, i, i]
    lib.dab_sched_contributors.restype = i
    lib.dab_sched_gang_size.argtypes = [i, i, i]
    lib.dab_sched_gang_size.restype = i
    dp = ctypes.POINTER(ctypes.c_double)
    lib.dab_dag_simulate.argtypes = [i, i, i, i, i, ctypes.c_double, ctypes.c_double, i, dp, dp]
    lib.dab_dag_simulate.restype = i
    lib.dab_dag_simulate_ways.argtypes = [i, i, i, i, i, ctypes.c_double, ctypes.c_double, i, i, dp, dp]
    lib.dab_dag_simulate_ways.restype = i
    lib.dab_sched_select.argtypes = [i] * 5
    lib.dab_sched_select.restype = i
    lib.dab_bwd_host_workspace_size.argtypes = [i] * 7
    lib.dab_bwd_host_workspace_size.restype = sz
    lib.dab_attn_bwd_host.argtypes = [vp] * 9 + [i] * 4 + [f, i, i, vp, sz, i, vp]
    lib.dab_attn_bwd_host.restype = i
    lib.dab_attn_fwd_block.argtypes = [vp] * 5 + [i] * 4 + [f, vp, i, vp, sz, vp]
    lib.dab_attn_fwd_block.restype = i
    lib.dab_bwd_block_workspace_size.argtypes = [i] * 5
    lib.dab_bwd_block_workspace_size.restype = sz
    lib.dab_attn_bwd_block.argtypes = [vp] * 9 + [i] * 4 + [f, vp, i, i, vp, sz, vp]
    lib.dab_attn_bwd_block.restype = i
    lib.dab_dag_critical_path.argtypes = [i, i, i, ctypes.c_double, ctypes.c_double, i]
    lib.dab_dag_critical_path.restype = ctypes.c_double
    lib.dab_attn_bwd_noalloc.argtypes = [vp] * 9 + [i] * 4 + [f, i, i, vp]
    lib.dab_attn_bwd_noalloc.restype = i
    lib.dab_noalloc_check_status.argtypes = [vp]
    lib.dab_noalloc_check_status.restype = i
    lib.dab_selftest_mma.argtypes = [i] + [vp] * 10
    lib.dab_selftest_mma.restype = i
    lib.dab_mma_peak.argtypes = [i, vp, vp]
    lib.dab_mma_peak.restype = i
    lib.dab_mma_peak_grid.argtypes = []
    lib.dab_mma_peak_grid.restype = i
    _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        raise DabError(code, what)


def _mask(mask) -> int:
    return MASKS[mask] if isinstance(mask, str) else int(mask)


def _sched(sched) -> int:
    return SCHEDS[sched] if isinstance(sched, str) else int(sched)


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("expected [B, H, S, d] tensors")
    return tuple(int(x) for x in q.shape)


def _dev_bf16(t: torch.Tensor, device) -> torch.Tensor:
    if t.dtype != torch.bfloat16:
        raise TypeError("expected bfloat16 tensors")
    return t.to(device, non_blocking=True).contiguous()


def default_scale(d: int) -> float:
    return 1.0 / float(d) ** 0.5


def workspace_size(B, H, S, d, mask="full", sched="serial") -> int:
    return int(load_library().dab_bwd_workspace_size(B, H, S, d, _mask(mask), _sched(sched)))


def workspace_layout(B, H, S, d, mask="full", sched="serial") -> WsLayout:
    L = WsLayout()
    _check(load_library().dab_bwd_workspace_layout(B, H, S, d, _mask(mask), _sched(sched),
                                                   ctypes.byref(L)), "dab_bwd_workspace_layout")
    return L


def block_workspace_size(B, H, S, d, sched="descending_q") -> int:
    n = int(load_library().dab_bwd_block_workspace_size(B, H, S, d, _sched(sched)))
    if n == 0:
        raise DabError(1, "dab_bwd_block_workspace_size")
    return n


def new_workspace(B, H, S, d, mask="full", sched="serial", device="cuda", block=False) -> torch.Tensor:
    n = block_workspace_size(B, H, S, d, sched) if block else workspace_size(B, H, S, d, mask, sched)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _tiles(tiles, S, dev):
    """Block mask as a contiguous uint8 [S/128, S/128] CUDA tensor."""
    t = torch.as_tensor(tiles)
    if tuple(t.shape) != (S // 128, S // 128):
        raise ValueError("tiles must be [S/128, S/128]")
    return (t != 0).to(device=dev, dtype=torch.uint8).contiguous()


def attn_fwd(q, k, v, mask="full", scale=None, workspace=None, out=None, lse=None, tiles=None):
    """O (bf16 [B,H,S,d]) and LSE (f32 [B,H,S]) on q's CUDA device.
    `tiles`: optional block mask [S/128, S/128] (dab_attn_fwd_block)."""
    lib = load_library()
    B, H, S, d = _shape(q)
    dev = q.device if q.is_cuda else torch.device("cuda")
    q, k, v = (_dev_bf16(t, dev) for t in (q, k, v))
    o = out if out is not None else torch.empty_like(q)
    lse_t = lse if lse is not None else torch.empty((B, H, S), dtype=torch.float32, device=dev)
    ws_ptr, ws_n = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    sc = float(scale if scale is not None else default_scale(d))
    if tiles is None:
        _check(lib.dab_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse_t.data_ptr(), B, H, S, d, sc, _mask(mask), ws_ptr, ws_n,
                                _stream(dev)), "dab_attn_fwd")
    else:
        t = _tiles(tiles, S, dev)
        _check(lib.dab_attn_fwd_block(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse_t.data_ptr(), B, H, S, d, sc, t.data_ptr(), _mask(mask),
                                      ws_ptr, ws_n, _stream(dev)), "dab_attn_fwd_block")
    return o, lse_t


def host_workspace_size(B, H, S, d, mask="full", sched="serial", chunks=0) -> int:
    n = load_library().dab_bwd_host_workspace_size(B, H, S, d, _mask(mask), _sched(sched), chunks)
    if n == 0:
        raise DabError(1, "dab_bwd_host_workspace_size")
    return n


def new_host_workspace(B, H, S, d, mask="full", sched="serial", chunks=0, device="cuda"):
    """Device workspace of the host-buffer path (dab_attn_bwd_host)."""
    return torch.empty(host_workspace_size(B, H, S, d, mask, sched, chunks), dtype=torch.uint8,
                       device=device)


def _attn_bwd_host(q, k, v, o, lse, dout, mask, sched, scale, workspace, out, chunks):
    """CPU tensors through dab_attn_bwd_host (copies overlapped with the
    computation inside the library); returns once the gradients are in host
    memory.  Pinned inputs and outputs give asynchronous copies."""
    lib = load_library()
    B, H, S, d = _shape(q)
    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v, o, dout = (t.contiguous() if t.dtype == torch.bfloat16 else t.to(torch.bfloat16).contiguous()
                        for t in (q, k, v, o, dout))
    lse = lse.contiguous()
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    if workspace is None:
        workspace = new_host_workspace(B, H, S, d, mask, sched, chunks, dev)
    if out is None:
        out = tuple(torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(3))
    dq, dk, dv = out
    _check(lib.dab_attn_bwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, d,
                                 float(scale if scale is not None else default_scale(d)), _mask(mask),
                                 _sched(sched), workspace.data_ptr(), workspace.numel(), chunks,
                                 _stream(dev)), "dab_attn_bwd_host")
    torch.cuda.current_stream(dev).synchronize()
    return dq, dk, dv


def attn_bwd(q, k, v, o, lse, dout, mask="full", sched="serial", scale=None, workspace=None,
             out=None, opts: BwdOpts | None = None, chunks: int = 0, tiles=None):
    """dQ, dK, dV (bf16 [B,H,S,d]) through the C ABI.

    Device tensors are used in place (dab_attn_bwd / dab_attn_bwd_ex).  CPU
    tensors go through dab_attn_bwd_host, which copies them to the device
    and the gradients back, overlapped with the computation in `chunks`
    groups of heads (0 = the library's default); `workspace` is then the
    device workspace of new_host_workspace() and `out` host tensors.
    """
    lib = load_library()
    B, H, S, d = _shape(q)
    host = not q.is_cuda
    if tiles is not None:
        return _attn_bwd_block(q, k, v, o, lse, dout, mask, sched, scale, workspace, out, tiles)
    if host:
        if opts is not None:
            raise ValueError("opts apply to device tensors only")
        return _attn_bwd_host(q, k, v, o, lse, dout, mask, sched, scale, workspace, out, chunks)
    dev = q.device
    q, k, v, o, dout = (_dev_bf16(t, dev) for t in (q, k, v, o, dout))
    lse = lse.to(dev, non_blocking=True).contiguous()
    if lse.dtype != torch.float32:
        raise TypeError("lse must be float32")
    if workspace is None:
        workspace = new_workspace(B, H, S, d, mask, sched, dev)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q))
    dq, dk, dv = out
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
            dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, d,
            float(scale if scale is not None else default_scale(d)), _mask(mask), _sched(sched),
            workspace.data_ptr(), workspace.numel(), _stream(dev))
    if opts is None:
        _check(lib.dab_attn_bwd(*args), "dab_attn_bwd")
    else:
        _check(lib.dab_attn_bwd_ex(*args, ctypes.byref(opts)), "dab_attn_bwd_ex")
    return dq, dk, dv


def _attn_bwd_block(q, k, v, o, lse, dout, mask, sched, scale, workspace, out, tiles):
    """dab_attn_bwd_block on CUDA tensors (mask: "full" or "causal")."""
    lib = load_library()
    B, H, S, d = _shape(q)
    dev = q.device
    q, k, v, o, dout = (_dev_bf16(t, dev) for t in (q, k, v, o, dout))
    t = _tiles(tiles, S, dev)
    if workspace is None:
        workspace = new_workspace(B, H, S, d, sched=sched, device=dev, block=True)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(q), torch.empty_like(q))
    dq, dk, dv = out
    _check(lib.dab_attn_bwd_block(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, S, d,
                                  float(scale if scale is not None else default_scale(d)), t.data_ptr(),
                                  _mask(mask), _sched(sched), workspace.data_ptr(), workspace.numel(),
                                  _stream(dev)), "dab_attn_bwd_block")
    return dq, dk, dv


def bwd_preprocess(o, lse, dout, mask, sched, workspace):
    lib = load_library()
    B, H, S, d = _shape(o)
    _check(lib.dab_bwd_preprocess(o.data_ptr(), lse.data_ptr(), dout.data_ptr(), B, H, S, d,
                                  _mask(mask), _sched(sched), workspace.data_ptr(),
                                  workspace.numel(), _stream(o.device)), "dab_bwd_preprocess")


def check_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream and return the workspace status code."""
    return int(load_library().dab_check_status(workspace.data_ptr(), _stream(workspace.device)))


# ------------------------------------------------------------ schedules (host)
def sched_units_per_head(sched, mask, N) -> int:
    return load_library().dab_sched_units_per_head(_sched(sched), _mask(mask), N)


def sched_unit_steps(sched, mask, N, u) -> int:
    return load_library().dab_sched_unit_steps(_sched(sched), _mask(mask), N, u)


def sched_unit(sched, mask, N, u):
    """[(kv_tile, q_tile), ...] of unit u, in execution order."""
    lib = load_library()
    kv, qt = ctypes.c_int(), ctypes.c_int()
    out = []
    for t in range(sched_unit_steps(sched, mask, N, u)):
        _check(lib.dab_sched_step(_sched(sched), _mask(mask), N, u, t, ctypes.byref(kv),
                                  ctypes.byref(qt)), "dab_sched_step")
        out.append((kv.value, qt.value))
    return out


def sched_rank(sched, mask, N, i, j) -> int:
    return load_library().dab_sched_rank(_sched(sched), _mask(mask), N, i, j)


def sched_contributors(mask, N, j) -> int:
    return load_library().dab_sched_contributors(_mask(mask), N, j)


def sched_gang_size(sched, mask, N) -> int:
    return load_library().dab_sched_gang_size(_sched(sched), _mask(mask), N)


def dag_simulate(sched, mask, N, heads, ctas, wc=1.0, wr=0.0, reducer_depth=0, ways=1):
    """(status, makespan, busy_fraction) of the schedule's DAG model."""
    mk, busy = ctypes.c_double(), ctypes.c_double()
    rc = load_library().dab_dag_simulate_ways(_sched(sched), _mask(mask), N, heads, ctas, wc, wr,
                                              reducer_depth, ways, ctypes.byref(mk),
                                              ctypes.byref(busy))
    return rc, mk.value, busy.value


def sched_select(mask, B: int, H: int, S: int, ctas: int) -> str:
    """The deterministic schedule the library runs for DAB_SCHED_AUTO on
    `ctas` CTAs (the SM count of the device)."""
    r = load_library().dab_sched_select(_mask(mask), B, H, S, ctas)
    if r < 0:
        raise DabError(1, "dab_sched_select")
    return SCHED_NAMES[r]


def dag_critical_path(sched, mask, N, wc=1.0, wr=0.0, reducer_depth=0) -> float:
    return load_library().dab_dag_critical_path(_sched(sched), _mask(mask), N, wc, wr, reducer_depth)


def selftest_mma(d: int, x, y, z, pm):
    """Run the tensor-core operand self-test; returns (out0, out1, out2, out3)."""
    lib = load_library()
    dev = x.device
    out0 = torch.empty((128, 128), dtype=torch.float32, device=dev)
    out1 = torch.empty((128, d), dtype=torch.float32, device=dev)
    out2 = torch.empty((128, d), dtype=torch.float32, device=dev)
    out3 = torch.empty((128, 128 if d == 128 else 64), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    _check(lib.dab_selftest_mma(d, x.data_ptr(), y.data_ptr(), z.data_ptr(), pm.data_ptr(),
                                out0.data_ptr(), out1.data_ptr(), out2.data_ptr(), out3.data_ptr(),
                                ws.data_ptr(), _stream(dev)), "dab_selftest_mma")
    _check(check_status(ws), "selftest device status")
    return out0, out1, out2, out3


def mma_peak(iters: int = 100000, device=None) -> dict:
    """Dense bf16 tensor throughput of the library's own tcgen05 path: one
    timed launch of `iters` x 4 MMAs (128 x 256 x 16) per SM, after one
    untimed warm-up launch.  Returns {"tflops", "ms", "grid", "iters"}."""
    lib = load_library()
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    stream = _stream(dev)
    grid = lib.dab_mma_peak_grid()
    _check(lib.dab_mma_peak(max(1, iters // 10), ws.data_ptr(), stream), "dab_mma_peak")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    _check(lib.dab_mma_peak(iters, ws.data_ptr(), stream), "dab_mma_peak")
    e1.record()
    e1.synchronize()
    _check(check_status(ws), "dab_mma_peak device status")
    ms = e0.elapsed_time(e1)
    flops = float(grid) * iters * 4 * 2 * 128 * 256 * 16
    return {"tflops": flops / (ms * 1e-3) / 1e12, "ms": ms, "grid": grid, "iters": iters}
