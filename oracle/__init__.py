"""Float64 CPU oracle for exact softmax attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm are the only users.  Nothing in the
product package imports this module, and this module imports nothing from the
product package.

The arithmetic lives in ``attn_oracle.c`` (plain C, float64, pthreads), which
writes out the definition of the attention gradient step by step; see the
header of that file for the steps and the passages they follow.  This module
only compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE float64 throughout)."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building if needed) and return a handle to the oracle library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    lib.oracle_attn_fwd_bwd.restype = ctypes.c_int
    lib.oracle_attn_fwd_bwd.argtypes = (
        [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        + [dp] * 4 + [dp] * 6 + [ctypes.c_int])
    lib.oracle_attn_bwd_given.restype = ctypes.c_int
    lib.oracle_attn_bwd_given.argtypes = (
        [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int]
        + [dp] * 6 + [dp] * 6 + [ctypes.c_int])
    lib.oracle_attn_fwd_bwd_block.restype = ctypes.c_int
    lib.oracle_attn_fwd_bwd_block.argtypes = (
        [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_void_p]
        + [dp] * 4 + [dp] * 6 + [ctypes.c_int])
    ip = ctypes.POINTER(ctypes.c_int)
    lib.oracle_attn_rows.restype = ctypes.c_int
    lib.oracle_attn_rows.argtypes = (
        [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int] + [dp] * 6
        + [ip, ctypes.c_int, ip, ctypes.c_int] + [dp] * 6 + [ctypes.c_int])
    return lib


def _f64(x) -> np.ndarray:
    """Exact widening to a contiguous float64 numpy array (bf16/f32 -> f64)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attn_fwd_bwd(q, k, v, dout, scale: float, causal: bool, tiles=None,
                 nthreads: int | None = None, lib=None) -> dict:
    """Forward + backward for inputs of shape [..., S, d] (leading dims = heads).

    `tiles`: optional block mask, [S/128][S/128] of 0/1 (row = query tile,
    column = key tile, 0 = masked), combined with `causal`.
    Returns a dict of float64 arrays: o, lse, D, dq, dk, dv.
    """
    lib = lib or load()
    q, k, v, dout = (_f64(t) for t in (q, k, v, dout))
    shape = q.shape
    S, d = shape[-2], shape[-1]
    BH = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    out = {n: np.empty(shape, np.float64) for n in ("o", "dq", "dk", "dv")}
    out["lse"] = np.empty(shape[:-1], np.float64)
    out["D"] = np.empty(shape[:-1], np.float64)
    tail = (_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["D"]),
            _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), int(nthreads or default_threads()))
    if tiles is None:
        rc = lib.oracle_attn_fwd_bwd(BH, S, d, float(scale), int(bool(causal)), *tail)
    else:
        t = np.ascontiguousarray(np.asarray(tiles) != 0, dtype=np.uint8)
        if t.shape != (S // 128, S // 128) or S % 128:
            raise ValueError("tiles must be [S/128][S/128]")
        rc = lib.oracle_attn_fwd_bwd_block(BH, S, d, float(scale), int(bool(causal)),
                                           t.ctypes.data_as(ctypes.c_void_p), *tail)
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd_bwd failed ({rc})")
    return out


def attn_bwd_given(q, k, v, o, lse, dout, scale: float, causal: bool,
                   nthreads: int | None = None, lib=None) -> dict:
    """Diagnostic backward using a supplied O and LSE (e.g. a GPU forward's)."""
    lib = lib or load()
    q, k, v, o, lse, dout = (_f64(t) for t in (q, k, v, o, lse, dout))
    shape = q.shape
    S, d = shape[-2], shape[-1]
    BH = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    out = {n: np.empty(shape, np.float64) for n in ("o", "dq", "dk", "dv")}
    out["lse"] = np.empty(shape[:-1], np.float64)
    out["D"] = np.empty(shape[:-1], np.float64)
    rc = lib.oracle_attn_bwd_given(
        BH, S, d, float(scale), int(bool(causal)),
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout),
        _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["D"]),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
        int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd_given failed ({rc})")
    return out


def attn_rows(q, k, v, dout, scale: float, causal: bool, qrows, krows,
              lse_all=None, D_all=None, nthreads: int | None = None, lib=None) -> dict:
    """Selected rows of one head ([S, d] inputs): O, LSE, D, dQ for `qrows`,
    dK, dV for `krows`.  `lse_all`/`D_all` ([S], from a whole-head run) skip
    the whole-head query pass that the key rows otherwise need."""
    lib = lib or load()
    q, k, v, dout = (_f64(t) for t in (q, k, v, dout))
    S, d = q.shape
    qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32))
    kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32))
    nq, nk = len(qr), len(kr)
    out = {"o": np.empty((nq, d)), "lse": np.empty(nq), "D": np.empty(nq),
           "dq": np.empty((nq, d)), "dk": np.empty((nk, d)), "dv": np.empty((nk, d))}
    la = _f64(lse_all) if lse_all is not None else None
    da = _f64(D_all) if D_all is not None else None
    ip = ctypes.POINTER(ctypes.c_int)
    rc = lib.oracle_attn_rows(
        S, d, float(scale), int(bool(causal)), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
        _ptr(la) if la is not None else None, _ptr(da) if da is not None else None,
        qr.ctypes.data_as(ip), nq, kr.ctypes.data_as(ip), nk,
        _ptr(out["o"]), _ptr(out["lse"]), _ptr(out["D"]), _ptr(out["dq"]),
        _ptr(out["dk"]), _ptr(out["dv"]), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_rows failed ({rc})")
    return out
