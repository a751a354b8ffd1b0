"""Pins that tie the float64 oracle to facts other than itself.

Each pin takes an oracle library handle, so the same checks run against the
committed oracle and against deliberately broken copies of it (the mutation
tests).  A pin raises AssertionError on failure.

What pins what:
  * finite differences   -- the backward (dQ, dK, dV) against the oracle's own
                            forward, by central differences of L = sum(dO * O);
  * hand-worked example  -- forward and backward on a 2-token case derived on
                            paper (tests/golden/two_key_worked_example.json);
  * closed forms         -- S = 1, Q = 0 (full and causal), causal row 0;
  * invariants           -- sum_c dK_c = 0, sum_c dV_c = sum_r dO_r, shift
                            invariance in K and V, key permutation, linearity;
  * torch autograd       -- an independent gradient engine on tiny inputs.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _run(lib, q, k, v, do, scale, causal):
    return oracle.attn_fwd_bwd(q, k, v, do, scale, causal, nthreads=2, lib=lib)


def _relerr(a, b):
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def pin_finite_differences(lib, tol=1e-6):
    """dQ, dK, dV equal central differences of L = sum(dO * O) (both masks)."""
    rng = np.random.default_rng(1234)
    h = 1e-6
    for causal in (False, True):
        for S, d in ((1, 4), (3, 4), (5, 8)):
            q, k, v, do = (_rand(rng, 1, S, d) for _ in range(4))
            scale = 0.7
            ref = _run(lib, q, k, v, do, scale, causal)

            def loss(qq, kk, vv):
                o = _run(lib, qq, kk, vv, do, scale, causal)["o"]
                return float(np.sum(do * o))

            for name, x, g in (("dq", q, ref["dq"]), ("dk", k, ref["dk"]),
                               ("dv", v, ref["dv"])):
                fd = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    xp = x.copy(); xp[idx] += h
                    xm = x.copy(); xm[idx] -= h
                    args_p = [q, k, v]; args_m = [q, k, v]
                    pos = {"dq": 0, "dk": 1, "dv": 2}[name]
                    args_p[pos] = xp; args_m[pos] = xm
                    fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
                err = float(np.max(np.abs(fd - g)))
                ref_mag = max(float(np.max(np.abs(fd))), 1e-3)
                assert err / ref_mag < tol, (
                    f"finite differences: {name} causal={causal} S={S} d={d}: "
                    f"rel err {err / ref_mag:.3e}")


def _golden_value(x):
    if isinstance(x, list):
        return [_golden_value(e) for e in x]
    if isinstance(x, str):
        coef = 1.0
        s = x
        if s.endswith("ln3"):
            c = s[:-3]
            coef = float(c) if c not in ("", "+") else 1.0
            if c == "-":
                coef = -1.0
            return coef * math.log(3.0)
        if s.startswith("ln"):
            return math.log(float(s[2:]))
        return float(s)
    return float(x)


def pin_worked_example(lib, tol=1e-12):
    """Forward and backward equal the hand-derived two-token example."""
    with open(os.path.join(GOLDEN, "two_key_worked_example.json")) as f:
        g = json.load(f)
    inp = {n: np.array(_golden_value(g["inputs"][n]), np.float64)[None]
           for n in ("q", "k", "v", "dout")}
    for mask in ("full", "causal"):
        out = _run(lib, inp["q"], inp["k"], inp["v"], inp["dout"],
                   g["inputs"]["scale"], mask == "causal")
        for name in ("lse", "o", "D", "dq", "dk", "dv"):
            want = np.array(_golden_value(g[mask][name]), np.float64)[None]
            got = out[name]
            assert np.allclose(got, want, rtol=0, atol=tol), (
                f"worked example {mask}/{name}: got {got.ravel()}, want {want.ravel()}")


def pin_closed_forms(lib, tol=1e-12):
    rng = np.random.default_rng(7)
    scale = 0.37
    # S = 1: a single key -> P = 1, O = V, LSE = scale q.k, all of dQ, dK vanish.
    for causal in (False, True):
        q, k, v, do = (_rand(rng, 2, 1, 6) for _ in range(4))
        out = _run(lib, q, k, v, do, scale, causal)
        assert np.allclose(out["o"], v, atol=tol)
        assert np.allclose(out["lse"][..., 0], scale * np.sum(q * k, -1)[..., 0], atol=tol)
        assert np.allclose(out["dv"], do, atol=tol)
        assert np.max(np.abs(out["dq"])) < tol and np.max(np.abs(out["dk"])) < tol
    # Q = 0, full mask: uniform attention.
    S, d = 7, 5
    k, v, do = (_rand(rng, 1, S, d) for _ in range(3))
    q = np.zeros((1, S, d))
    out = _run(lib, q, k, v, do, scale, False)
    assert np.allclose(out["lse"], math.log(S), atol=tol), "Q=0 full: LSE = ln S"
    vbar = v.mean(axis=1, keepdims=True)
    assert np.allclose(out["o"], np.broadcast_to(vbar, v.shape), atol=tol)
    assert np.max(np.abs(out["dk"])) < tol, "Q=0: dK = 0"
    assert np.allclose(out["dv"], np.broadcast_to(do.sum(1, keepdims=True) / S, v.shape), atol=tol)
    # dQ_r = (scale/S) sum_c (dO_r . (v_c - vbar)) k_c
    want = np.zeros_like(q)
    for r in range(S):
        for c in range(S):
            want[0, r] += (scale / S) * np.dot(do[0, r], v[0, c] - vbar[0, 0]) * k[0, c]
    assert np.allclose(out["dq"], want, atol=1e-12)
    # Q = 0, causal: row r averages keys 0..r.
    out = _run(lib, q, k, v, do, scale, True)
    for r in range(S):
        assert abs(out["lse"][0, r] - math.log(r + 1)) < tol, "Q=0 causal: LSE_r = ln(r+1)"
        vb = v[0, : r + 1].mean(axis=0)
        assert np.allclose(out["o"][0, r], vb, atol=tol)
        wq = np.zeros(d)
        for c in range(r + 1):
            wq += (scale / (r + 1)) * np.dot(do[0, r], v[0, c] - vb) * k[0, c]
        assert np.allclose(out["dq"][0, r], wq, atol=1e-12)
    for c in range(S):
        wv = sum(do[0, r] / (r + 1) for r in range(c, S))
        assert np.allclose(out["dv"][0, c], wv, atol=tol)
    # causal row 0: one visible key -> O_0 = v_0, dQ_0 = 0 exactly.
    q, k, v, do = (_rand(rng, 1, 6, 4) for _ in range(4))
    out = _run(lib, q, k, v, do, scale, True)
    assert np.allclose(out["o"][0, 0], v[0, 0], atol=tol)
    assert np.all(out["dq"][0, 0] == 0.0), "causal row 0: dQ_0 = 0 exactly"
    assert abs(out["lse"][0, 0] - scale * np.dot(q[0, 0], k[0, 0])) < tol


def pin_invariants(lib, tol=1e-10):
    rng = np.random.default_rng(99)
    S, d, scale = 9, 6, 0.41
    for causal in (False, True):
        q, k, v, do = (_rand(rng, 2, S, d) for _ in range(4))
        base = _run(lib, q, k, v, do, scale, causal)
        # sum_c dK_c = 0: every row of dS sums to zero over its visible keys.
        assert np.max(np.abs(base["dk"].sum(axis=1))) < tol, "sum dK = 0"
        # sum_c dV_c = sum_r dO_r: every row of P sums to one.
        assert np.allclose(base["dv"].sum(axis=1), do.sum(axis=1), atol=tol), "sum dV = sum dO"
        # V + 1 c^T: P unchanged, so dQ and dK unchanged; O shifts by c.
        cvec = _rand(rng, 1, 1, d)
        sh = _run(lib, q, k, v + cvec, do, scale, causal)
        assert _relerr(sh["dq"], base["dq"]) < 1e-9, "V shift leaves dQ"
        assert _relerr(sh["dk"], base["dk"]) < 1e-9, "V shift leaves dK"
        assert np.allclose(sh["o"], base["o"] + cvec, atol=tol)
        # K + 1 c^T: scores shift by a per-row constant -> P, O, dQ, dK, dV unchanged.
        sk = _run(lib, q, k + cvec, v, do, scale, causal)
        for n in ("o", "dq", "dk", "dv"):
            assert _relerr(sk[n], base[n]) < 1e-9, f"K shift leaves {n}"
        assert np.allclose(sk["lse"], base["lse"] + scale * np.sum(q * cvec, -1), atol=tol)
        # Linearity in dO.
        s2 = _run(lib, q, k, v, 2.0 * do, scale, causal)
        for n in ("dq", "dk", "dv"):
            assert np.allclose(s2[n], 2.0 * base[n], atol=tol), f"{n} linear in dO"
    # Full mask: permuting keys and values together permutes dK, dV only.
    q, k, v, do = (_rand(rng, 1, S, d) for _ in range(4))
    perm = rng.permutation(S)
    base = _run(lib, q, k, v, do, scale, False)
    pm = _run(lib, q, k[:, perm], v[:, perm], do, scale, False)
    for n in ("o", "lse", "dq"):
        assert _relerr(pm[n], base[n]) < 1e-12, f"key permutation leaves {n}"
    for n in ("dk", "dv"):
        assert _relerr(pm[n], base[n][:, perm]) < 1e-12, f"key permutation permutes {n}"


def pin_autograd(lib, tol=1e-10):
    """An independent gradient engine (torch autograd, float64) on tiny inputs."""
    import torch
    rng = np.random.default_rng(5)
    for causal in (False, True):
        S, d, scale = 6, 5, 0.5
        q, k, v, do = (_rand(rng, 2, S, d) for _ in range(4))
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        s = scale * tq @ tk.transpose(-1, -2)
        if causal:
            s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
        o = torch.softmax(s, dim=-1) @ tv
        (o * torch.tensor(do)).sum().backward()
        out = _run(lib, q, k, v, do, scale, causal)
        assert _relerr(out["o"], o.detach().numpy()) < tol
        assert _relerr(out["lse"], torch.logsumexp(s, -1).detach().numpy()) < tol
        for n, t in (("dq", tq), ("dk", tk), ("dv", tv)):
            assert _relerr(out[n], t.grad.numpy()) < tol, f"autograd {n} causal={causal}"


def _run_tiles(lib, q, k, v, do, scale, causal, tiles):
    return oracle.attn_fwd_bwd(q, k, v, do, scale, causal, tiles=tiles, nthreads=2, lib=lib)


def pin_block_autograd(lib, tol=1e-10):
    """Block masks: torch autograd (float64) with the element mask spelled
    out from an asymmetric tile table (every row keeps a visible key)."""
    import torch
    rng = np.random.default_rng(7)
    S, d, scale = 384, 6, 0.4
    for causal, tiles in ((False, [[0, 1, 0], [1, 0, 1], [1, 1, 0]]),
                          (True, [[1, 0, 0], [1, 1, 0], [0, 1, 1]])):
        t = np.array(tiles, dtype=np.uint8)
        q, k, v, do = (_rand(rng, 1, S, d) for _ in range(4))
        r = np.arange(S)
        vis = t[r[:, None] // 128, r[None, :] // 128].astype(bool)
        if causal:
            vis &= r[None, :] <= r[:, None]
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        sc = (scale * tq @ tk.transpose(-1, -2)).masked_fill(torch.tensor(~vis), float("-inf"))
        o = torch.softmax(sc, dim=-1) @ tv
        (o * torch.tensor(do)).sum().backward()
        out = _run_tiles(lib, q, k, v, do, scale, causal, t)
        assert _relerr(out["o"], o.detach().numpy()) < tol, f"block o causal={causal}"
        assert _relerr(out["lse"], torch.logsumexp(sc, -1).detach().numpy()) < tol
        for n, g in (("dq", tq), ("dk", tk), ("dv", tv)):
            assert _relerr(out[n], g.grad.numpy()) < tol, f"block autograd {n} causal={causal}"


def pin_block_documents(lib, tol=1e-13):
    """A block-diagonal table (documents of whole tiles) is independent
    attention on each document: the same as the unmasked oracle run on each
    document's rows alone."""
    rng = np.random.default_rng(8)
    S, d, scale = 512, 5, 0.6
    docs = ((0, 1), (1, 3), (3, 4))          # tile ranges
    t = np.zeros((4, 4), np.uint8)
    for a, b in docs:
        t[a:b, a:b] = 1
    q, k, v, do = (_rand(rng, 2, S, d) for _ in range(4))
    for causal in (False, True):
        whole = _run_tiles(lib, q, k, v, do, scale, causal, t)
        for a, b in docs:
            sl = slice(128 * a, 128 * b)
            part = _run(lib, q[:, sl], k[:, sl], v[:, sl], do[:, sl], scale, causal)
            for n in ("o", "lse", "dq", "dk", "dv"):
                assert _relerr(whole[n][:, sl], part[n]) < tol, f"document {a}-{b} {n} causal={causal}"


def pin_block_empty_tiles(lib, tol=1e-13):
    """A query tile with every key masked has no softmax (LSE -inf, O, D, dQ
    zero); a key tile nobody sees gets zero dK and dV; the rest is the
    unmasked problem with that tile's rows and keys removed."""
    rng = np.random.default_rng(9)
    S, d, scale = 384, 4, 0.8
    t = np.array([[1, 0, 1], [0, 0, 0], [1, 0, 1]], np.uint8)
    q, k, v, do = (_rand(rng, 1, S, d) for _ in range(4))
    out = _run_tiles(lib, q, k, v, do, scale, False, t)
    mid = slice(128, 256)
    assert np.all(np.isneginf(out["lse"][:, mid]))
    for n in ("o", "D", "dq", "dk", "dv"):
        assert np.all(out[n][:, mid] == 0.0), f"empty tile {n}"
    keep = np.r_[0:128, 256:384]
    rest = _run(lib, q[:, keep], k[:, keep], v[:, keep], do[:, keep], scale, False)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert _relerr(out[n][:, keep], rest[n]) < tol, f"empty tiles: rest {n}"


ALL_PINS = (pin_finite_differences, pin_worked_example, pin_closed_forms,
            pin_invariants, pin_autograd, pin_block_autograd, pin_block_documents,
            pin_block_empty_tiles)
