"""Benchmark: deterministic attention backward TFLOP/s on GB300.

One step = one pass of the whole backward hot path (preprocess, then the main
kernel, which also converts dQ to bf16 in its tail) over the workload B=2, H=16, S=8192, d=128 with the causal mask
(Q and K scaled by 0.5, seed 2) and again with the full mask at the same
shape, each with the fastest of the three deterministic schedules in this
run's per-schedule table (named in `config.schedules`).  FLOPs: 10*B*H*S^2*d for the full
mask, half for causal (exp, preprocess and convert not counted).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `--impl reference` times the float64 CPU oracle on the
host cores on bounded row samples of the same workload.  Under torchrun each
rank runs its own replica (the path does not shard); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "deterministic attn-bwd TFLOP/s (causal+full) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
B, H, S, D = 2, 16, 8192, 128
SEED, QK_SCALE = 2, 0.5
ALL_SCHEDS = ("serial", "descending_q", "shift", "atomic")
DET_SCHEDS = ("serial", "descending_q", "shift")

# DRAM bytes (read + write, MB) of one main-kernel launch at B=1, H=16,
# S=8192, d=128 per (mask, schedule), from ncu captures of that launch,
# keyed by the SHA-1 of the kernel source they were taken on (or of a source
# that differs from it in comments only).  Traffic scales with the number of
# heads, so the B=2 launch moves twice as much.  Reported only while the
# source is unchanged.
TRAFFIC_CAPTURES = {
    "a1187a10e664449de754d08b0cce1bf6b0e2a036": {
        "causal/serial": 461.5 + 401.4, "causal/descending_q": 393.0 + 350.6,
        "causal/shift": 446.8 + 448.6, "causal/atomic": 202.8 + 88.3,
        "full/serial": 399.1 + 363.4, "full/descending_q": 399.2 + 363.6,
        "full/shift": 432.6 + 441.5, "full/atomic": 202.6 + 87.8,
    },
}
MASKS = ("causal", "full")


def flops(mask: str) -> float:
    f = 10.0 * B * H * S * S * D
    return f if mask == "full" else f / 2.0


def workload_name() -> str:
    return f"attn_bwd_b{B}h{H}s{S}d{D}_causal+full"


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "hbm_gbs": float(p["hbm_gbs"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def traffic_for_current_kernel(scheds: dict):
    """Mean DRAM bytes per launch of the timed launches (one per mask)."""
    import hashlib
    path = os.path.join(ROOT, "deterministic_attn_backward_gb300", "csrc", "bwd.cu")
    with open(path, "rb") as f:
        h = hashlib.sha1(f.read()).hexdigest()
    caps = TRAFFIC_CAPTURES.get(h, {})
    per = [caps.get(f"{m}/{scheds[m]}") for m in MASKS]
    if any(x is None for x in per):
        return None
    return round(2 * sum(per) / len(per) * 1e6)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over the process group (identity at N=1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def run_ours(args, rank: int, world: int, local_rank: int) -> dict | None:
    import torch
    import deterministic_attn_backward_gb300 as dab
    from deterministic_attn_backward_gb300 import inputs

    dab.load_library()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream(dev)
    q, k, v, do = inputs.make_qkvdo(B, H, S, D, SEED, QK_SCALE)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    fwd = {m: dab.attn_fwd(qd, kd, vd, m) for m in MASKS}
    ws = {m: dab.new_workspace(B, H, S, D, m, "serial", dev) for m in MASKS}  # largest (ordered)
    outs = {m: tuple(torch.empty_like(qd) for _ in range(3)) for m in MASKS}
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def bwd(mask, sched):
        o, lse = fwd[mask]
        dab.attn_bwd(qd, kd, vd, o, lse, dod, mask, sched, workspace=ws[mask], out=outs[mask])

    step_scheds = {"causal": "shift", "full": "shift"}  # replaced by the fastest below

    def step():
        for m in MASKS:
            bwd(m, step_scheds[m])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    def check():
        for m in MASKS:
            st = dab.check_status(ws[m])
            if st != 0:
                raise RuntimeError(f"device status {st} ({m})")

    step()
    check()

    # ---- per-schedule table: device time per call of the whole hot path;
    # `main_ms`: the main kernel alone (events around its launch; for the
    # ordered schedules it includes the dQ convert in its tail, for atomic
    # the separate convert pass is left out), so that the deterministic and
    # atomic schedules are also compared on like work; `plain_add`: the
    # ordered schedules with DAB_BWD_PLAIN_ADD (load + add + store, no float
    # atomic; same bits as the default red.add.f32)
    def timed_calls(m, sched, flags=0, reps=10):
        o_, lse_ = fwd[m]
        opts_ = dab.BwdOpts(spin_timeout_ns=0, flags=flags, grid=0)
        for _ in range(3):
            dab.attn_bwd(qd, kd, vd, o_, lse_, dod, m, sched, workspace=ws[m], out=outs[m], opts=opts_)
        torch.cuda.synchronize(dev)
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(reps):
            dab.attn_bwd(qd, kd, vd, o_, lse_, dod, m, sched, workspace=ws[m], out=outs[m], opts=opts_)
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    def main_kernel_ms(m, sched, reps=10):
        o_, lse_ = fwd[m]
        flags = dab.DAB_BWD_SKIP_PREPROCESS | (dab.DAB_BWD_SKIP_CONVERT if sched == "atomic" else 0)
        opts_ = dab.BwdOpts(spin_timeout_ns=0, flags=flags, grid=0)
        tot = 0.0
        for it in range(reps + 2):
            dab.bwd_preprocess(o_, lse_, dod, m, sched, ws[m])
            a, b_ = ev(), ev()
            a.record(stream)
            dab.attn_bwd(qd, kd, vd, o_, lse_, dod, m, sched, workspace=ws[m], out=outs[m], opts=opts_)
            b_.record(stream)
            b_.synchronize()
            if it >= 2:
                tot += a.elapsed_time(b_)
        return tot / reps

    per = {}
    for m in MASKS:
        per[m] = {}
        for sched in ALL_SCHEDS:
            ms = timed_calls(m, sched)
            mk = main_kernel_ms(m, sched)
            per[m][sched] = {"ms": round(ms, 4), "tflops": round(flops(m) / ms / 1e9, 2),
                             "main_ms": round(mk, 4), "main_tflops": round(flops(m) / mk / 1e9, 2)}
            if sched != "atomic":
                pm = timed_calls(m, sched, dab.DAB_BWD_PLAIN_ADD)
                per[m][sched]["plain_add"] = {"ms": round(pm, 4),
                                              "tflops": round(flops(m) / pm / 1e9, 2),
                                              "vs_red": round(pm / ms, 4)}
        check()
        # a step runs, per mask, the fastest deterministic schedule
        step_scheds[m] = min(DET_SCHEDS, key=lambda x: per[m][x]["ms"])
        ts, ta = per[m]["serial"]["ms"], per[m]["atomic"]["ms"]
        ms_, ma = per[m]["serial"]["main_ms"], per[m]["atomic"]["main_ms"]
        for sched in ("descending_q", "shift"):
            gap, gap_m = ts - ta, ms_ - ma
            per[m][sched]["gap_closure"] = (round((ts - per[m][sched]["ms"]) / gap, 3)
                                            if abs(gap) > 1e-9 else None)
            per[m][sched]["gap_closure_main"] = (round((ms_ - per[m][sched]["main_ms"]) / gap_m, 3)
                                                 if abs(gap_m) > 1e-9 else None)

    # ---- the dominant kernel alone (events around each main-kernel launch,
    # as the step launches it: with the dQ convert in its tail)
    opts = dab.BwdOpts(spin_timeout_ns=0, flags=dab.DAB_BWD_SKIP_PREPROCESS, grid=0)
    main_ms = {}
    for m in MASKS:
        o, lse = fwd[m]
        sched = step_scheds[m]
        tot, reps = 0.0, 10
        for it in range(reps + 3):
            dab.bwd_preprocess(o, lse, dod, m, sched, ws[m])
            a, b_ = ev(), ev()
            a.record(stream)
            dab.attn_bwd(qd, kd, vd, o, lse, dod, m, sched, workspace=ws[m], out=outs[m], opts=opts)
            b_.record(stream)
            b_.synchronize()
            if it >= 3:
                tot += a.elapsed_time(b_)
        main_ms[m] = tot / reps
    check()

    # ---- side kernels alone (HBM-bound): preprocess, and the separate convert
    # pass (the atomic schedule's; the ordered ones convert in the main
    # kernel's tail) with the main kernel skipped, on the causal workspace
    side = side_kernels(dab, qd, kd, vd, dod, fwd["causal"], "causal", step_scheds["causal"],
                        ws["causal"], outs["causal"], stream, ev)
    # the forward that produces O and LSE (the path's prerequisite, not part
    # of a step): CUDA events around each call, median of 5 after 2 warm-up;
    # algorithmic FLOPs 4*B*H*S^2*d (two products), half for causal
    fwd_t = {}
    for m in MASKS:
        ts = []
        for it in range(7):
            a, b_ = ev(), ev()
            a.record(stream)
            dab.attn_fwd(qd, kd, vd, m)
            b_.record(stream)
            b_.synchronize()
            if it >= 2:
                ts.append(a.elapsed_time(b_))
        ms_f = statistics.median(ts)
        fl = 0.4 * flops(m)
        fwd_t[m] = {"ms": round(ms_f, 4), "tflops": round(fl / ms_f / 1e9, 1)}
    side["forward"] = fwd_t
    own_peak = dab.mma_peak(iters=20000)
    check()

    # ---- the timed region
    for _ in range(args.warmup):
        step()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    e0, e1 = ev(), ev()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    barrier()
    ms_total = e0.elapsed_time(e1)
    clocks = sampler.stop() if sampler else None
    check()
    ms_total = max_over_ranks(ms_total, world, dev)

    # ---- end to end: host buffers through the public API (dab_attn_bwd_host:
    # the copies in and out overlap the computation inside the library), the
    # copies in the timed region
    host_in = {m: tuple(t.cpu().pin_memory() for t in (q, k, v, fwd[m][0], fwd[m][1], do))
               for m in MASKS}
    host_out = {m: tuple(torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
                         for _ in range(3)) for m in MASKS}
    host_ws = {m: dab.new_host_workspace(B, H, S, D, m, step_scheds[m], 0, dev) for m in MASKS}
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for m in MASKS:
            dab.attn_bwd(*host_in[m], mask=m, sched=step_scheds[m], workspace=host_ws[m],
                         out=host_out[m])

    for _ in range(2):
        e2e_step()
    barrier()
    c0, c1 = ev(), ev()
    c0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    c1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(c0.elapsed_time(c1), world, dev) / e2e_steps
    check()
    for m in MASKS:
        st = dab.check_status(host_ws[m])
        if st != 0:
            raise RuntimeError(f"device status {st} (host path, {m})")
    h2d = sum(t.numel() * t.element_size() for m in MASKS for t in host_in[m])
    d2h = sum(t.numel() * t.element_size() for m in MASKS for t in host_out[m])

    if rank != 0:
        return None
    peaks = load_peaks()
    step_flops = flops("causal") + flops("full")
    ms_step = ms_total / args.steps
    value = world * step_flops / (ms_step * 1e9)
    main_avg = (main_ms["causal"] + main_ms["full"]) / 2.0
    achieved = step_flops / 2.0 / main_avg / 1e9   # algorithmic FLOPs per launch / launch time
    peak = peaks["bf16_tflops"]
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": workload_name(), "B": B, "H": H, "S": S, "d": D,
                   "masks": list(MASKS), "schedules": step_scheds, "seed": SEED,
                   "qk_scale": QK_SCALE,
                   "l2": "inputs exceed L2 (5 x 64 MiB read per call), no flush",
                   "parallelism": f"replicas x{world}"},
        "frac_of_peak": round(value / world / peak, 4),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic_for_current_kernel(step_scheds),
                     "kernel": "bwd_kernel<128>", "peak_source": peaks["source"] + " (burst)",
                     "launch_ms": {m: round(x, 4) for m, x in main_ms.items()}},
        "own_tensor_peak": {"tflops": round(own_peak["tflops"], 1),
                            "frac": round(achieved / own_peak["tflops"], 4),
                            "how": "dab_mma_peak: one CTA per SM, back-to-back tcgen05.mma "
                                   "128x256x16 from shared memory"},
        "side_kernels": side,
        "per_schedule": per,
        "auto_schedules": {m: dab.sched_select(m, B, H, S,
                                               torch.cuda.get_device_properties(dev).multi_processor_count)
                           for m in MASKS},
        "e2e": {"value": round(world * step_flops / (e2e_ms * 1e9), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        # per mask: preprocess + main kernel (+ the convert pass for atomic)
        "gpu_launches": sum(2 + (step_scheds[m] == "atomic") for m in MASKS) * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu_baseline(),
    }


def side_kernels(dab, qd, kd, vd, dod, fwd_m, mask, sched, ws, out, stream, ev, reps=10) -> dict:
    """Preprocess and convert timed alone (CUDA events, median of `reps`), with
    their algorithmic bytes: preprocess reads O, dO, LSE and writes D and
    LSE*log2(e); convert reads one f32 accumulator and writes bf16 dQ (the
    minimum), and `actual_bytes` counts the accumulation buffers it really
    reads (four for the ordered schedules)."""
    o, lse = fwd_m
    Bq, Hq, Sq, Dq = qd.shape
    rows, elems = Bq * Hq * Sq, Bq * Hq * Sq * Dq
    peaks = load_peaks()

    def timed(fn):
        ts = []
        for it in range(reps + 3):
            a, b_ = ev(), ev()
            a.record(stream)
            fn()
            b_.record(stream)
            b_.synchronize()
            if it >= 3:
                ts.append(a.elapsed_time(b_))
        return statistics.median(ts)

    pre_ms = timed(lambda: dab.bwd_preprocess(o, lse, dod, mask, sched, ws))
    conv_opts = dab.BwdOpts(spin_timeout_ns=0,
                            flags=dab.DAB_BWD_SKIP_PREPROCESS | dab.DAB_BWD_SKIP_MAIN, grid=0)
    conv_ms = timed(lambda: dab.attn_bwd(qd, kd, vd, o, lse, dod, mask, sched, workspace=ws,
                                         out=out, opts=conv_opts))
    ways = 1 if sched == "atomic" else 4
    pre_b = 4 * elems + 12 * rows
    conv_b, conv_actual = 6 * elems, (4 * ways + 2) * elems
    gbs = lambda b, ms: round(b / (ms * 1e-3) / 1e9, 1)
    hbm = peaks["hbm_gbs"]
    return {"preprocess": {"ms": round(pre_ms, 4), "bytes": pre_b, "gbs": gbs(pre_b, pre_ms),
                           "frac": round(pre_b / (pre_ms * 1e-3) / 1e9 / hbm, 3)},
            "convert": {"ms": round(conv_ms, 4), "bytes": conv_b, "gbs": gbs(conv_b, conv_ms),
                        "actual_bytes": conv_actual, "actual_gbs": gbs(conv_actual, conv_ms),
                        "frac_actual": round(conv_actual / (conv_ms * 1e-3) / 1e9 / hbm, 3)},
            "peak_gbs": hbm, "peak_source": peaks["source"]}


# Measurement configurations: (name, B, H, S, d, seed, qk scale, masks).
SWEEP_CONFIGS = [
    ("C1", 4, 16, 2048, 64, 1, 1.0, ("full",)),
    ("C2", 2, 16, 8192, 128, 2, 0.5, ("causal", "full")),
    ("C3", 1, 32, 16384, 128, 3, 1.0, ("full", "causal")),
] + [(f"C4-s{s_}-d{d_}", 32768 // s_, 16, s_, d_, 4, 1.0, ("full", "causal"))
     for d_ in (64, 128) for s_ in (1024, 2048, 4096, 8192, 16384, 32768)]


# Block-mask configurations (tile flags over 128 x 128 tiles): a sliding
# window of `w` tiles before the query (causal), and documents of `w` tiles
# (block diagonal, causal inside a document).  FLOPs count the visible tiles
# (10 * 128^2 * d each; a causal diagonal tile counts half).
BLOCK_CONFIGS = [
    ("BM-window-1k", 2, 16, 8192, 128, 2, 0.5, "window", 8),
    ("BM-docs-2k", 2, 16, 8192, 128, 2, 0.5, "docs", 16),
    ("BM-docs-8k", 1, 16, 32768, 128, 4, 1.0, "docs", 64),
]


def block_tiles(kind: str, N: int, w: int):
    import numpy as np
    j, i = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")   # j: query tile, i: key tile
    if kind == "window":
        return ((i <= j) & (j - i < w)).astype(np.uint8)
    return (j // w == i // w).astype(np.uint8)


def run_block_sweep(reps: int) -> None:
    """Block masks: every schedule that supports them, one JSON line per config."""
    import numpy as np
    import torch
    import deterministic_attn_backward_gb300 as dab
    from deterministic_attn_backward_gb300 import inputs
    dab.load_library()
    peak = load_peaks()["bf16_tflops"]
    stream = torch.cuda.current_stream()
    for name, b, h, s_, d, seed, qks, kind, w in BLOCK_CONFIGS:
        N = s_ // 128
        t = block_tiles(kind, N, w)
        jj, ii = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")
        vis = (t.astype(bool) & (ii <= jj)).astype(np.float64)           # the causal mask applies too
        vis[np.arange(N), np.arange(N)] *= 0.5                            # causal diagonal tiles
        fl = float(vis.sum()) * 10.0 * 128 * 128 * d * b * h
        q, k, v, do = (x.cuda() for x in inputs.make_qkvdo(b, h, s_, d, seed, qks))
        o, lse = dab.attn_fwd(q, k, v, "causal", tiles=t)
        ws = dab.new_workspace(b, h, s_, d, sched="serial", block=True)
        out = tuple(torch.empty_like(q) for _ in range(3))
        row = {"config": name, "B": b, "H": h, "S": s_, "d": d, "mask": f"causal+{kind}{w}",
               "visible_tiles": float(vis.sum()), "scheds": {}}
        for sched in ("serial", "descending_q", "atomic"):
            ts = []
            for it in range(3 + reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dab.attn_bwd(q, k, v, o, lse, do, "causal", sched, workspace=ws, out=out, tiles=t)
                e1.record(stream)
                e1.synchronize()
                if it >= 3:
                    ts.append(e0.elapsed_time(e1))
            ms = statistics.median(ts)
            tf = fl / (ms * 1e-3) / 1e12
            row["scheds"][sched] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                    "frac": round(tf / peak, 4), "status": dab.check_status(ws)}
        print(json.dumps(row), flush=True)
        del q, k, v, do, ws, out
        torch.cuda.empty_cache()


def run_sweep(which: str, reps: int) -> None:
    """Every schedule on every measurement configuration: per (config, mask)
    one JSON line with ms, TFLOP/s, fraction of the measured peak and the gap
    closure (T_serial - T_sched) / (T_serial - T_atomic); medians of `reps`
    timed calls after three warm-up calls."""
    import torch
    import deterministic_attn_backward_gb300 as dab
    from deterministic_attn_backward_gb300 import inputs
    dab.load_library()
    peak = load_peaks()["bf16_tflops"]
    stream = torch.cuda.current_stream()
    for name, b, h, s_, d, seed, qks, masks in SWEEP_CONFIGS:
        if which != "all" and not name.startswith(which):
            continue
        q, k, v, do = (t.cuda() for t in inputs.make_qkvdo(b, h, s_, d, seed, qks))
        ws = dab.new_workspace(b, h, s_, d, "full", "serial")
        out = tuple(torch.empty_like(q) for _ in range(3))
        for mask in masks:
            o, lse = dab.attn_fwd(q, k, v, mask)
            fl = 10.0 * b * h * s_ * s_ * d * (1.0 if mask == "full" else 0.5)
            row = {"config": name, "B": b, "H": h, "S": s_, "d": d, "mask": mask, "scheds": {}}
            for sched in ALL_SCHEDS:
                ts = []
                for it in range(3 + reps):
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws, out=out)
                    e1.record(stream)
                    e1.synchronize()
                    if it >= 3:
                        ts.append(e0.elapsed_time(e1))
                st = dab.check_status(ws)
                ms = statistics.median(ts)
                tf = fl / (ms * 1e-3) / 1e12
                row["scheds"][sched] = {"ms": round(ms, 4), "tflops": round(tf, 1),
                                        "frac": round(tf / peak, 4), "status": st}
            sc = row["scheds"]
            gap = sc["serial"]["ms"] - sc["atomic"]["ms"]
            for sched in ("descending_q", "shift"):
                sc[sched]["gap_closure"] = (round((sc["serial"]["ms"] - sc[sched]["ms"]) / gap, 3)
                                            if abs(gap) > 1e-9 else None)
            print(json.dumps(row), flush=True)
        del q, k, v, do, ws, out
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- oracle
def _oracle_head_time(q, k, v, do, b, h, mask, lib, threads):
    import oracle
    args = [t[b, h].unsqueeze(0) for t in (q, k, v, do)]
    t0 = time.perf_counter()
    out = oracle.attn_fwd_bwd(*args, 1.0 / D ** 0.5, mask == "causal", nthreads=threads, lib=lib)
    return time.perf_counter() - t0, out


def cpu_baseline() -> dict:
    """The oracle on two whole heads of the workload (one per mask)."""
    import oracle
    from deterministic_attn_backward_gb300 import inputs
    q, k, v, do = inputs.make_qkvdo(B, H, S, D, SEED, QK_SCALE)
    lib, threads = oracle.load(), oracle.default_threads()
    secs = fl = 0.0
    for (b, h), m in (((0, 0), "causal"), ((B - 1, H - 1), "full")):
        dt, _ = _oracle_head_time(q, k, v, do, b, h, m, lib, threads)
        secs += dt
        fl += flops(m) / (B * H)
    return {"value": round(fl / secs / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"2 whole heads of the workload (head (0,0) causal, head ({B-1},{H-1}) full),"
                      f" float64 forward+backward, {secs:.1f} s"}


def run_reference(args, rank: int) -> dict | None:
    """The oracle as it stands, on bounded row samples of the workload.

    Set-up (untimed): one whole head per mask through the oracle, for the
    LSE_r and D_r every key row needs.  Each step then recomputes, for that
    head, ROWS query rows (O, LSE, D, dQ) and ROWS key rows (dK, dV) per mask,
    rotating the rows from step to step; one query row plus one key row is
    1/S of the head's backward FLOPs.
    """
    if rank != 0:
        return None
    import oracle
    from deterministic_attn_backward_gb300 import inputs
    rows_per_step = 64
    q, k, v, do = inputs.make_qkvdo(B, H, S, D, SEED, QK_SCALE)
    lib, threads = oracle.load(), oracle.default_threads()
    prep = {}
    for (b, h), m in (((0, 0), "causal"), ((B - 1, H - 1), "full")):
        _, whole = _oracle_head_time(q, k, v, do, b, h, m, lib, threads)
        prep[m] = ([t[b, h] for t in (q, k, v, do)], whole["lse"][0], whole["D"][0])
    secs = fl = 0.0
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        f = 0.0
        for m in MASKS:
            args_h, lse_all, D_all = prep[m]
            rows = [((i * rows_per_step + x) * 97) % S for x in range(rows_per_step)]
            oracle.attn_rows(*args_h, 1.0 / D ** 0.5, m == "causal", rows, rows,
                             lse_all=lse_all, D_all=D_all, nthreads=threads, lib=lib)
            f += flops(m) / (B * H) * (2 * rows_per_step) / (2 * S)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            secs += dt
            fl += f
    value = fl / secs / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / max(1, args.steps) * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(), "B": B, "H": H, "S": S, "d": D,
                   "masks": list(MASKS), "seed": SEED, "qk_scale": QK_SCALE},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"per step and mask: {rows_per_step} query rows (O, LSE, D, dQ)"
                                   f" and {rows_per_step} key rows (dK, dV) of one head, float64;"
                                   " the head's LSE and D computed once, untimed"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_case(spec: str, reps: int) -> dict:
    """One configuration "B,H,S,d,mask,sched": `reps` backward calls after
    three warm-up calls, each timed with CUDA events (used to drive profilers
    and size sweeps; prints per-call milliseconds and TFLOP/s)."""
    import torch
    import deterministic_attn_backward_gb300 as dab
    from deterministic_attn_backward_gb300 import inputs
    b, h, s_, d = (int(x) for x in spec.split(",")[:4])
    mask, sched = spec.split(",")[4:6]
    q, k, v, do = (t.cuda() for t in inputs.make_qkvdo(b, h, s_, d, 7, 0.5))
    o, lse = dab.attn_fwd(q, k, v, mask)
    ws = dab.new_workspace(b, h, s_, d, mask, sched)
    out = tuple(torch.empty_like(q) for _ in range(3))
    ms = []
    for i in range(3 + reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dab.attn_bwd(q, k, v, o, lse, do, mask, sched, workspace=ws, out=out)
        e1.record()
        e1.synchronize()
        if i >= 3:
            ms.append(e0.elapsed_time(e1))
    st = dab.check_status(ws)
    f = 10.0 * b * h * s_ * s_ * d * (1.0 if mask == "full" else 0.5)
    med = statistics.median(ms)
    return {"case": spec, "status": st, "ms": [round(x, 4) for x in ms],
            "tflops": round(f / med / 1e9, 2)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--case", default=None, help="B,H,S,d,mask,sched: time one configuration")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--sweep", default=None,
                    help="all | C1 | C2 | C3 | C4 | block: every schedule on the measurement "
                         "configurations (block: the block-mask ones)")
    args = ap.parse_args()
    if args.sweep:
        if args.sweep in ("all", "block"):
            if args.sweep == "all":
                run_sweep("all", max(args.reps, 5))
            run_block_sweep(max(args.reps, 5))
        else:
            run_sweep(args.sweep, max(args.reps, 5))
        return
    if args.case:
        for spec in args.case.split(";"):
            print(json.dumps(run_case(spec, args.reps)), flush=True)
        return
    args.warmup = max(3, args.warmup)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
