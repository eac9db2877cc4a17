#!/usr/bin/env python
"""Benchmark of the mHC layer on GB300: one step = mhc_pre -> mhc_post ->
mhc_post_bwd -> mhc_pre_bwd over one batch (the whole hot path), on synthetic
inputs resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 5] [--iters 20]

Prints ONE JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
batch of T tokens (weak scaling) and the parameter gradients dphi, db, dalpha
are summed over ranks with one NCCL all-reduce per step, the layer's only
exchange.  ``--impl reference`` times the float64 CPU oracle (the reference
arm) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import collections
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mHC fused fwd(+bwd) tokens/s and HBM GB/s vs GB300 peak at n=4, D=5120"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
STEP_OPS = ("mhc_pre", "mhc_post", "mhc_post_bwd", "mhc_pre_bwd")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", type=int, default=5)
    p.add_argument("--iters", type=int, default=20)
    p.add_argument("--tokens", type=int, default=None,
                   help="override the workload's T (smaller cases for profiling)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cross-layer", action="store_true",
                   help="skip the side measurements (mhc_post_pre, mhc_post_norm, "
                        "the recompute backward)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def algorithmic_bytes(w):
    """Bytes each op must move per launch (activations once, gates, saved
    state; phi and the parameter gradients once per launch)."""
    a = 2 if w.dtype == "bf16" else 4
    K, D, T, G = w.K, w.D, w.T, w.G
    gates_pre = 4 * (w.n + w.n + w.n * w.n + G + 1)      # H_pre, H_post, H_res, proj, inv_rms
    per_tok = {
        "mhc_pre": a * K + a * D + gates_pre,
        "mhc_post": a * K + a * D + 4 * (w.n + w.n * w.n) + a * K,
        "mhc_post_bwd": 3 * a * K + 2 * a * D + 2 * 4 * (w.n + w.n * w.n),
        "mhc_pre_bwd": a * D + 3 * a * K + 4 * (G + 1 + w.n + w.n * w.n),
    }
    per_launch = {"mhc_pre": 4 * K * G, "mhc_post": 0, "mhc_post_bwd": 0,
                  "mhc_pre_bwd": 2 * 4 * K * G}
    return {op: per_tok[op] * T + per_launch[op] for op in STEP_OPS}, per_tok


def cross_layer_bytes(w):
    """Bytes mhc_post_pre must move per launch: x, y and layer l's gates in,
    x_next, x_in, layer l + 1's gates and saved state out, phi once."""
    a = 2 if w.dtype == "bf16" else 4
    per_tok = (a * w.K + a * w.D + 4 * (w.n + w.n * w.n) + a * w.K + a * w.D
               + 4 * (w.n + w.n + w.n * w.n + w.G + 1))
    return per_tok * w.T + 4 * w.K * w.G, per_tok


def run_cross_layer(w, inp, dev, reps=20):
    """mhc_post_pre (layer l's residual update fused with layer l + 1's pre
    step) against mhc_post then mhc_pre, CUDA events on the stream, inputs
    larger than L2.  A side measurement: not part of the timed step."""
    import torch
    from mhc_pre_gb300 import binding as B
    from mhc_pre_gb300 import workloads as W
    g = W.make_layer_gates(w, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fused():
        B.mhc_post_pre(inp["x"], inp["y"], g["H_post_l"], g["H_res_l"], inp["phi"], inp["b"],
                       inp["alpha"], w.iters, w.eps)

    def separate():
        xn = B.mhc_post(inp["x"], inp["y"], g["H_post_l"], g["H_res_l"])
        B.mhc_pre(xn, inp["phi"], inp["b"], inp["alpha"], w.iters, w.eps)

    out = {}
    for name, f in (("fused", fused), ("separate", separate)):
        for _ in range(3):
            f()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            f()
        e.record(stream)
        torch.cuda.synchronize()
        out[name] = s.elapsed_time(e) / reps
    assert B.get_last_device_error() == B.MHC_OK
    nb, per_tok = cross_layer_bytes(w)
    peak, kind = peaks()
    return {"op": "mhc_post_pre", "fused_ms": out["fused"], "separate_ms": out["separate"],
            "GBps": nb / out["fused"] / 1e6, "frac_of_" + kind: nb / out["fused"] / 1e6 / peak,
            "algorithmic_bytes_per_token": per_tok,
            "launches": B.kernel_launches("mhc_post_pre", w.dtype, w.T, w.n, w.D)}


def run_post_norm(w, inp, dev, reps=10):
    """mhc_post_norm / mhc_post_norm_bwd with both stability steps (sandwich
    and block normalisation) on the step's inputs: a side measurement, not
    part of the timed step.  Bytes: x, y, gates in and x_next out (forward);
    g_next, x, y, gates in and dx, dy, dH out (backward); saved r_y, s."""
    import torch
    from mhc_pre_gb300 import binding as B
    from mhc_pre_gb300 import workloads as W
    g = W.make_layer_gates(w, device=dev)
    stream = torch.cuda.current_stream(dev)
    flags = B.SANDWICH_NORM | B.BLOCK_NORM
    f = B.mhc_post_norm(inp["x"], inp["y"], g["H_post_l"], g["H_res_l"], flags, w.eps)

    def timed(fn):
        for _ in range(3):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    fwd = timed(lambda: B.mhc_post_norm(inp["x"], inp["y"], g["H_post_l"], g["H_res_l"], flags, w.eps))
    bwd = timed(lambda: B.mhc_post_norm_bwd(inp["g_next"], inp["x"], inp["y"], g["H_post_l"], g["H_res_l"],
                                            flags, f.inv_rms_y, f.inv_rms_out, w.eps))
    assert B.get_last_device_error() == B.MHC_OK
    a = 2 if w.dtype == "bf16" else 4
    gates = 4 * (w.n + w.n * w.n)
    fb = w.T * (2 * a * w.K + a * w.D + gates + 8)
    bb = w.T * (3 * a * w.K + 2 * a * w.D + 2 * gates + 8)
    peak, kind = peaks()
    return {"op": "mhc_post_norm (sandwich + block)", "fwd_ms": fwd, "bwd_ms": bwd,
            "fwd_GBps": fb / fwd / 1e6, "bwd_GBps": bb / bwd / 1e6,
            "fwd_frac_of_" + kind: fb / fwd / 1e6 / peak, "bwd_frac_of_" + kind: bb / bwd / 1e6 / peak}


def run_recompute(w, inp, dev, reps=10):
    """The recompute-oriented backward on the step's inputs: mhc_pre_gates
    (the gates and saved state from x alone) and mhc_layer_bwd_recompute
    against mhc_post_bwd + mhc_pre_bwd on saved state.  A side measurement,
    not part of the timed step."""
    import torch
    from mhc_pre_gb300 import binding as B
    stream = torch.cuda.current_stream(dev)
    x, y, phi, b, alpha = (inp[k] for k in ("x", "y", "phi", "b", "alpha"))
    f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    ws = torch.empty((B.layer_bwd_recompute_workspace_bytes(x.dtype, w.T, w.n, w.D),),
                     dtype=torch.uint8, device=dev)
    ws_bwd = torch.empty((B.pre_bwd_workspace_bytes(x.dtype, w.T, w.n, w.D),), dtype=torch.uint8, device=dev)

    def saved():
        pb = B.mhc_post_bwd(inp["g_next"], x, y, f.H_post, f.H_res)
        B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj, f.inv_rms, pb.dx,
                      w.iters, workspace=ws_bwd)

    def timed(fn):
        for _ in range(3):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    gates = timed(lambda: B.mhc_pre_gates(x, phi, b, alpha, w.iters, w.eps))
    rec = timed(lambda: B.mhc_layer_bwd_recompute(inp["g_in"], inp["g_next"], x, y, phi, b, alpha,
                                                  w.iters, w.eps, workspace=ws))
    sav = timed(saved)
    assert B.get_last_device_error() == B.MHC_OK
    a = 2 if w.dtype == "bf16" else 4
    saved_state = 4 * (w.G + 1)                                   # proj, inv_rms
    gb = w.T * (a * w.K + 4 * (w.n + w.n + w.n * w.n) + saved_state) + 4 * w.K * w.G
    peak, kind = peaks()
    return {"op": "mhc_pre_gates, mhc_layer_bwd_recompute", "gates_ms": gates,
            "gates_GBps": gb / gates / 1e6, "gates_frac_of_" + kind: gb / gates / 1e6 / peak,
            "bwd_recompute_ms": rec, "bwd_saved_state_ms": sav,
            "saved_state_bytes_per_token": {"saved": saved_state, "recompute": 0},
            "launches": B.kernel_launches("mhc_layer_bwd_recompute", w.dtype, w.T, w.n, w.D)}


class ClockSampler:
    """nvidia-smi sampler for the clocks and throttle reasons of one GPU."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for r in csv.reader(io.StringIO(out)):
            if len(r) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + r[0].strip().split(".")[1]) if "." in r[0] else 0.0
                rows.append((ts + frac, float(r[1]), float(r[2]), r[5].strip(), r[6].strip(),
                             r[7].strip(), r[8].strip()))
            except (ValueError, IndexError):
                continue
        inside = [x for x in rows if t0 - 0.15 <= x[0] <= t1 + 0.15]
        if len(inside) < 3:       # short timed region: nearest samples around it
            rows.sort(key=lambda x: abs(x[0] - 0.5 * (t0 + t1)))
            inside = rows[:5]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for x in inside:
            for name, v in zip(names, x[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def oracle_rate(w, seconds: float, chunk: int = 256):
    """Tokens/s of the float64 oracle (fwd + bwd of the whole layer) on
    chunks of the workload, repeated for about ``seconds``."""
    from mhc_pre_gb300 import workloads as W
    from tests import parity as P
    sample = W.make_inputs(w.with_(T=chunk, backward=True), device="cpu")
    inp = {k: P.f64(v) for k, v in sample.items()}
    done, t0 = 0, time.perf_counter()
    while True:
        P.run_oracle(inp, w.iters, w.eps, True)
        done += chunk
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return done / el, done, el


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from mhc_pre_gb300 import workloads as W
    from tests import parity as P
    w = W.WORKLOADS[args.workload].with_(iters=args.iters, backward=True)
    # calibrate: size each step so that warmup + steps take about 2 minutes
    rate, _, _ = oracle_rate(w, 1.0, chunk=4)
    per_step = 120.0 / max(1, args.steps + args.warmup)
    S = int(max(1, min(256, rate * per_step)))
    sample = W.make_inputs(w.with_(T=S), device="cpu")
    inp = {k: P.f64(v) for k, v in sample.items()}
    for _ in range(args.warmup):
        P.run_oracle(inp, w.iters, w.eps, True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        P.run_oracle(inp, w.iters, w.eps, True)
    el = time.perf_counter() - t0
    value = S * args.steps / el
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),      # the same workload as the CUDA arm ...
        "sample_tokens_per_step": S,        # ... of which each step times a bounded sample
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"float64 NumPy oracle, fwd+bwd of the whole layer on {S} "
                                   f"tokens per step of the {w.name} workload"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, tokens=None):
    return {"workload": f"mhc layer fwd+bwd: {w.name}", "T": w.T if tokens is None else tokens,
            "n": w.n, "D": w.D, "iters": w.iters, "alpha": w.alpha, "b_std": w.b_std,
            "step": "mhc_pre+mhc_post+mhc_post_bwd+mhc_pre_bwd",
            "l2": "inputs larger than L2 (no flush)"}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from mhc_pre_gb300 import binding as B
    from mhc_pre_gb300 import build as mbuild
    from mhc_pre_gb300 import workloads as W
    from mhc_pre_gb300.dp import allreduce_param_grads

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    mbuild.build()

    w = W.WORKLOADS[args.workload].with_(iters=args.iters, backward=True)
    if args.tokens is not None and args.tokens != w.T:
        # a smaller case of the same shape, for profiling; the name says so
        w = w.with_(T=args.tokens, name=f"{w.name}, T overridden to {args.tokens}")
    inp = W.make_inputs(w, device=dev, seed=1000 + w.wid + 7919 * rank)
    ws = torch.empty((max(B.pre_bwd_workspace_bytes(torch.bfloat16, w.T, w.n, w.D), 16),),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STEP_OPS) + 1)]
          for _ in range(args.steps)]

    def step(i=None, src=None):
        e = ev[i] if i is not None else None
        a = inp if src is None else src
        if e: e[0].record(stream)
        f = B.mhc_pre(a["x"], a["phi"], a["b"], a["alpha"], w.iters, w.eps)
        if e: e[1].record(stream)
        xn = B.mhc_post(a["x"], a["y"], f.H_post, f.H_res)
        if e: e[2].record(stream)
        pb = B.mhc_post_bwd(a["g_next"], a["x"], a["y"], f.H_post, f.H_res)
        if e: e[3].record(stream)
        qb = B.mhc_pre_bwd(a["g_in"], pb.dH_post, pb.dH_res, a["x"], a["phi"], a["b"],
                           a["alpha"], f.proj, f.inv_rms, pb.dx, w.iters, workspace=ws)
        if e: e[4].record(stream)
        if world > 1:
            allreduce_param_grads(qb.dphi, qb.db, qb.dalpha)
        return {"x_in": f.x_in, "x_next": xn, "dx": qb.dx, "dy": pb.dy,
                "dphi": qb.dphi, "db": qb.db, "dalpha": qb.dalpha}

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if B.get_last_device_error() != B.MHC_OK:
        raise RuntimeError("device error during warm-up")

    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    if world > 1:
        t = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    clocks = sampler.stop(w0, w1) if sampler else None
    assert B.get_last_device_error() == B.MHC_OK

    per_op_ms = {op: statistics.fmean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                 for j, op in enumerate(STEP_OPS)}
    nbytes, per_tok = algorithmic_bytes(w)
    peak, peak_kind = peaks()
    kernels = {op: {"ms": per_op_ms[op], "GBps": nbytes[op] / per_op_ms[op] / 1e6,
                    "frac_of_" + peak_kind: nbytes[op] / per_op_ms[op] / 1e6 / peak,
                    "frac_of_8TBps_nominal": nbytes[op] / per_op_ms[op] / 1e6 / NOMINAL_HBM_GBS,
                    "bytes": nbytes[op]}
               for op in STEP_OPS}
    dom = max(STEP_OPS, key=lambda op: per_op_ms[op])
    achieved = nbytes[dom] / per_op_ms[dom] / 1e6
    traffic = ncu_traffic(dom, w)

    # ---- end to end: pinned host inputs in, parameter gradients out ----------
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, inp, step, stream, dev, world)

    # ---- side measurement: the cross-layer step (rank 0, N = 1) --------------
    cross = post_norm = recompute = decode = sweep = None
    if rank == 0 and world == 1 and not args.no_cross_layer:
        cross = run_cross_layer(w, inp, dev)
        post_norm = run_post_norm(w, inp, dev)
        recompute = run_recompute(w, inp, dev)
        decode = run_decode(w, dev)
        sweep = run_sweep(w, inp, dev)

    # ---- float64 oracle on the host cores (rank 0, N = 1) --------------------
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        rate, done, el = oracle_rate(w, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle",
               "sample": f"float64 NumPy oracle, fwd+bwd of the whole layer, {done} tokens "
                         f"(256-token chunks, D={w.D}) in {el:.1f} s"}

    launches_per_step = launches(w)
    value = world * w.T * args.steps / (elapsed_ms / 1e3)
    step_bytes = sum(nbytes.values())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "config": workload_config(w),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic,
                     "algorithmic_bytes_per_token": per_tok[dom], "tokens_per_launch": w.T},
        "step_hbm": {"GBps": step_bytes / (elapsed_ms / args.steps) / 1e6,
                     "frac_of_" + peak_kind: step_bytes / (elapsed_ms / args.steps) / 1e6 / peak,
                     "frac_of_8TBps_nominal": step_bytes / (elapsed_ms / args.steps) / 1e6 / NOMINAL_HBM_GBS},
        "roofline_forward": {"bound": "hbm", "kernel": "mhc_pre",
                             "achieved": nbytes["mhc_pre"] / per_op_ms["mhc_pre"] / 1e6,
                             "peak": NOMINAL_HBM_GBS, "peak_kind": "nominal 8 TB/s",
                             "unit": "GB/s",
                             "frac": nbytes["mhc_pre"] / per_op_ms["mhc_pre"] / 1e6 / NOMINAL_HBM_GBS,
                             "frac_of_" + peak_kind: nbytes["mhc_pre"] / per_op_ms["mhc_pre"] / 1e6 / peak,
                             "target_frac": 0.70,
                             "target_met": nbytes["mhc_pre"] / per_op_ms["mhc_pre"] / 1e6 >= 0.70 * NOMINAL_HBM_GBS},
        "kernels": kernels,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "cross_layer": cross,
        "post_norm": post_norm,
        "recompute": recompute,
        "decode": decode,
        "sinkhorn_sweep": sweep,
        "memory": memory_accounting(w),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def launches(w):
    """Kernels of this library launched per step (mhc_kernel_launches of each op)."""
    from mhc_pre_gb300 import binding as B
    return sum(B.kernel_launches(op, w.dtype, w.T, w.n, w.D) for op in STEP_OPS)


def kernel_sources_sha256():
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "mhc_pre_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))
                   + glob.glob(os.path.join(csrc, "*.h")))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(op, w):
    """DRAM bytes per launch of ``op`` from the committed ncu summary (per
    token, scaled to this workload); None when the summary was taken on
    other kernel sources or another width."""
    import re
    path = os.path.join(ROOT, "profiles", "step_T32768_D5120_launches_dram.md")
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    m = re.search(r"sources_sha256: ([0-9a-f]{64})", text)
    if m is None or m.group(1) != kernel_sources_sha256() or w.D != 5120 or w.n != 4:
        return None
    m = re.search(r"traffic_per_token %s (\d+)" % re.escape(op), text)
    return int(m.group(1)) * w.T if m else None


def run_e2e(args, w, inp, step, stream, dev, world):
    """The step through the public API with the host in the loop, as a round
    trip: every step's inputs are copied from pinned host memory, and every
    result (x_in, x_next, dx, dy and the parameter gradients) copied back to
    pinned host memory, all inside the timed region.  The inputs of step
    i + 1 are copied on a second stream into a second set of device buffers
    while step i computes; the results of step i are copied back on a third
    stream while step i + 1 computes (the copies, bound by the host link,
    dominate).  The host keeps at most three steps in flight, as a training
    loop that reads each step's results does: it waits for the results of
    step i - 3 to reach the host before it issues step i.  Unbounded, it
    queues the whole run at once, and every queued step's outputs stay
    allocated until their copy back ends, which fills the device and makes
    the allocator free and re-allocate in the middle of the run."""
    import torch
    host = {k: v.to("cpu").pin_memory() for k, v in inp.items()}
    keys = ("x", "y", "g_in", "g_next", "phi", "b", "alpha")
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    act = inp["x"].dtype
    out_h = {"x_in": torch.empty((w.T, w.D), dtype=act, pin_memory=True),
             "x_next": torch.empty((w.T, w.n, w.D), dtype=act, pin_memory=True),
             "dx": torch.empty((w.T, w.n, w.D), dtype=act, pin_memory=True),
             "dy": torch.empty((w.T, w.D), dtype=act, pin_memory=True),
             "dphi": torch.empty((w.K, w.G), pin_memory=True),
             "db": torch.empty((w.G,), pin_memory=True),
             "dalpha": torch.empty((3,), pin_memory=True)}
    d2h = sum(v.numel() * v.element_size() for v in out_h.values())
    bufs = [{k: inp[k] for k in keys}, {k: torch.empty_like(inp[k]) for k in keys}]
    copy_stream, back_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    consumed = [torch.cuda.Event(), torch.cuda.Event()]
    computed = torch.cuda.Event()
    in_flight = collections.deque()                     # results not yet on the host
    DEPTH = 3

    def copy_in(bi):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[bi])        # the step that last read these buffers is done
            for k in keys:
                bufs[bi][k].copy_(host[k], non_blocking=True)
            copied[bi].record(copy_stream)

    def copy_out(res):
        computed.record(stream)
        back_stream.wait_event(computed)
        with torch.cuda.stream(back_stream):
            for k, t in res.items():
                out_h[k].copy_(t, non_blocking=True)
                t.record_stream(back_stream)            # not reused before the copy is done
        done = torch.cuda.Event()
        done.record(back_stream)
        in_flight.append(done)

    def run(n):
        for ev in consumed:
            ev.record(stream)
        copy_in(0)
        for i in range(n):
            bi = i & 1
            while len(in_flight) >= DEPTH:
                in_flight.popleft().synchronize()
            stream.wait_event(copied[bi])
            if i + 1 < n:
                copy_in(bi ^ 1)
            res = step(src=bufs[bi])
            consumed[bi].record(stream)
            copy_out(res)
        stream.wait_stream(back_stream)                 # the last results are on the host

    steps = args.steps
    run(min(3, args.warmup))
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    run(steps)
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return {"value": world * w.T * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms / steps,
            "path": "pinned host -> device copies (next step's on a second stream, overlapping this "
                    "step's compute), the four C-ABI calls, every result (x_in, x_next, dx, dy, dphi, "
                    "db, dalpha) -> pinned host on a third stream (overlapping the next step); at most "
                    "3 steps in flight (the host waits for step i-3's results before issuing step i)"}


def graph_latency_us(fn, dev, calls=20, reps=7):
    """Device time of one call of `fn`, from a CUDA graph of `calls`
    back-to-back calls replayed `reps` times (median), so host launch overhead
    does not count."""
    import torch
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(calls):
            fn()
    ts = []
    with torch.cuda.stream(s):   # replay() launches on the current stream
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            g.replay()
            b.record(s)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / calls)
    return statistics.median(ts)


def run_decode(w, dev):
    """Decode-sized batches (T = 1, 8, 32, 64 at the workload's width): latency of
    mhc_pre, of the inference critical path (mhc_pre_critical: x_in, H_pre,
    saved state) and of its side (mhc_post_res_gates: H_post, H_res with
    Sinkhorn, which a second stream overlaps with the sublayer)."""
    from mhc_pre_gb300 import binding as B
    from mhc_pre_gb300 import workloads as W
    out = {}
    for T in (1, 8, 32, 64):
        wd = w.with_(T=T, backward=False)
        inp = W.make_inputs(wd, device=dev)
        x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
        c = B.mhc_pre_critical(x, phi, b, alpha, wd.eps)
        out[str(T)] = {
            "mhc_pre_us": graph_latency_us(lambda: B.mhc_pre(x, phi, b, alpha, wd.iters, wd.eps), dev),
            "critical_path_us": graph_latency_us(lambda: B.mhc_pre_critical(x, phi, b, alpha, wd.eps), dev),
            "side_gates_us": graph_latency_us(lambda: B.mhc_post_res_gates(c.proj, b, alpha, wd.iters), dev),
        }
    assert B.get_last_device_error() == B.MHC_OK
    return {"op": "mhc_pre / mhc_pre_critical + mhc_post_res_gates (side stream)",
            "timing": "CUDA graph of 20 calls, median of 7 replays, inputs L2-warm", "T": out}


def run_sweep(w, inp, dev, reps=10):
    """The Sinkhorn round count of the large-batch workload swept over
    {5, 20, 50}: time of each op that runs Sinkhorn (mhc_pre forward, the
    mhc_pre_bwd recompute with its reverse pass)."""
    import torch
    from mhc_pre_gb300 import binding as B
    stream = torch.cuda.current_stream(dev)
    x, y, phi, b, alpha = (inp[k] for k in ("x", "y", "phi", "b", "alpha"))
    ws = torch.empty((B.pre_bwd_workspace_bytes(x.dtype, w.T, w.n, w.D),), dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(reps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    out = {}
    for iters in (5, 20, 50):
        f = B.mhc_pre(x, phi, b, alpha, iters, w.eps)
        pb = B.mhc_post_bwd(inp["g_next"], x, y, f.H_post, f.H_res)
        dx0 = pb.dx.clone()
        out[str(iters)] = {
            "mhc_pre_ms": timed(lambda: B.mhc_pre(x, phi, b, alpha, iters, w.eps)),
            "mhc_pre_bwd_ms": timed(lambda: B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha,
                                                          f.proj, f.inv_rms, dx0, iters, workspace=ws)),
        }
    assert B.get_last_device_error() == B.MHC_OK
    return {"op": "Sinkhorn rounds swept (large-batch workload)", "iters": out}


def memory_accounting(w):
    """What the backward of one mHC layer keeps per token beyond its inputs,
    set beside the Ascend mHC operator article's count for an unfused
    composition: 2 (7N - 3) B S D bytes more per layer (bf16 values).  Both
    modes keep x (the hc_pre input) and y (the sublayer output), as any
    residual layer does; the saved-state mode adds proj and inv_rms, 100 B per
    token for each mHC op, and the recompute mode (mhc_layer_bwd_recompute)
    adds nothing.  A layer has two mHC ops (attention and MLP/MoE); across
    layers, mhc_post_pre restores layer l + 1's x from layer l's (x, y)."""
    N, D = w.n, w.D
    pages = 2 * (7 * N - 3) * D
    saved = 2 * 4 * (w.G + 1)
    B_, S_ = 1, 4096
    return {"per_token_bytes_per_layer": {"pages_unfused_extra": pages, "saved_state": saved, "recompute": 0},
            "per_layer_bytes_B1_S4096": {"pages_unfused_extra": pages * B_ * S_,
                                         "saved_state": saved * B_ * S_, "recompute": 0},
            "saved_state_fraction_of_pages": saved / pages,
            "formula": "2*(7N-3)*B*S*D (pages), N=%d D=%d" % (N, D)}


if __name__ == "__main__":
    sys.exit(main())
