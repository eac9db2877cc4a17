"""Helpers for GPU-vs-oracle parity tests (test infrastructure).

Tolerances (the layer's stated bar):
  * float32 activations: max |gpu - ref| <= 1e-5 on every output (scaled by
    the output's largest magnitude for the reductions dH_post, dH_res, dphi,
    db, dalpha);
  * bf16 activations: gate matrices H_pre, H_post, H_res max abs <= 1e-4;
    every other output per element |gpu - ref| <= 2e-2 * (|ref| + rms(ref))
    (2e-2 relative, with a floor at 2e-2 of the output's RMS for entries near
    zero), plus a relative Frobenius error <= 2e-2.
"""

from __future__ import annotations

import numpy as np
import torch

from mhc_pre_gb300 import binding as B
from oracle import mhc_oracle as O

GATE_ATOL_BF16 = 1e-4
REL_BF16 = 2e-2
ATOL_F32 = 1e-5


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def close_rel(name, got, ref, rel=REL_BF16):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = rel * (np.abs(ref) + rms)
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (rms {rms:.3g})")
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert fro <= rel, f"{name}: relative Frobenius error {fro:.3g}"


def close_abs(name, got, ref, atol):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite output"
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= atol, f"{name}: max abs error {err:.3g} > {atol:.1g}"


def run_gpu(inp, iters, eps, backward):
    """The whole layer through the C ABI; returns float64 numpy arrays."""
    x, y, phi, b, alpha = (inp[k] for k in ("x", "y", "phi", "b", "alpha"))
    f = B.mhc_pre(x, phi, b, alpha, iters, eps)
    xn = B.mhc_post(x, y, f.H_post, f.H_res)
    out = dict(x_in=f.x_in, H_pre=f.H_pre, H_post=f.H_post, H_res=f.H_res,
               proj=f.proj, inv_rms=f.inv_rms, x_next=xn)
    if backward:
        pb = B.mhc_post_bwd(inp["g_next"], x, y, f.H_post, f.H_res)
        out.update(dy=pb.dy, dH_post=pb.dH_post, dH_res=pb.dH_res)
        qb = B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha,
                           f.proj, f.inv_rms, pb.dx, iters)
        out.update(dx=qb.dx, dphi=qb.dphi, db=qb.db, dalpha=qb.dalpha)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    return out


def run_oracle(inp_np, iters, eps, backward):
    """The float64 oracle on the same (already quantised) inputs."""
    p = inp_np
    f = O.mhc_pre(p["x"], p["phi"], p["b"], p["alpha"], iters, eps)
    out = dict(x_in=f["x_in"], H_pre=f["H_pre"], H_post=f["H_post"], H_res=f["H_res"],
               proj=f["proj"], inv_rms=f["inv_rms"],
               x_next=O.mhc_post(p["x"], p["y"], f["H_post"], f["H_res"]))
    if backward:
        pb = O.mhc_post_bwd(p["g_next"], p["x"], p["y"], f["H_post"], f["H_res"])
        qb = O.mhc_pre_bwd(p["g_in"], pb["dH_post"], pb["dH_res"], p["x"], p["phi"],
                           p["b"], p["alpha"], iters, eps)
        out.update(dy=pb["dy"], dH_post=pb["dH_post"], dH_res=pb["dH_res"],
                   dx=pb["dx"] + qb["dx"], dphi=qb["dphi"], db=qb["db"],
                   dalpha=qb["dalpha"])
    return out


POST_PRE_KEYS = ("x_next", "x_in", "H_pre", "H_post", "H_res", "proj", "inv_rms")


def run_gpu_post_pre(inp, gates, iters, eps):
    """The cross-layer step through the C ABI; float64 numpy arrays."""
    o = B.mhc_post_pre(inp["x"], inp["y"], gates["H_post_l"], gates["H_res_l"], inp["phi"],
                       inp["b"], inp["alpha"], iters, eps)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    return {k: f64(getattr(o, k)) for k in POST_PRE_KEYS}


def run_oracle_post_pre(inp_np, gates_np, iters, eps, store):
    """The float64 oracle's cross-layer step on the same inputs."""
    p = inp_np
    return O.mhc_post_pre(p["x"], p["y"], gates_np["H_post_l"], gates_np["H_res_l"], p["phi"],
                          p["b"], p["alpha"], iters, eps, store)


GATES = ("H_pre", "H_post", "H_res")


def compare(got, ref, fp32: bool, keys=None):
    keys = keys if keys is not None else ref.keys()
    for k in keys:
        g = got[k] if isinstance(got[k], np.ndarray) else f64(got[k])
        if fp32:
            scale = 1.0
            if k in ("dphi", "db", "dalpha", "dH_post", "dH_res"):
                # sums over tokens or over D: the bound scales with the sum
                scale = max(1.0, float(np.max(np.abs(ref[k]))))
            close_abs(k, g, ref[k], ATOL_F32 * scale)
        elif k in GATES:
            close_abs(k, g, ref[k], GATE_ATOL_BF16)
        elif k == "inv_rms":
            close_abs(k, g / ref[k], np.ones_like(ref[k]), 1e-5)
        elif k == "proj":
            close_abs(k, g, ref[k], 1e-4 * max(1.0, float(np.max(np.abs(ref[k])))))
        else:
            close_rel(k, g, ref[k])
