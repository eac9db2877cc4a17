"""Helpers for GPU-vs-oracle parity tests (test infrastructure).

Tolerances (the layer's stated bar):
  * float32 activations: max |gpu - ref| <= 1e-5 on every per-token output
    (x_in, x_next, the gates, proj, inv_rms, dx, dy).  The reductions
    dH_post, dH_res (sums over D) and dphi, db, dalpha (sums over T) are held
    to 1e-5 times max(1, their largest magnitude): a float32 sum of N terms
    carries an error proportional to the terms' magnitudes, so an absolute
    1e-5 on an entry of size 50 would ask for two float32 units, which no
    summation order guarantees;
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


def bf16_unit(v):
    """One unit in the last place of bfloat16 at the magnitude of v (8
    significant bits)."""
    v = np.asarray(v, dtype=np.float64)
    return np.ldexp(1.0, np.frexp(np.where(v == 0.0, 1e-38, v))[1] - 8)


def compare_post_pre(got, ref, inp_np, gates_np, fp32: bool):
    """The cross-layer step against the oracle's composition.

    x_next is the update rounded to its storage type.  The kernel sums in
    float32 and rounds once; the oracle rounds the exact value once.  The two
    agree except where the float32 sum lands on the other side of a rounding
    boundary, which moves that element by one bfloat16 unit.  The bf16 check
    is therefore: within one unit of the oracle's stored value, and within
    the usual 2e-2 relative bound.  Where the terms cancel, the float32 sum's
    own error (at most (n + 1) 2^-24 times the sum of the terms' magnitudes,
    the standard bound for n + 1 roundings) can exceed a unit of the small
    result, so that bound is added.

    Every later output is a function of the stored x_next, so a flipped
    element propagates: to first order, inv_rms moves by at most
    (1/2) sum_k (2 |x_k| |dx_k| + dx_k^2) / sum_k x_k^2 of its value, and each
    logit's projection by |proj| times that plus inv_rms * sum_k |phi_kg| |dx_k|,
    where dx is the difference of the two stored x_next.  Those terms are
    added to the bounds of ``compare``; the gates keep their plain bound.
    """
    xg = np.asarray(got["x_next"] if isinstance(got["x_next"], np.ndarray) else f64(got["x_next"]))
    xr = ref["x_next"]
    if fp32:
        compare(got, ref, True, keys=POST_PRE_KEYS)
        return
    close_rel("x_next", xg, xr)
    diff = np.abs(xg - xr)
    n = xr.shape[1]
    mag = O.mhc_post(np.abs(inp_np["x"]), np.abs(inp_np["y"]), np.abs(gates_np["H_post_l"]),
                     np.abs(gates_np["H_res_l"]))
    allowed = bf16_unit(xr) + 2.0 * (n + 1) * 2.0 ** -24 * mag
    assert np.all(diff <= allowed), f"x_next: {int(np.sum(diff > allowed))} elements beyond one bf16 unit"
    phi = inp_np["phi"]
    T = xr.shape[0]
    K = int(np.prod(xr.shape[1:]))
    xf = np.abs(xr.reshape(T, K))
    dxf = diff.reshape(T, K)
    ss = np.sum(xf * xf, axis=1)
    rel_inv = 0.5 * np.sum(2.0 * xf * dxf + dxf * dxf, axis=1) / np.maximum(ss, 1e-300)
    inv = ref["inv_rms"]
    gi = np.asarray(got["inv_rms"] if isinstance(got["inv_rms"], np.ndarray) else f64(got["inv_rms"]))
    err_inv = np.abs(gi / inv - 1.0)
    assert np.all(err_inv <= 1e-5 + rel_inv), f"inv_rms: worst relative error {float(np.max(err_inv - rel_inv)):.3g}"
    gp = np.asarray(got["proj"] if isinstance(got["proj"], np.ndarray) else f64(got["proj"]))
    pr = ref["proj"]
    flip = inv[:, None] * (dxf @ np.abs(np.asarray(phi, dtype=np.float64))) + np.abs(pr) * rel_inv[:, None]
    base = 1e-4 * max(1.0, float(np.max(np.abs(pr))))
    err = np.abs(gp - pr)
    bad = err > base + flip
    assert not np.any(bad), f"proj: {int(bad.sum())} elements out of tolerance (worst excess " \
                            f"{float(np.max(err - base - flip)):.3g})"
    compare(got, ref, False, keys=("x_in", "H_pre", "H_post", "H_res"))


GATES = ("H_pre", "H_post", "H_res")


def compare(got, ref, fp32: bool, keys=None):
    keys = keys if keys is not None else ref.keys()
    for k in keys:
        g = got[k] if isinstance(got[k], np.ndarray) else f64(got[k])
        if fp32:
            scale = 1.0
            if k in ("dphi", "db", "dalpha", "dH_post", "dH_res"):
                # float32 sums over tokens or over D: their rounding error is
                # proportional to their magnitude
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
