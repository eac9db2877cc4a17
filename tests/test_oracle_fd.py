"""Central finite differences pin the oracle's backward of the whole layer.

Loss of one mHC layer with the sublayer output y as an independent input:
    L = <g_in, x_in> + <g_next, x_next>
with x_in from ``mhc_pre`` and x_next from ``mhc_post`` (openPangu 2.0 notes,
section 5.3).  The analytic gradient is ``mhc_post_bwd`` followed by
``mhc_pre_bwd`` (dx = post part + pre part).  Central differences in float64
with h = 1e-6 are an independent computation of the same derivative.
"""

import numpy as np
import pytest

from oracle import mhc_oracle as O

N, D, T = 4, 8, 2
G = 2 * N + N * N
EPS = 1e-6


def _inputs(seed, logit_scale=1.0):
    r = np.random.default_rng(seed)
    return dict(
        x=r.normal(size=(T, N, D)),
        y=r.normal(size=(T, D)),
        phi=r.normal(size=(N * D, G)) * 0.3 * logit_scale,
        b=r.normal(size=G) * 0.3,
        alpha=np.array([0.9, 1.1, 1.3]),
        g_in=r.normal(size=(T, D)),
        g_next=r.normal(size=(T, N, D)),
    )


def _loss(p, iters):
    f = O.mhc_pre(p["x"], p["phi"], p["b"], p["alpha"], iters, EPS)
    xn = O.mhc_post(p["x"], p["y"], f["H_post"], f["H_res"])
    return np.sum(p["g_in"] * f["x_in"]) + np.sum(p["g_next"] * xn)


def _analytic(p, iters):
    f = O.mhc_pre(p["x"], p["phi"], p["b"], p["alpha"], iters, EPS)
    pb = O.mhc_post_bwd(p["g_next"], p["x"], p["y"], f["H_post"], f["H_res"])
    qb = O.mhc_pre_bwd(p["g_in"], pb["dH_post"], pb["dH_res"], p["x"],
                       p["phi"], p["b"], p["alpha"], iters, EPS)
    return dict(x=pb["dx"] + qb["dx"], y=pb["dy"], phi=qb["dphi"],
                b=qb["db"], alpha=qb["dalpha"])


def _fd(p, name, iters, h=1e-6):
    base = p[name]
    out = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        q = {k: v.copy() for k, v in p.items()}
        q[name][idx] = base[idx] + h
        lp = _loss(q, iters)
        q[name][idx] = base[idx] - h
        lm = _loss(q, iters)
        out[idx] = (lp - lm) / (2 * h)
    return out


@pytest.mark.parametrize("iters", [1, 5, 20])
@pytest.mark.parametrize("name", ["x", "y", "phi", "b", "alpha"])
def test_gradient_matches_central_differences(name, iters):
    p = _inputs(100 + iters)
    ana = _analytic(p, iters)[name]
    fd = _fd(p, name, iters)
    err = np.linalg.norm(ana - fd) / max(np.linalg.norm(fd), 1e-30)
    assert err < 1e-6, f"{name} iters={iters}: rel err {err:.2e}"


def test_gradient_peaked_logits():
    # logits x10 (like the large-batch bandwidth workload): peaked exp(L)
    p = _inputs(7, logit_scale=10.0)
    ana = _analytic(p, 20)
    for name in ("x", "phi", "b", "alpha"):
        fd = _fd(p, name, 20, h=1e-7)
        err = np.linalg.norm(ana[name] - fd) / np.linalg.norm(fd)
        assert err < 1e-5, f"{name}: rel err {err:.2e}"


def test_rmsnorm_gradient_orthogonal_to_x_without_eps():
    # With eps = 0 the projection path sees only x / rms(x): its gradient
    # has no component along x (scale invariance), token by token.
    p = _inputs(3)
    f = O.mhc_pre(p["x"], p["phi"], p["b"], p["alpha"], 20, 0.0)
    pb = O.mhc_post_bwd(p["g_next"], p["x"], p["y"], f["H_post"], f["H_res"])
    qb = O.mhc_pre_bwd(np.zeros((T, D)), pb["dH_post"], pb["dH_res"], p["x"],
                       p["phi"], p["b"], p["alpha"], 20, 0.0)
    dots = np.einsum("tid,tid->t", qb["dx"], p["x"])
    assert np.max(np.abs(dots)) < 1e-12 * np.max(np.abs(qb["dx"]))
