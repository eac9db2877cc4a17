"""Golden fixtures: the pages' printed numbers and a frozen oracle result."""

import json
import os

import numpy as np

from mhc_pre_gb300 import workloads as W
from oracle import mhc_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    with open(os.path.join(GOLDEN, "page_facts.json")) as f:
        return {d["key"]: d["value"] for d in json.load(f)["facts"]}


def test_workloads_follow_page_facts():
    f = _facts()
    for w in W.WORKLOADS.values():
        assert w.n == f["n_streams"]
        assert w.iters == f["sinkhorn_rounds"]
        assert w.G == 2 * f["n_streams"] + f["n_streams"] ** 2
    assert W.WORKLOADS[2].D == f["hidden_size_pro"]
    assert W.WORKLOADS[3].D == f["hidden_size_flash"]
    shapes = {(w.T, w.n, w.D) for w in W.WORKLOADS.values()}
    for B, S, N, D in f["op_shapes"]:
        assert (B * S, N, D) in shapes
    B, S, D, N = f["activation_shape"]
    assert (B * S, N, D) in shapes


def test_oracle_gate_ranges_follow_page_facts():
    f = _facts()
    lg = np.random.default_rng(0).normal(size=(100, 24)) * 8
    hp, hq = O.gates(lg, 4)
    lo, hi = f["H_pre_range"]
    assert np.all((hp > lo) & (hp < hi))
    lo, hi = f["H_post_range"]
    assert np.all((hq > lo) & (hq < hi))


def test_oracle_reproduces_frozen_tiny_case():
    with open(os.path.join(GOLDEN, "tiny_case.json")) as fh:
        doc = json.load(fh)
    p = {k: np.array(v) for k, v in doc["inputs"].items()}
    it, eps = doc["iters"], doc["eps"]
    f = O.mhc_pre(p["x"], p["phi"], p["b"], p["alpha"], it, eps)
    xn = O.mhc_post(p["x"], p["y"], f["H_post"], f["H_res"])
    pb = O.mhc_post_bwd(p["g_next"], p["x"], p["y"], f["H_post"], f["H_res"])
    qb = O.mhc_pre_bwd(p["g_in"], pb["dH_post"], pb["dH_res"], p["x"],
                       p["phi"], p["b"], p["alpha"], it, eps)
    got = dict(x_in=f["x_in"], H_pre=f["H_pre"], H_post=f["H_post"],
               H_res=f["H_res"], x_next=xn, dx=pb["dx"] + qb["dx"],
               dy=pb["dy"], dphi=qb["dphi"], db=qb["db"], dalpha=qb["dalpha"])
    for k, v in doc["outputs"].items():
        np.testing.assert_allclose(got[k], np.array(v), rtol=1e-12,
                                   atol=1e-14, err_msg=k)
