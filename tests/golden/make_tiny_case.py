"""Writes tiny_case.json: a frozen float64 oracle result on a tiny input.

Calls only the oracle.  Re-run it (python tests/golden/make_tiny_case.py) only
together with a deliberate change of the oracle's arithmetic, and name the
passage of the pages that justifies that change in the commit message.
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import mhc_oracle as O  # noqa: E402


def main():
    r = np.random.default_rng(20261202)
    T, n, D = 2, 4, 8
    G = 2 * n + n * n
    inp = dict(x=r.normal(size=(T, n, D)), y=r.normal(size=(T, D)),
               phi=r.normal(size=(n * D, G)) * 0.2, b=r.normal(size=G) * 0.1,
               alpha=np.array([0.5, 0.7, 0.9]), g_in=r.normal(size=(T, D)),
               g_next=r.normal(size=(T, n, D)))
    iters, eps = 20, 1e-6
    f = O.mhc_pre(inp["x"], inp["phi"], inp["b"], inp["alpha"], iters, eps)
    xn = O.mhc_post(inp["x"], inp["y"], f["H_post"], f["H_res"])
    pb = O.mhc_post_bwd(inp["g_next"], inp["x"], inp["y"], f["H_post"],
                        f["H_res"])
    qb = O.mhc_pre_bwd(inp["g_in"], pb["dH_post"], pb["dH_res"], inp["x"],
                       inp["phi"], inp["b"], inp["alpha"], iters, eps)
    out = dict(x_in=f["x_in"], H_pre=f["H_pre"], H_post=f["H_post"],
               H_res=f["H_res"], x_next=xn, dx=pb["dx"] + qb["dx"],
               dy=pb["dy"], dphi=qb["dphi"], db=qb["db"], dalpha=qb["dalpha"])
    doc = dict(_about="frozen oracle output, written by make_tiny_case.py",
               iters=iters, eps=eps,
               inputs={k: v.tolist() for k, v in inp.items()},
               outputs={k: v.tolist() for k, v in out.items()})
    with open(os.path.join(HERE, "tiny_case.json"), "w") as fh:
        json.dump(doc, fh)


if __name__ == "__main__":
    main()
