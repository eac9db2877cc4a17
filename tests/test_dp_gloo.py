"""Data-parallel path on CPU: two gloo ranks split the tokens, run the layer's
forward and backward on their own shard, and sum dphi, db, dalpha with
``allreduce_param_grads``.  The result must equal the full-batch backward:
the parameters are shared by all tokens, every other output is per token
(openPangu 2.0 notes, section 5.3).

The per-rank compute here is the float64 oracle, so this checks the host
logic of the multi-rank path (token split, packed all-reduce, write-back)
without a GPU; the GPU path runs the same helper over NCCL.
"""

import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

from mhc_pre_gb300.dp import allreduce_param_grads, shard_range
from oracle import mhc_oracle as O

N, D, ITERS, EPS = 4, 16, 20, 1e-6
G = 2 * N + N * N


def _inputs(T, seed=5):
    r = np.random.default_rng(seed)
    return dict(x=r.normal(size=(T, N, D)), y=r.normal(size=(T, D)),
                phi=r.normal(size=(N * D, G)) * 0.2, b=r.normal(size=G) * 0.3,
                alpha=np.array([0.7, 1.1, 1.4]), g_in=r.normal(size=(T, D)),
                g_next=r.normal(size=(T, N, D)))


def _layer_grads(p, lo, hi):
    sl = slice(lo, hi)
    x, y = p["x"][sl], p["y"][sl]
    f = O.mhc_pre(x, p["phi"], p["b"], p["alpha"], ITERS, EPS)
    pb = O.mhc_post_bwd(p["g_next"][sl], x, y, f["H_post"], f["H_res"])
    qb = O.mhc_pre_bwd(p["g_in"][sl], pb["dH_post"], pb["dH_res"], x, p["phi"], p["b"],
                       p["alpha"], ITERS, EPS)
    return dict(dx=pb["dx"] + qb["dx"], dy=pb["dy"], dphi=qb["dphi"], db=qb["db"],
                dalpha=qb["dalpha"])


def _rank_main(rank, world, port, T, out_dir):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = _inputs(T)
        lo, hi = shard_range(T, rank, world)
        g = _layer_grads(p, lo, hi)
        dphi = torch.from_numpy(g["dphi"].astype(np.float32))
        db = torch.from_numpy(g["db"].astype(np.float32))
        dalpha = torch.from_numpy(g["dalpha"].astype(np.float32))
        allreduce_param_grads(dphi, db, dalpha)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), lo=lo, hi=hi, dx=g["dx"],
                 dy=g["dy"], dphi=dphi.numpy(), db=db.numpy(), dalpha=dalpha.numpy())
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run(world, T, tmp_path):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, T, str(tmp_path)))
             for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=120)
    for pr in procs:
        if pr.is_alive():
            pr.kill()
            pr.join()
    assert all(pr.exitcode == 0 for pr in procs), [pr.exitcode for pr in procs]
    return [dict(np.load(tmp_path / f"rank{r}.npz")) for r in range(world)]


@pytest.mark.parametrize("T", [7, 1])
def test_two_ranks_match_the_full_batch(T, tmp_path):
    world = 2
    ranks = _run(world, T, tmp_path)
    full = _layer_grads(_inputs(T), 0, T)
    for r in ranks:
        # the summed parameter gradients are the full-batch ones, on every rank
        # (fp32 transport of float64 values: relative 1e-6)
        for k in ("dphi", "db", "dalpha"):
            np.testing.assert_allclose(r[k], full[k], rtol=1e-5,
                                       atol=1e-6 * np.abs(full[k]).max())
        # per-token outputs of a shard are the full batch's rows, untouched
        lo, hi = int(r["lo"]), int(r["hi"])
        np.testing.assert_allclose(r["dx"], full["dx"][lo:hi], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["dy"], full["dy"][lo:hi], rtol=1e-12, atol=1e-12)
    assert sorted((int(r["lo"]), int(r["hi"])) for r in ranks)[0][0] == 0


@pytest.mark.parametrize("T,world", [(0, 1), (7, 2), (1, 2), (10, 3), (32768, 8), (5, 8)])
def test_shard_range_partitions_the_tokens(T, world):
    ranges = [shard_range(T, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= (1 if T % world else 0)


def test_shard_range_rejects_bad_arguments():
    for args in ((4, 2, 2), (4, -1, 2), (4, 0, 0), (-1, 0, 1)):
        with pytest.raises(ValueError):
            shard_range(*args)
