"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Element by element on the same seeded inputs at sizes the oracle finishes in
seconds (several tiles and a ragged tail), on the five workloads, and on
sampled tokens at the large-batch size in the configuration the benchmark
times.  Tolerances are documented in tests/parity.py.
"""

import numpy as np
import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W
from oracle import mhc_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _inputs(w, dev):
    inp = W.make_inputs(w, device="cpu")
    return {k: v.to(dev) for k, v in inp.items()}, {k: P.f64(v) for k, v in inp.items()}


def _check(w, iters=None, backward=None, keys=None):
    dev = _dev()
    iters = w.iters if iters is None else iters
    backward = w.backward if backward is None else backward
    gi, ci = _inputs(w.with_(backward=backward), dev)
    got = P.run_gpu(gi, iters, w.eps, backward)
    ref = P.run_oracle(ci, iters, w.eps, backward)
    P.compare(got, ref, fp32=(w.dtype == "f32"), keys=keys)


# ------------------------------------------------------------ workloads ---

def test_workload1_tiny_fp32_fwd_bwd():
    _check(W.WORKLOADS[1], backward=True)


def test_workload2_bf16_s1024_d5120():
    _check(W.WORKLOADS[2])


def test_workload3_bf16_s2048_d2560():
    _check(W.WORKLOADS[3])


def test_workload4_bf16_fwd_bwd_s4096():
    _check(W.WORKLOADS[4])


# ----------------------------------------------------- ragged / edge cases ---

@pytest.mark.parametrize("T,D,dtype", [
    (1, 5120, "bf16"), (3, 8, "bf16"), (65, 40, "bf16"), (130, 264, "bf16"),
    (200, 1024, "bf16"), (333, 2560, "bf16"), (129, 5120, "bf16"),
    # widths that give clusters of 1 and 16 with 4, 5 and 3 chunks per CTA,
    # and one (6144) that the one-pass backward does not take
    (64, 256, "bf16"), (150, 320, "bf16"), (100, 3072, "bf16"), (160, 6144, "bf16"),
    (1, 4, "f32"), (67, 12, "f32"), (130, 260, "f32"),
    # fewer tokens than one 64-token tile (decode-sized batches)
    (2, 5120, "bf16"), (17, 5120, "bf16"), (63, 2560, "bf16"), (5, 1024, "bf16"),
    # the split-K cluster kernel (one cluster per eight tokens, at most 56
    # tokens, widths a multiple of 512), its edges, and the first batch past it
    (8, 5120, "bf16"), (8, 512, "bf16"), (4, 6144, "bf16"), (3, 2560, "bf16"), (9, 5120, "bf16"),
    (32, 5120, "bf16"), (26, 1024, "bf16"), (56, 5120, "bf16"), (57, 5120, "bf16"),
    # widths past the cluster kernels' (a phi slice of at most 1280 columns per
    # CTA): the CUDA-core forward, and the two-pass tensor-core backward from
    # one 128-token tile up
    (160, 8192, "bf16"), (33, 8192, "bf16"), (130, 10240, "bf16"),
])
def test_ragged_shapes_fwd_bwd(T, D, dtype):
    w = W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=40 + T % 50)
    _check(w, backward=True)


@pytest.mark.parametrize("iters", [1, 5, 50, 64])
def test_sinkhorn_round_counts(iters):
    w = W.WORKLOADS[5].with_(T=300, D=1024)
    _check(w, iters=iters, backward=True)


def test_zero_alpha_degenerate_gates():
    # alpha = 0: the logits are the bias alone, identical for every token
    w = W.WORKLOADS[4].with_(T=96, D=512, alpha=0.0)
    dev = _dev()
    gi, ci = _inputs(w, dev)
    got = P.run_gpu(gi, w.iters, w.eps, True)
    ref = P.run_oracle(ci, w.iters, w.eps, True)
    P.compare(got, ref, fp32=False)
    hr = P.f64(got["H_res"])
    assert np.max(np.abs(hr - hr[0:1])) == 0.0


def test_peaked_logits_large_batch_shape_small_T():
    # the x10 logits of the large-batch workload at a size the oracle runs fully
    w = W.WORKLOADS[5].with_(T=257, D=5120)
    _check(w, backward=True)


def test_empty_batch_is_a_noop():
    dev = _dev()
    x = torch.empty((0, 4, 64), dtype=torch.bfloat16, device=dev)
    phi = torch.zeros((256, 24), device=dev)
    f = B.mhc_pre(x, phi, torch.zeros(24, device=dev), torch.zeros(3, device=dev))
    assert f.x_in.shape == (0, 64)
    xn = B.mhc_post(x, torch.empty((0, 64), dtype=torch.bfloat16, device=dev), f.H_post, f.H_res)
    assert xn.shape == (0, 4, 64)


def test_empty_batch_writes_zero_param_grads():
    """An empty batch contributes zero parameter gradient (a data-parallel rank
    with no tokens still takes part in the sum): each backward entry point
    writes the zeros itself, through the C ABI, over buffers that start as NaN."""
    dev = _dev()
    L = B.lib()
    D = 64
    s = torch.cuda.current_stream().cuda_stream

    def grads():
        return [torch.full((4 * D, 24), float("nan"), device=dev), torch.full((24,), float("nan"), device=dev),
                torch.full((3,), float("nan"), device=dev)]

    g = grads()
    assert L.mhc_pre_bwd(B.MHC_BF16, *([None] * 9), 0, 4, D, 20, None, *[t.data_ptr() for t in g],
                         None, 0, s) == B.MHC_OK
    torch.cuda.synchronize()
    assert all(torch.count_nonzero(t).item() == 0 for t in g)
    g = grads()
    assert L.mhc_pre_bwd_noalloc(B.MHC_BF16, *([None] * 9), 0, 4, D, 20, None,
                                 *[t.data_ptr() for t in g], s) == B.MHC_OK
    torch.cuda.synchronize()
    assert all(torch.count_nonzero(t).item() == 0 for t in g)
    g = grads()
    assert L.mhc_layer_bwd_recompute(B.MHC_F32, *([None] * 7), 0, 4, D, 20, 1e-6, None, None,
                                     *[t.data_ptr() for t in g], None, 0, s) == B.MHC_OK
    torch.cuda.synchronize()
    assert all(torch.count_nonzero(t).item() == 0 for t in g)
    assert B.get_last_device_error() == B.MHC_OK


def test_invariants_hold_on_gpu_output():
    # properties that hold at any size: ranges, exact column sums, stream sums
    w = W.WORKLOADS[5].with_(T=2048, D=2560)
    dev = _dev()
    gi, _ = _inputs(w, dev)
    got = P.run_gpu(gi, w.iters, w.eps, False)
    hp, hq, hr = (P.f64(got[k]) for k in ("H_pre", "H_post", "H_res"))
    assert np.all((hp > 0) & (hp < 1)) and np.all((hq > 0) & (hq < 2))
    assert np.all(hr >= 0)
    assert np.max(np.abs(hr.sum(axis=1) - 1.0)) < 1e-5     # columns: exact up to fp32
    assert np.max(np.abs(hr.sum(axis=2) - 1.0)) < 2e-3     # rows: converged


# -------------------------------------------- large batch, sampled tokens ---

def _sampled_tokens(T, count, seed):
    r = np.random.default_rng(seed)
    idx = set([0, 1, T - 2, T - 1, T // 2, 127, 128, 129])
    idx.update(r.integers(0, T, size=count).tolist())
    return np.array(sorted(i for i in idx if 0 <= i < T))


@pytest.mark.parametrize("iters", list(W.SINKHORN_SWEEP))
def test_large_batch_forward_sampled_tokens(iters):
    """T=32768, D=5120 as the benchmark runs it: inputs drawn on the device,
    every per-token output checked on sampled tokens against the oracle."""
    dev = _dev()
    w = W.WORKLOADS[5]
    inp = W.make_inputs(w, device=dev)
    f = B.mhc_pre(inp["x"], inp["phi"], inp["b"], inp["alpha"], iters, w.eps)
    xn = B.mhc_post(inp["x"], inp["y"], f.H_post, f.H_res)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    idx = _sampled_tokens(w.T, 48, iters)
    ti = torch.as_tensor(idx, device=dev)
    sub = {k: P.f64(inp[k][ti]) for k in ("x", "y")}
    for k in ("phi", "b", "alpha"):
        sub[k] = P.f64(inp[k])
    ref = P.run_oracle(sub, iters, w.eps, False)
    got = dict(x_in=f.x_in[ti], H_pre=f.H_pre[ti], H_post=f.H_post[ti], H_res=f.H_res[ti],
               proj=f.proj[ti], inv_rms=f.inv_rms[ti], x_next=xn[ti])
    P.compare(got, ref, fp32=False)


def test_large_batch_backward_sampled_and_reduced():
    """Backward at T=32768: per-token gradients on sampled tokens; dphi, db,
    dalpha (sums over all tokens) against the oracle run chunk by chunk."""
    dev = _dev()
    w = W.WORKLOADS[5]
    inp = W.make_inputs(w, device=dev)
    got = P.run_gpu(inp, w.iters, w.eps, True)
    idx = _sampled_tokens(w.T, 24, 7)
    ti = torch.as_tensor(idx, device=dev)
    sub = {k: P.f64(inp[k][ti]) for k in ("x", "y", "g_in", "g_next")}
    for k in ("phi", "b", "alpha"):
        sub[k] = P.f64(inp[k])
    ref = P.run_oracle(sub, w.iters, w.eps, True)
    P.compare({k: got[k][ti] for k in ("dx", "dy", "dH_post", "dH_res")}, ref,
              fp32=False, keys=("dx", "dy", "dH_post", "dH_res"))
    # parameter gradients: the oracle's sums over token chunks
    dphi = np.zeros_like(P.f64(inp["phi"]))
    db = np.zeros(24)
    dal = np.zeros(3)
    phi, b, al = (P.f64(inp[k]) for k in ("phi", "b", "alpha"))
    chunk = 2048
    for t0 in range(0, w.T, chunk):
        sl = slice(t0, t0 + chunk)
        x = P.f64(inp["x"][sl])
        f = O.mhc_pre(x, phi, b, al, w.iters, w.eps)
        pb = O.mhc_post_bwd(P.f64(inp["g_next"][sl]), x, P.f64(inp["y"][sl]),
                            f["H_post"], f["H_res"])
        qb = O.mhc_pre_bwd(P.f64(inp["g_in"][sl]), pb["dH_post"], pb["dH_res"], x, phi, b,
                           al, w.iters, w.eps)
        dphi += qb["dphi"]
        db += qb["db"]
        dal += qb["dalpha"]
    P.close_rel("dphi", P.f64(got["dphi"]), dphi)
    P.close_rel("db", P.f64(got["db"]), db)
    P.close_rel("dalpha", P.f64(got["dalpha"]), dal)
