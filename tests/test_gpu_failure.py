"""Failure path of the bounded waits, made to run out on purpose (GPU).

Every wait on an mbarrier in the tensor-core kernels gives up after a bounded
time, latches a device error word and lets the kernel leave, so that a lost
arrival shows up as MHC_ERR_TIMEOUT instead of a hung GPU.  The test hook
mhc_test_force_timeout arms one such wait, on an mbarrier nothing arrives on,
in the prologue of the forward kernel and of the pre backward's cluster
kernel (before any copy or tensor-memory allocation), with a limit of about
100 us.  Nothing here faults, traps or hangs: the waits end by themselves.
"""

import time

import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _run(inp, w):
    x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
    f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    pb = B.mhc_post_bwd(inp["g_next"], x, inp["y"], f.H_post, f.H_res)
    qb = B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj, f.inv_rms,
                       pb.dx, w.iters)
    return f, qb


def test_forced_timeout_is_reported_and_the_context_stays_usable():
    dev = _dev()
    L = B.lib()
    # a bf16 shape the tensor-core forward and the one-pass backward take
    w = W.WORKLOADS[4].with_(T=256, D=5120, wid=81)
    assert B.kernel_launches("mhc_pre", "bf16", w.T, 4, w.D) == 1
    inp = W.make_inputs(w, device=dev)
    ref_f, ref_b = _run(inp, w)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    try:
        assert L.mhc_test_force_timeout(1) == B.MHC_OK
        t0 = time.monotonic()
        x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
        B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
        assert B.get_last_device_error() == B.MHC_ERR_TIMEOUT
        pb = B.mhc_post_bwd(inp["g_next"], x, inp["y"], ref_f.H_post, ref_f.H_res)
        B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, ref_f.proj, ref_f.inv_rms,
                      pb.dx, w.iters)
        assert B.get_last_device_error() == B.MHC_ERR_TIMEOUT
        # the waits gave up after their short limit: nothing hung
        assert time.monotonic() - t0 < 30.0
    finally:
        assert L.mhc_test_force_timeout(0) == B.MHC_OK
    # the error was read and cleared; the same calls now succeed and give the
    # results of the first run bit for bit
    f, qb = _run(inp, w)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for k in ("x_in", "H_pre", "H_post", "H_res", "proj", "inv_rms"):
        assert torch.equal(getattr(f, k), getattr(ref_f, k)), k
    for k in ("dx", "dphi", "db", "dalpha"):
        assert torch.equal(getattr(qb, k), getattr(ref_b, k)), k


def test_forced_timeout_in_the_small_batch_forward():
    """Two tokens take the cluster split-K forward for small batches: its
    bounded wait gives up under the same hook, the status is reported, and
    the next call gives the first run's outputs bit for bit."""
    dev = _dev()
    L = B.lib()
    w = W.WORKLOADS[4].with_(T=2, D=5120, wid=82)
    inp = W.make_inputs(w, device=dev)
    x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
    ref = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    try:
        assert L.mhc_test_force_timeout(1) == B.MHC_OK
        t0 = time.monotonic()
        B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
        assert B.get_last_device_error() == B.MHC_ERR_TIMEOUT
        assert time.monotonic() - t0 < 30.0
    finally:
        assert L.mhc_test_force_timeout(0) == B.MHC_OK
    f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for k in ("x_in", "H_pre", "H_post", "H_res", "proj", "inv_rms"):
        assert torch.equal(getattr(f, k), getattr(ref, k)), k
