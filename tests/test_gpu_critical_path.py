"""The inference critical-path split (openPangu 2.0 notes, section 11.3),
on the GPU: mhc_pre_critical (x_in, H_pre and the saved state, no Sinkhorn)
and mhc_post_res_gates (H_post, H_res from the saved projection), run on two
streams with an event between them.

Checks: every output against the float64 oracle (tolerances of
tests/parity.py); bit-identity with mhc_pre on tensor-core, sub-tile and
fallback shapes; and a two-stream run whose residual update equals the
one-stream mhc_pre + mhc_post result.
"""

import numpy as np
import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _split(inp, w, side_stream=None):
    x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
    c = B.mhc_pre_critical(x, phi, b, alpha, w.eps)
    g = B.mhc_post_res_gates(c.proj, b, alpha, w.iters)
    return c, g


@pytest.mark.parametrize("wid", [1, 2, 3])
def test_split_matches_the_oracle(wid):
    dev = _dev()
    w = W.WORKLOADS[wid].with_(backward=False)
    cpu = W.make_inputs(w, device="cpu")
    gi = {k: v.to(dev) for k, v in cpu.items()}
    c, g = _split(gi, w)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    got = {"x_in": c.x_in, "H_pre": c.H_pre, "proj": c.proj, "inv_rms": c.inv_rms, "H_post": g.H_post,
           "H_res": g.H_res}
    ref = P.run_oracle({k: P.f64(v) for k, v in cpu.items()}, w.iters, w.eps, False)
    P.compare({k: P.f64(v) for k, v in got.items()}, ref, fp32=(w.dtype == "f32"), keys=got.keys())


@pytest.mark.parametrize("T,D,dtype", [
    (1, 5120, "bf16"), (63, 2560, "bf16"), (129, 5120, "bf16"), (2048, 2560, "bf16"),
    (65, 40, "bf16"), (67, 12, "f32"),
])
def test_split_equals_mhc_pre_bit_for_bit(T, D, dtype):
    dev = _dev()
    w = W.WORKLOADS[5].with_(T=T, D=D, dtype=dtype, backward=False, wid=40 + T % 17)
    inp = W.make_inputs(w, device=dev)
    f = B.mhc_pre(inp["x"], inp["phi"], inp["b"], inp["alpha"], w.iters, w.eps)
    c, g = _split(inp, w)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for k in ("x_in", "H_pre", "proj", "inv_rms"):
        assert torch.equal(getattr(c, k), getattr(f, k)), k
    for k in ("H_post", "H_res"):
        assert torch.equal(getattr(g, k), getattr(f, k)), k


def test_two_streams_with_an_event():
    """Critical path and residual update on the main stream, the side gates on
    a second stream ordered by events, a stand-in sublayer in between."""
    dev = _dev()
    w = W.WORKLOADS[2].with_(T=512, backward=False)
    inp = W.make_inputs(w, device=dev)
    x, y, phi, b, alpha = (inp[k] for k in ("x", "y", "phi", "b", "alpha"))
    ref_f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    ref_next = B.mhc_post(x, y, ref_f.H_post, ref_f.H_res)
    torch.cuda.synchronize()
    main, side = torch.cuda.current_stream(dev), torch.cuda.Stream(dev)
    c = B.mhc_pre_critical(x, phi, b, alpha, w.eps)
    proj_ready = torch.cuda.Event()
    proj_ready.record(main)
    side.wait_event(proj_ready)
    with torch.cuda.stream(side):
        g = B.mhc_post_res_gates(c.proj, b, alpha, w.iters, stream=side)
        gates_ready = torch.cuda.Event()
        gates_ready.record(side)
    # the sublayer runs on x_in meanwhile (a stand-in: any work on the main stream)
    sub = (c.x_in.float() @ torch.ones((w.D, 8), device=dev)).sum()
    main.wait_event(gates_ready)
    x_next = B.mhc_post(x, y, g.H_post, g.H_res)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    assert torch.isfinite(sub)
    assert torch.equal(c.x_in, ref_f.x_in)
    assert torch.equal(x_next, ref_next)


def test_launch_counts():
    _dev()
    assert B.kernel_launches("mhc_pre_critical", "bf16", 4096, 4, 5120) == 1
    assert B.kernel_launches("mhc_pre_critical", "f32", 64, 4, 256) == 2
    assert B.kernel_launches("mhc_post_res_gates", "f32", 64, 4, 256) == 1
