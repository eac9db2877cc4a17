"""GPU parity of the cross-layer step mhc_post_pre (layer l's residual update,
then layer l + 1's pre forward on the stored x_next) against the float64
oracle's composition, element by element; x_next against mhc_post bit for
bit; sampled tokens at the large-batch size.  Tolerances: tests/parity.py
(compare_post_pre: x_next within one bf16 unit of the exact update rounded
once, and the bounds on proj and inv_rms that such a one-unit difference
implies).
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


def _inputs(w, dev):
    inp = W.make_inputs(w.with_(backward=False), device="cpu")
    gates = W.make_layer_gates(w, device="cpu")
    return ({k: v.to(dev) for k, v in inp.items()}, {k: v.to(dev) for k, v in gates.items()},
            {k: P.f64(v) for k, v in inp.items()}, {k: P.f64(v) for k, v in gates.items()})


def _check(w):
    dev = _dev()
    gi, gg, ci, cg = _inputs(w, dev)
    got = P.run_gpu_post_pre(gi, gg, w.iters, w.eps)
    ref = P.run_oracle_post_pre(ci, cg, w.iters, w.eps, store=w.dtype)
    P.compare_post_pre(got, ref, ci, cg, fp32=(w.dtype == "f32"))
    return gi, gg, got


@pytest.mark.parametrize("wid", [1, 2, 3])
def test_post_pre_workloads(wid):
    _check(W.WORKLOADS[wid])


@pytest.mark.parametrize("T,D,dtype", [
    (129, 5120, "bf16"), (333, 2560, "bf16"), (200, 1024, "bf16"), (64, 256, "bf16"),
    # fewer tokens than one tile
    (1, 5120, "bf16"), (17, 5120, "bf16"), (63, 2560, "bf16"),
    # shapes the fused kernel does not take: mhc_post, then mhc_pre
    (65, 40, "bf16"), (67, 12, "f32"),
])
def test_post_pre_ragged_and_fallback_shapes(T, D, dtype):
    _check(W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=60 + T % 30))


def test_post_pre_peaked_logits():
    # the x10 logits of the large-batch workload at a size the oracle runs fully
    _check(W.WORKLOADS[5].with_(T=257, D=5120))


def test_post_pre_x_next_matches_post_bit_for_bit():
    w = W.WORKLOADS[3].with_(T=1000)
    dev = _dev()
    gi, gg, _, _ = _inputs(w, dev)
    o = B.mhc_post_pre(gi["x"], gi["y"], gg["H_post_l"], gg["H_res_l"], gi["phi"], gi["b"],
                       gi["alpha"], w.iters, w.eps)
    xn = B.mhc_post(gi["x"], gi["y"], gg["H_post_l"], gg["H_res_l"])
    f = B.mhc_pre(xn, gi["phi"], gi["b"], gi["alpha"], w.iters, w.eps)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    assert torch.equal(o.x_next, xn)
    # the pre step of the fused kernel sees the same x_next: its gates agree
    # with mhc_pre's up to the order of the fp32 sums
    for k in ("H_pre", "H_post", "H_res"):
        assert torch.max(torch.abs(getattr(o, k) - getattr(f, k))).item() < 1e-5


def test_post_pre_launch_counts():
    _dev()
    assert B.kernel_launches("mhc_post_pre", "bf16", 32768, 4, 5120) == 2
    assert B.kernel_launches("mhc_post_pre", "bf16", 65, 4, 40) == 3
    assert B.kernel_launches("mhc_post_pre", "f32", 64, 4, 256) == 3


def test_post_pre_large_batch_sampled_tokens():
    """T=32768, D=5120: inputs drawn on the device, sampled tokens against the
    oracle's composition."""
    dev = _dev()
    w = W.WORKLOADS[5]
    inp = W.make_inputs(w.with_(backward=False), device=dev)
    gates = W.make_layer_gates(w, device=dev)
    o = B.mhc_post_pre(inp["x"], inp["y"], gates["H_post_l"], gates["H_res_l"], inp["phi"],
                       inp["b"], inp["alpha"], w.iters, w.eps)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    r = np.random.default_rng(5)
    idx = sorted(set([0, 63, 64, 127, 128, w.T // 2, w.T - 65, w.T - 1]) |
                 set(r.integers(0, w.T, size=40).tolist()))
    ti = torch.as_tensor(idx, device=dev)
    sub = {k: P.f64(inp[k][ti]) for k in ("x", "y")}
    for k in ("phi", "b", "alpha"):
        sub[k] = P.f64(inp[k])
    subg = {k: P.f64(v[ti]) for k, v in gates.items()}
    ref = P.run_oracle_post_pre(sub, subg, w.iters, w.eps, store="bf16")
    got = {k: P.f64(getattr(o, k)[ti]) for k in P.POST_PRE_KEYS}
    P.compare_post_pre(got, ref, sub, subg, fp32=False)
