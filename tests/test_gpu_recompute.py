"""GPU checks of the recompute-oriented backward (mhc_pre_gates and
mhc_layer_bwd_recompute): the layer's backward from its inputs x and y alone.

- mhc_pre_gates writes the gates and the saved state bit for bit as mhc_pre
  does (same kernel, mix skipped), on the tensor-core path, the CUDA-core
  path and partial tiles;
- mhc_layer_bwd_recompute gives bit for bit what mhc_post_bwd then
  mhc_pre_bwd give on mhc_pre's saved state, and matches the float64
  oracle's layer backward element by element (tolerances: tests/parity.py);
- both hold at the large-batch size (T = 32768, D = 5120).
"""

import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W
from tests import parity as P

pytestmark = pytest.mark.gpu

LAYER_BWD_KEYS = ("dx", "dy", "dphi", "db", "dalpha")


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _saved_state_bwd(a, w):
    f = B.mhc_pre(a["x"], a["phi"], a["b"], a["alpha"], w.iters, w.eps)
    pb = B.mhc_post_bwd(a["g_next"], a["x"], a["y"], f.H_post, f.H_res)
    qb = B.mhc_pre_bwd(a["g_in"], pb.dH_post, pb.dH_res, a["x"], a["phi"], a["b"], a["alpha"],
                       f.proj, f.inv_rms, pb.dx, w.iters)
    return f, dict(dx=qb.dx, dy=pb.dy, dphi=qb.dphi, db=qb.db, dalpha=qb.dalpha)


def _recompute_bwd(a, w):
    r = B.mhc_layer_bwd_recompute(a["g_in"], a["g_next"], a["x"], a["y"], a["phi"], a["b"],
                                  a["alpha"], w.iters, w.eps)
    return r._asdict()


def _check_bit_exact(w):
    dev = _dev()
    a = W.make_inputs(w.with_(backward=True), device=dev)
    f, saved = _saved_state_bwd(a, w)
    g = B.mhc_pre_gates(a["x"], a["phi"], a["b"], a["alpha"], w.iters, w.eps)
    rec = _recompute_bwd(a, w)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for k in ("H_pre", "H_post", "H_res", "proj", "inv_rms"):
        assert torch.equal(getattr(g, k), getattr(f, k)), k
    for k in LAYER_BWD_KEYS:
        assert torch.equal(rec[k], saved[k]), k
    return a, rec


@pytest.mark.parametrize("wid", [1, 2, 3, 4])
def test_recompute_matches_saved_state_bit_for_bit(wid):
    _check_bit_exact(W.WORKLOADS[wid])


@pytest.mark.parametrize("T,D,dtype", [(1, 5120, "bf16"), (17, 2560, "bf16"), (129, 5120, "bf16"),
                                       (65, 40, "bf16"), (67, 12, "f32")])
def test_recompute_ragged_and_small_shapes(T, D, dtype):
    _check_bit_exact(W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=80 + T % 10))


@pytest.mark.parametrize("wid", [1, 3])
def test_layer_bwd_recompute_against_oracle(wid):
    w = W.WORKLOADS[wid].with_(backward=True)
    dev = _dev()
    inp = W.make_inputs(w, device="cpu")
    got = _recompute_bwd({k: v.to(dev) for k, v in inp.items()}, w)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    ref = P.run_oracle({k: P.f64(v) for k, v in inp.items()}, w.iters, w.eps, backward=True)
    P.compare(got, ref, fp32=(w.dtype == "f32"), keys=LAYER_BWD_KEYS)


def test_recompute_large_batch_bit_for_bit():
    """T = 32768, D = 5120: the gates-only launch and the recompute backward
    against the saved-state path, every element."""
    _check_bit_exact(W.WORKLOADS[5])


def test_recompute_launch_counts():
    _dev()
    assert B.kernel_launches("mhc_pre_gates", "bf16", 32768, 4, 5120) == 1
    assert B.kernel_launches("mhc_layer_bwd_recompute", "bf16", 32768, 4, 5120) == 7
