"""GPU parity of the residual update with openPangu's stability changes
(mhc_post_norm / mhc_post_norm_bwd: sandwich normalisation of the sublayer
output, block post-normalisation of the multi-stream state) against the
float64 oracle, every flag combination; tolerances as tests/parity.py.
"""

import numpy as np
import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W
from oracle import mhc_oracle as O
from tests import parity as P

pytestmark = pytest.mark.gpu

FLAGS = [0, B.SANDWICH_NORM, B.BLOCK_NORM, B.SANDWICH_NORM | B.BLOCK_NORM]


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _run(w, flags, dev, sample=None):
    inp = W.make_inputs(w.with_(backward=True), device="cpu")
    gates = W.make_layer_gates(w, device="cpu")
    g = {k: v.to(dev) for k, v in {**inp, **gates}.items()}
    f = B.mhc_post_norm(g["x"], g["y"], g["H_post_l"], g["H_res_l"], flags, w.eps)
    b = B.mhc_post_norm_bwd(g["g_next"], g["x"], g["y"], g["H_post_l"], g["H_res_l"], flags,
                            f.inv_rms_y, f.inv_rms_out, w.eps)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    got = dict(x_next=f.x_next, inv_rms_y=f.inv_rms_y, inv_rms_out=f.inv_rms_out,
               dx=b.dx, dy=b.dy, dH_post=b.dH_post, dH_res=b.dH_res)
    c = {k: P.f64(v) for k, v in {**inp, **gates}.items()}
    if sample is not None:
        got = {k: P.f64(v)[sample] for k, v in got.items()}
        c = {k: (v[sample] if v.ndim and v.shape[0] == w.T else v) for k, v in c.items()}
    ref = O.mhc_post_norm(c["x"], c["y"], c["H_post_l"], c["H_res_l"], flags, w.eps)
    ref.update(O.mhc_post_norm_bwd(c["g_next"], c["x"], c["y"], c["H_post_l"], c["H_res_l"], flags, w.eps))
    return got, ref


def _compare(got, ref, fp32):
    for k in ("inv_rms_y", "inv_rms_out"):
        g = got[k] if isinstance(got[k], np.ndarray) else P.f64(got[k])
        P.close_abs(k, g / ref[k], np.ones_like(ref[k]), 1e-5)
    P.compare(got, ref, fp32=fp32, keys=("x_next", "dx", "dy", "dH_post", "dH_res"))


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("wid", [1, 2, 3])
def test_post_norm_workloads(flags, wid):
    w = W.WORKLOADS[wid]
    got, ref = _run(w, flags, _dev())
    _compare(got, ref, fp32=(w.dtype == "f32"))


@pytest.mark.parametrize("T,D,dtype", [(333, 2560, "bf16"), (7, 40, "bf16"), (65, 8192, "bf16"),
                                       (67, 12, "f32"), (5, 4096, "f32")])
def test_post_norm_ragged_shapes(T, D, dtype):
    w = W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=70 + T % 20)
    got, ref = _run(w, B.SANDWICH_NORM | B.BLOCK_NORM, _dev())
    _compare(got, ref, fp32=(dtype == "f32"))


def test_no_flags_matches_mhc_post_bit_for_bit():
    dev = _dev()
    w = W.WORKLOADS[3]
    inp = W.make_inputs(w, device=dev)
    gates = W.make_layer_gates(w, device=dev)
    f = B.mhc_post_norm(inp["x"], inp["y"], gates["H_post_l"], gates["H_res_l"], 0, w.eps)
    xn = B.mhc_post(inp["x"], inp["y"], gates["H_post_l"], gates["H_res_l"])
    torch.cuda.synchronize()
    assert torch.equal(f.x_next, xn)
    assert torch.all(f.inv_rms_y == 1) and torch.all(f.inv_rms_out == 1)


def test_width_limit_and_flags_are_checked():
    dev = _dev()
    x = torch.zeros((4, 4, 8200), dtype=torch.bfloat16, device=dev)
    y = torch.zeros((4, 8200), dtype=torch.bfloat16, device=dev)
    h, r = torch.zeros((4, 4), device=dev), torch.zeros((4, 4, 4), device=dev)
    with pytest.raises(B.MhcError):
        B.mhc_post_norm(x, y, h, r, 3)
    with pytest.raises(B.MhcError):
        B.mhc_post_norm(x[:, :, :64].contiguous(), y[:, :64].contiguous(), h, r, 4)


def test_post_norm_large_batch_sampled_tokens():
    w = W.WORKLOADS[5]
    idx = np.array(sorted({0, 1, 4095, 4096, w.T // 2, w.T - 1} |
                          set(np.random.default_rng(3).integers(0, w.T, 24).tolist())))
    got, ref = _run(w, B.SANDWICH_NORM | B.BLOCK_NORM, _dev(), sample=idx)
    _compare(got, ref, fp32=False)
