"""mhc_pre_bwd_noalloc against mhc_pre_bwd, through the C ABI (GPU).

Some callers cannot allocate device memory: a custom-op or plugin interface
that gives an op no workspace, a runtime that forbids allocation once it runs,
or a loop that cannot afford cudaMalloc's implicit synchronisation.
mhc_pre_bwd_noalloc serves them from a fixed scratch array inside the library.
This checks it against the entry point that takes a caller workspace, on two
calls in a row with different sizes: the array keeps the previous call's
contents, and nothing of it may leak into the next result.
"""

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


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = _dev()
    # first call: T * 256 B of records leaves room for 7 dphi token blocks
    # (the workspace entry point uses 16), so the two also differ in how
    # dphi is split; second call: smaller and ragged, after the first has
    # filled the array with its own values
    for seed, T, D in ((71, 4096, 5120), (72, 333, 2560)):
        w = W.WORKLOADS[4].with_(T=T, D=D, wid=seed)
        inp = W.make_inputs(w, device=dev)
        x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
        f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
        pb = B.mhc_post_bwd(inp["g_next"], x, inp["y"], f.H_post, f.H_res)
        ref = B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj,
                            f.inv_rms, pb.dx.clone(), w.iters)
        got = B.mhc_pre_bwd_noalloc(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha,
                                    f.proj, f.inv_rms, pb.dx.clone(), w.iters)
        torch.cuda.synchronize()
        assert B.get_last_device_error() == B.MHC_OK
        for name in ("dx", "dphi", "db", "dalpha"):
            P.close_rel(name, P.f64(getattr(got, name)), P.f64(getattr(ref, name)))
