"""mhc_pre_bwd_noalloc against mhc_pre_bwd, through the C ABI (GPU), on every
backward path (one-pass cluster, two-pass tensor-core, CUDA-core; bf16 and
float32).

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


@pytest.mark.parametrize("wid,T,D,dtype", [
    # float32 activations (the tiny workload's shape): the CUDA-core backward
    (73, 64, 256, "f32"),
    # bf16 widths the one-pass cluster kernel does not tile, at sizes where the
    # fixed array caps the dphi token blocks below the workspace plan's 16:
    # the two-pass tensor-core backward (6 blocks) and the CUDA-core one (14)
    (74, 4096, 6144, "bf16"),
    (75, 8192, 2600, "bf16"),
])
def test_noalloc_matches_workspace_entry_point_on_other_paths(wid, T, D, dtype):
    dev = _dev()
    w = W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=wid)
    inp = W.make_inputs(w, device=dev)
    x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
    f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    pb = B.mhc_post_bwd(inp["g_next"], x, inp["y"], f.H_post, f.H_res)
    for _ in range(2):
        ref = B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj,
                            f.inv_rms, pb.dx.clone(), w.iters)
        got = B.mhc_pre_bwd_noalloc(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha,
                                    f.proj, f.inv_rms, pb.dx.clone(), w.iters)
        torch.cuda.synchronize()
        assert B.get_last_device_error() == B.MHC_OK
        for name in ("dx", "dphi", "db", "dalpha"):
            g, r = P.f64(getattr(got, name)), P.f64(getattr(ref, name))
            if dtype == "f32":
                # the same kernels summing the same values in a different
                # split of token blocks: float32 rounding only
                P.close_abs(name, g, r, P.ATOL_F32 * max(1.0, float(abs(r).max())))
            else:
                P.close_rel(name, g, r)


_CAPTURE_SCRIPT = r"""
import torch
from mhc_pre_gb300 import binding as B

dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
L = B.lib()
T, D = 64, 256
z = lambda *s: torch.zeros(*s, device=dev)
g_in, x, dx = z(T, D), z(T, 4, D), z(T, 4, D)
dH_post, dH_res, phi, b, alpha = z(T, 4), z(T, 4, 4), z(4 * D, 24), z(24), z(3)
proj, inv_rms = z(T, 24), torch.ones(T, device=dev)
dphi, db, dalpha = z(4 * D, 24), z(24), z(3)
args = [t.data_ptr() for t in (g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms)]
outs = [t.data_ptr() for t in (dx, dphi, db, dalpha)]
s = torch.cuda.Stream()
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph, stream=s):
    st_capture = L.mhc_pre_bwd_noalloc(B.MHC_F32, *args, T, 4, D, 20, *outs, s.cuda_stream)
st_after = L.mhc_pre_bwd_noalloc(B.MHC_F32, *args, T, 4, D, 20, *outs, s.cuda_stream)
torch.cuda.synchronize()
print("STATUS", st_capture, st_after, B.get_last_device_error())
"""


def test_first_call_while_capturing_is_refused():
    """In a fresh process, the first call comes while its stream is being
    captured: it must return MHC_ERR_UNSUPPORTED without launching anything;
    the next call, outside the capture, looks the array up and succeeds."""
    import os
    import subprocess
    import sys
    _dev()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_SCRIPT], cwd=root, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("STATUS")][-1]
    assert line.split()[1:] == [str(B.MHC_ERR_UNSUPPORTED), str(B.MHC_OK), str(B.MHC_OK)], line


@pytest.mark.parametrize("wid,T,D,dtype", [(76, 333, 2560, "bf16"), (77, 64, 256, "f32")])
def test_noalloc_against_the_oracle(wid, T, D, dtype):
    """The layer's backward with mhc_pre_bwd_noalloc in place of mhc_pre_bwd,
    element by element against the float64 oracle (the same tolerances as
    the parity tests), so that this entry point is pinned to the oracle
    directly and not only through the workspace entry point."""
    import numpy as np
    dev = _dev()
    w = W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=wid, backward=True)
    cpu = W.make_inputs(w, device="cpu")
    inp = {k: v.to(dev) for k, v in cpu.items()}
    ref = P.run_oracle({k: P.f64(v) for k, v in cpu.items()}, w.iters, w.eps, True)
    x, phi, b, alpha = inp["x"], inp["phi"], inp["b"], inp["alpha"]
    f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    pb = B.mhc_post_bwd(inp["g_next"], x, inp["y"], f.H_post, f.H_res)
    qb = B.mhc_pre_bwd_noalloc(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj, f.inv_rms,
                               pb.dx, w.iters)
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    got = dict(dx=qb.dx, dphi=qb.dphi, db=qb.db, dalpha=qb.dalpha)
    P.compare(got, ref, fp32=(dtype == "f32"), keys=("dx", "dphi", "db", "dalpha"))
    assert np.isfinite(P.f64(qb.dphi)).all()
