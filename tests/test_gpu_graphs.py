"""The library's calls inside CUDA graphs: a whole fwd+bwd step, the
cross-layer step (a memset, a cluster kernel and a second kernel launched
with programmatic dependent launch) and the recompute-oriented backward
(seven launches), captured once and replayed, give the same bits as the same
calls run eagerly."""

import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _step(a, w, ws):
    f = B.mhc_pre(a["x"], a["phi"], a["b"], a["alpha"], w.iters, w.eps)
    xn = B.mhc_post(a["x"], a["y"], f.H_post, f.H_res)
    pb = B.mhc_post_bwd(a["g_next"], a["x"], a["y"], f.H_post, f.H_res)
    qb = B.mhc_pre_bwd(a["g_in"], pb.dH_post, pb.dH_res, a["x"], a["phi"], a["b"], a["alpha"],
                       f.proj, f.inv_rms, pb.dx, w.iters, workspace=ws)
    return [f.x_in, f.H_pre, f.H_res, xn, pb.dy, qb.dx, qb.dphi, qb.db, qb.dalpha]


def test_step_in_a_cuda_graph_matches_eager():
    dev = _dev()
    w = W.WORKLOADS[4].with_(T=1000)
    a = W.make_inputs(w, device=dev)
    ws = torch.empty((B.pre_bwd_workspace_bytes(torch.bfloat16, w.T, w.n, w.D),), dtype=torch.uint8, device=dev)
    eager = [t.clone() for t in _step(a, w, ws)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        _step(a, w, ws)              # warm-up on the capture stream
    torch.cuda.current_stream(dev).wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = _step(a, w, ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for e, o in zip(eager, out):
        assert torch.equal(e, o)


def test_cross_layer_step_in_a_cuda_graph_matches_eager():
    dev = _dev()
    w = W.WORKLOADS[2].with_(T=2000)
    a = W.make_inputs(w, device=dev)
    gates = W.make_layer_gates(w, device=dev)
    run = lambda: B.mhc_post_pre(a["x"], a["y"], gates["H_post_l"], gates["H_res_l"], a["phi"], a["b"],
                                 a["alpha"], w.iters, w.eps)
    eager = [t.clone() for t in run()]
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream(dev).wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for e, o in zip(eager, out):
        assert torch.equal(e, o)


def test_recompute_backward_in_a_cuda_graph_matches_eager():
    dev = _dev()
    w = W.WORKLOADS[4].with_(T=1000)
    a = W.make_inputs(w, device=dev)
    ws = torch.empty((B.layer_bwd_recompute_workspace_bytes(torch.bfloat16, w.T, w.n, w.D),),
                     dtype=torch.uint8, device=dev)
    run = lambda: B.mhc_layer_bwd_recompute(a["g_in"], a["g_next"], a["x"], a["y"], a["phi"], a["b"],
                                            a["alpha"], w.iters, w.eps, workspace=ws)
    eager = [t.clone() for t in run()]
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream(dev).wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = run()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    for e, o in zip(eager, out):
        assert torch.equal(e, o)


_SMALL_BATCH_CAPTURE_SCRIPT = r"""
import torch
from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W

dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
w = W.WORKLOADS[5].with_(T=4, backward=False)
a = W.make_inputs(w, device=dev)
s = torch.cuda.Stream(dev)
s.wait_stream(torch.cuda.current_stream(dev))
g = torch.cuda.CUDAGraph()
# the first small-batch call of the process is made inside the capture
with torch.cuda.graph(g, stream=s):
    f = B.mhc_pre(a["x"], a["phi"], a["b"], a["alpha"], w.iters, w.eps)
g.replay()
torch.cuda.synchronize()
e = B.mhc_pre(a["x"], a["phi"], a["b"], a["alpha"], w.iters, w.eps)
torch.cuda.synchronize()
same = all(torch.equal(getattr(f, k), getattr(e, k)) for k in ("x_in", "H_pre", "H_post", "H_res", "proj", "inv_rms"))
print("RESULT", int(same), B.get_last_device_error())
"""


def test_small_batch_forward_captured_as_the_first_call():
    """In a fresh process, the first call of the small-batch forward (T = 4)
    happens inside a CUDA-graph capture, where the library looks up its
    cluster occupancy: the replayed graph gives the eager call's bits."""
    import os
    import subprocess
    import sys
    _dev()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _SMALL_BATCH_CAPTURE_SCRIPT], cwd=root, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT")][-1]
    assert line.split()[1:] == ["1", str(B.MHC_OK)], line
