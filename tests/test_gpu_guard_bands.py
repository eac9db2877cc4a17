"""No entry point writes outside its outputs (GPU).

compute-sanitizer is not available here, so every output and workspace
buffer the binding hands to the library is surrounded by 4 KB guard bands
filled with a sentinel byte; after each call the bands must be untouched.
The results must also equal those of the same calls on plain buffers bit for
bit.  The shapes cover ragged tiles, batches below one tile, widths the
tensor-core kernels do not take (the CUDA-core fallbacks) and float32.
"""

import math

import pytest
import torch

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096
SENTINEL = 0xA5


class GuardedAllocator:
    """torch.empty with GUARD sentinel bytes on both sides of every buffer."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype=None, device=None):
        dtype = dtype if dtype is not None else torch.float32
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.uint8, device=device)
        self.bufs.append((buf, n))
        return buf[GUARD:GUARD + n].view(dtype).view(shape)

    def check(self, where):
        torch.cuda.synchronize()
        for i, (buf, n) in enumerate(self.bufs):
            head, tail = buf[:GUARD], buf[GUARD + n:]
            bad = int((head != SENTINEL).sum().item()) + int((tail != SENTINEL).sum().item())
            assert bad == 0, f"{where}: buffer {i} ({n} bytes): {bad} guard bytes overwritten"


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)


def _layer(inp, gates, w, fp32):
    """Every entry point once, through the binding; returns all outputs."""
    x, y, phi, b, alpha = (inp[k] for k in ("x", "y", "phi", "b", "alpha"))
    out = {}
    f = B.mhc_pre(x, phi, b, alpha, w.iters, w.eps)
    out.update({"pre." + k: getattr(f, k) for k in f._fields})
    g = B.mhc_pre_gates(x, phi, b, alpha, w.iters, w.eps)
    out.update({"gates." + k: getattr(g, k) for k in g._fields})
    out["post.x_next"] = B.mhc_post(x, y, f.H_post, f.H_res)
    pb = B.mhc_post_bwd(inp["g_next"], x, y, f.H_post, f.H_res)
    out.update({"post_bwd." + k: getattr(pb, k).clone() for k in pb._fields})
    qb = B.mhc_pre_bwd(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj, f.inv_rms,
                       pb.dx, w.iters)
    out.update({"pre_bwd." + k: getattr(qb, k) for k in qb._fields})
    na = B.mhc_pre_bwd_noalloc(inp["g_in"], pb.dH_post, pb.dH_res, x, phi, b, alpha, f.proj,
                               f.inv_rms, out["post_bwd.dx"].clone(), w.iters)
    out.update({"noalloc." + k: getattr(na, k) for k in na._fields})
    lr = B.mhc_layer_bwd_recompute(inp["g_in"], inp["g_next"], x, y, phi, b, alpha, w.iters, w.eps)
    out.update({"recompute." + k: getattr(lr, k) for k in lr._fields})
    pp = B.mhc_post_pre(x, y, gates["H_post_l"], gates["H_res_l"], phi, b, alpha, w.iters, w.eps)
    out.update({"post_pre." + k: getattr(pp, k) for k in pp._fields})
    flags = B.SANDWICH_NORM | B.BLOCK_NORM
    pn = B.mhc_post_norm(x, y, f.H_post, f.H_res, flags, w.eps)
    out.update({"post_norm." + k: getattr(pn, k) for k in pn._fields})
    pnb = B.mhc_post_norm_bwd(inp["g_next"], x, y, f.H_post, f.H_res, flags, pn.inv_rms_y,
                              pn.inv_rms_out, w.eps)
    out.update({"post_norm_bwd." + k: getattr(pnb, k) for k in pnb._fields})
    torch.cuda.synchronize()
    assert B.get_last_device_error() == B.MHC_OK
    return out


@pytest.mark.parametrize("T,D,dtype", [
    (129, 5120, "bf16"), (333, 2560, "bf16"),   # ragged last tiles, tensor-core kernels
    (1, 5120, "bf16"), (63, 2560, "bf16"),      # batches below one tile
    (65, 40, "bf16"), (67, 12, "f32"),          # CUDA-core fallbacks
])
def test_outputs_stay_inside_their_buffers(T, D, dtype, monkeypatch):
    dev = _dev()
    w = W.WORKLOADS[4].with_(T=T, D=D, dtype=dtype, wid=70 + T % 20)
    inp = W.make_inputs(w, device=dev)
    gates = W.make_layer_gates(w, device=dev)
    plain = _layer(inp, gates, w, dtype == "f32")
    guarded = GuardedAllocator()
    monkeypatch.setattr(B, "_empty", guarded)
    got = _layer(inp, gates, w, dtype == "f32")
    monkeypatch.undo()
    guarded.check(f"T={T} D={D} {dtype}")
    assert len(guarded.bufs) > 30
    for k, v in plain.items():
        assert torch.equal(got[k], v), k
