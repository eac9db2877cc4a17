"""Seeded synthetic inputs for the mHC layer workloads.

This module only draws random numbers and casts them to the activation dtype;
it holds none of the layer's arithmetic.  It is the one piece shared by the
tests, the benchmark and the float64 oracle's callers.

Shapes follow the pages: n = 4 residual streams and 20 Sinkhorn rounds
(openPangu 2.0 notes, model table in section 01), hidden sizes D = 5120 (Pro)
and 2560 (Flash) (same table), and the operator shapes B=1, S=1024, D=5120 and
B=1, S=2048, D=2560 of the Ascend mHC Triton operator article (paragraph on
the 5.5x comparison), plus B=1, S=4096, D=5120 from its activation-memory
paragraph.  Draw order per workload: x, y, phi, b, g_in, g_next, each from
N(0, std) in float32, with a generator seeded 1000 + workload id.
"""

from __future__ import annotations

from dataclasses import dataclass, replace

import torch

N_STREAMS = 4


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    T: int
    D: int
    dtype: str            # "f32" or "bf16": activations x, y, x_in, x_next, grads
    iters: int = 20
    alpha: float = 0.01   # the same scale for the pre, post and res groups
    b_std: float = 0.1
    phi_std: float = 0.02
    eps: float = 1e-6
    backward: bool = False
    n: int = N_STREAMS

    @property
    def K(self) -> int:
        return self.n * self.D

    @property
    def G(self) -> int:
        return 2 * self.n + self.n * self.n

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    1: Workload(1, "tiny fp32 forward T=64 D=256", T=64, D=256, dtype="f32"),
    2: Workload(2, "bf16 forward B=1 S=1024 D=5120", T=1024, D=5120,
                dtype="bf16"),
    3: Workload(3, "bf16 forward B=1 S=2048 D=2560 (Flash width)", T=2048,
                D=2560, dtype="bf16"),
    4: Workload(4, "bf16 forward+backward B=1 S=4096 D=5120", T=4096, D=5120,
                dtype="bf16", backward=True),
    # logits x10: alpha 0.1 instead of 0.01 and b ~ N(0, 1) instead of N(0, 0.1)
    5: Workload(5, "bf16 large batch B=8 S=4096 D=5120, logits x10", T=32768,
                D=5120, dtype="bf16", alpha=0.1, b_std=1.0, backward=True),
}

SINKHORN_SWEEP = (5, 20, 50)


def torch_dtype(w: Workload):
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def make_inputs(w: Workload, device="cpu", seed=None):
    """Draw the inputs of workload ``w`` on ``device`` (a torch device).

    Returns a dict of tensors: x [T, n, D], y [T, D] (activation dtype),
    phi [n*D, G], b [G], alpha [3] (float32), and, for workloads with a
    backward, g_in [T, D] and g_next [T, n, D] (activation dtype).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + w.wid if seed is None else seed)
    act = torch_dtype(w)

    def draw(shape, std):
        return torch.randn(shape, generator=gen, device=device,
                           dtype=torch.float32).mul_(std)

    out = {}
    out["x"] = draw((w.T, w.n, w.D), 1.0).to(act)
    out["y"] = draw((w.T, w.D), 1.0).to(act)
    out["phi"] = draw((w.K, w.G), w.phi_std)
    out["b"] = draw((w.G,), w.b_std)
    out["alpha"] = torch.full((3,), w.alpha, dtype=torch.float32,
                              device=device)
    if w.backward:
        out["g_in"] = draw((w.T, w.D), 1.0).to(act)
        out["g_next"] = draw((w.T, w.n, w.D), 1.0).to(act)
    return out


def make_layer_gates(w: Workload, device="cpu", seed=None):
    """Gates of a previous layer for the cross-layer step: H_post [T, n] and
    H_res [T, n, n] (float32), uniform on (0, 2) and (0, 1/2).  Plain random
    numbers (the step only combines them linearly); their own generator,
    seeded 2000 + workload id, so the other inputs stay as they are.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(2000 + w.wid if seed is None else seed)
    H_post = torch.rand((w.T, w.n), generator=gen, device=device, dtype=torch.float32).mul_(2.0)
    H_res = torch.rand((w.T, w.n, w.n), generator=gen, device=device, dtype=torch.float32).mul_(0.5)
    return {"H_post_l": H_post, "H_res_l": H_res}
