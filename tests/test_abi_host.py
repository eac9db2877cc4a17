"""Host-side checks of the C-ABI library: it loads, exports every function
``include/mhc.h`` declares, and rejects bad arguments before any launch.

No call here reaches the GPU: every argument set is refused by host
validation, which runs before any CUDA call, or is a T = 0 call that launches
nothing and writes nothing.  (For T = 0 the backward entry points write zero
parameter gradients; with fake addresses those calls are only checked for
their refusals here, and tests/test_gpu_parity.py checks the zeros on a GPU.)
"""

import os
import re

import pytest

from mhc_pre_gb300 import binding as B
from mhc_pre_gb300 import build as mbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mhc.h")

# fake, never dereferenced device addresses
A = 0x7F0000000000          # 16-byte aligned
MIS = A + 8                 # misaligned


@pytest.fixture(scope="module")
def L():
    mbuild.build()
    return B.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mhc_\w+)\s*\(", src)))


def test_header_declares_the_four_ops():
    names = _declared()
    for op in ("mhc_pre", "mhc_post", "mhc_post_bwd", "mhc_pre_bwd"):
        assert op in names


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert set(names) == set(B.EXPORTS), "binding and header disagree"
    for name in names:
        assert hasattr(L, name), name


def test_version_and_status_strings(L):
    assert "sm_103a" in B.version()
    for code in range(6):
        s = B.status_string(code)
        assert s.startswith("MHC_")
    assert B.status_string(99) == "MHC_ERR_UNKNOWN"


def _pre(L, dt=B.MHC_BF16, x=A, T=8, n=4, D=64, iters=20, eps=1e-6, outs=None):
    outs = outs or [A] * 6
    return L.mhc_pre(dt, x, A, A, A, T, n, D, iters, eps, *outs, None)


def test_pre_validation(L):
    assert _pre(L, n=3) == B.MHC_ERR_UNSUPPORTED
    assert _pre(L, D=60) == B.MHC_ERR_UNSUPPORTED        # bf16 needs D % 8
    assert _pre(L, dt=B.MHC_F32, D=62) == B.MHC_ERR_UNSUPPORTED
    assert _pre(L, dt=7) == B.MHC_ERR_INVALID_ARG
    assert _pre(L, T=-1) == B.MHC_ERR_INVALID_ARG
    assert _pre(L, D=0) == B.MHC_ERR_INVALID_ARG
    assert _pre(L, x=None) == B.MHC_ERR_INVALID_ARG
    assert _pre(L, x=MIS) == B.MHC_ERR_MISALIGNED
    assert _pre(L, outs=[A, A, A, MIS, A, A]) == B.MHC_ERR_MISALIGNED
    assert _pre(L, iters=0) == B.MHC_ERR_INVALID_ARG
    assert _pre(L, iters=B.MAX_ITERS + 1) == B.MHC_ERR_UNSUPPORTED
    assert _pre(L, eps=-1.0) == B.MHC_ERR_INVALID_ARG
    assert _pre(L, eps=float("nan")) == B.MHC_ERR_INVALID_ARG
    # T = 0 is a no-op that touches nothing, even with null pointers
    assert L.mhc_pre(B.MHC_BF16, None, None, None, None, 0, 4, 64, 20, 1e-6,
                     None, None, None, None, None, None, None) == B.MHC_OK


def _post_pre(L, dt=B.MHC_BF16, x=A, T=8, n=4, D=64, iters=20, eps=1e-6, outs=None, ws=A, nws=4096):
    outs = outs or [A] * 7
    return L.mhc_post_pre(dt, x, A, A, A, A, A, A, T, n, D, iters, eps, *outs, ws, nws, None)


def test_post_pre_validation(L):
    assert _post_pre(L, n=3) == B.MHC_ERR_UNSUPPORTED
    assert _post_pre(L, D=60) == B.MHC_ERR_UNSUPPORTED
    assert _post_pre(L, dt=7) == B.MHC_ERR_INVALID_ARG
    assert _post_pre(L, T=-1) == B.MHC_ERR_INVALID_ARG
    assert _post_pre(L, x=None) == B.MHC_ERR_INVALID_ARG
    assert _post_pre(L, x=MIS) == B.MHC_ERR_MISALIGNED
    assert _post_pre(L, outs=[A, A, A, A, MIS, A, A]) == B.MHC_ERR_MISALIGNED
    assert _post_pre(L, iters=0) == B.MHC_ERR_INVALID_ARG
    assert _post_pre(L, iters=B.MAX_ITERS + 1) == B.MHC_ERR_UNSUPPORTED
    assert _post_pre(L, eps=float("nan")) == B.MHC_ERR_INVALID_ARG
    # T = 0 is a no-op that touches nothing, even with null pointers
    assert L.mhc_post_pre(B.MHC_BF16, *([None] * 7), 0, 4, 64, 20, 1e-6, *([None] * 7),
                          None, 0, None) == B.MHC_OK
    # shapes the fused kernel never takes need no workspace
    assert L.mhc_post_pre_workspace_bytes(B.MHC_F32, 64, 4, 256) == 0
    assert L.mhc_post_pre_workspace_bytes(B.MHC_BF16, 0, 4, 5120) == 0
    assert L.mhc_post_pre_workspace_bytes(B.MHC_BF16, 64, 4, 60) == 0


def test_post_and_post_bwd_validation(L):
    assert L.mhc_post(B.MHC_BF16, A, A, A, A, 4, 2, 64, A, None) == B.MHC_ERR_UNSUPPORTED
    assert L.mhc_post(B.MHC_BF16, A, None, A, A, 4, 4, 64, A, None) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_post(B.MHC_BF16, A, A, A, A, 4, 4, 64, MIS, None) == B.MHC_ERR_MISALIGNED
    assert L.mhc_post(B.MHC_F32, None, None, None, None, 0, 4, 64, None, None) == B.MHC_OK
    args = [A] * 5
    assert L.mhc_post_bwd(B.MHC_BF16, *args, 4, 4, 12, A, A, A, A, None) == B.MHC_ERR_UNSUPPORTED
    assert L.mhc_post_bwd(B.MHC_BF16, *args, 4, 4, 64, A, None, A, A, None) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_post_bwd(B.MHC_BF16, *args, 0, 4, 64, None, None, None, None, None) == B.MHC_OK


def test_pre_bwd_workspace_and_validation(L):
    ws = L.mhc_pre_bwd_workspace_bytes(B.MHC_BF16, 4096, 4, 5120)
    # per-token records (256 B) plus at least one dphi partial (K x 24 fp32)
    assert ws >= 4096 * 256 + 4 * 5120 * 24 * 4
    assert ws % 16 == 0
    assert L.mhc_pre_bwd_workspace_bytes(B.MHC_BF16, 0, 4, 5120) == 0
    assert L.mhc_pre_bwd_workspace_bytes(B.MHC_BF16, 16, 3, 5120) == 0

    def call(T=16, n=4, D=64, iters=20, ws_ptr=A, ws_bytes=None, dx=A, dphi=A):
        need = L.mhc_pre_bwd_workspace_bytes(B.MHC_BF16, max(T, 0), 4, D)
        wb = need if ws_bytes is None else ws_bytes
        return L.mhc_pre_bwd(B.MHC_BF16, A, A, A, A, A, A, A, A, A, T, n, D, iters,
                             dx, dphi, A, A, ws_ptr, wb, None)

    assert call(n=5) == B.MHC_ERR_UNSUPPORTED
    assert call(iters=0) == B.MHC_ERR_INVALID_ARG
    assert call(iters=B.MAX_ITERS + 1) == B.MHC_ERR_UNSUPPORTED
    assert call(ws_ptr=None) == B.MHC_ERR_INVALID_ARG
    assert call(dx=MIS) == B.MHC_ERR_MISALIGNED
    need = L.mhc_pre_bwd_workspace_bytes(B.MHC_BF16, 16, 4, 64)
    assert call(ws_bytes=need - 16) == B.MHC_ERR_INVALID_ARG
    # T = 0 writes zero parameter gradients: their pointers must be valid
    assert call(T=0, ws_ptr=None, ws_bytes=0, dx=None, dphi=None) == B.MHC_ERR_INVALID_ARG
    assert call(T=0, ws_ptr=None, ws_bytes=0, dx=None, dphi=MIS) == B.MHC_ERR_MISALIGNED


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((2, 4, 8), dtype=torch.bfloat16)
    phi = torch.zeros((32, 24))
    with pytest.raises(ValueError):
        B.mhc_pre(x, phi, torch.zeros(24), torch.zeros(3))


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU path"):
        B.lib(str(tmp_path / "absent.so"))


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    # 16 MiB of scratch: T * 256 B of records, one 4*D x 24 float partial and
    # D * 256 B of bf16 phi blocks must fit; the refusal comes before any CUDA call.
    args = [A] * 9

    def call(T, D):
        return L.mhc_pre_bwd_noalloc(B.MHC_BF16, *args, T, 4, D, 20, A, A, A, A, None)

    assert call(60000, 5120) == B.MHC_ERR_UNSUPPORTED
    assert call(1 << 20, 64) == B.MHC_ERR_UNSUPPORTED
    # T = 0 writes zero parameter gradients: their pointers must be valid
    assert L.mhc_pre_bwd_noalloc(B.MHC_BF16, *args, 0, 4, 5120, 20, None, None, A, A,
                                 None) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_pre_bwd_noalloc(B.MHC_BF16, *args, 0, 4, 5120, 20, None, A, MIS, A,
                                 None) == B.MHC_ERR_MISALIGNED
    assert L.mhc_pre_bwd_noalloc(B.MHC_BF16, *args, 16, 4, 64, 0, A, A, A, A,
                                 None) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_pre_bwd_noalloc(B.MHC_BF16, *args, 16, 4, 64, 20, MIS, A, A, A,
                                 None) == B.MHC_ERR_MISALIGNED


def test_pre_gates_validation(L):
    def call(dt=B.MHC_BF16, x=A, T=8, n=4, D=64, iters=20, eps=1e-6, outs=None):
        outs = outs or [A] * 5
        return L.mhc_pre_gates(dt, x, A, A, A, T, n, D, iters, eps, *outs, None)

    assert call(n=3) == B.MHC_ERR_UNSUPPORTED
    assert call(D=60) == B.MHC_ERR_UNSUPPORTED
    assert call(dt=7) == B.MHC_ERR_INVALID_ARG
    assert call(x=None) == B.MHC_ERR_INVALID_ARG
    assert call(outs=[A, A, A, MIS, A]) == B.MHC_ERR_MISALIGNED
    assert call(iters=0) == B.MHC_ERR_INVALID_ARG
    assert call(eps=float("inf")) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_pre_gates(B.MHC_BF16, *([None] * 4), 0, 4, 64, 20, 1e-6, *([None] * 5), None) == B.MHC_OK
    assert L.mhc_kernel_launches(b"mhc_pre_gates", B.MHC_BF16, 8, 4, 64) == 1
    assert L.mhc_kernel_launches(b"mhc_layer_bwd_recompute", B.MHC_F32, 8, 4, 64) == 7


def test_layer_bwd_recompute_workspace_and_validation(L):
    T, D = 4096, 5120
    ws = L.mhc_layer_bwd_recompute_workspace_bytes(B.MHC_BF16, T, 4, D)
    # recomputed gates and saved state (196 B per token) and the gate
    # gradients (80 B per token) before the pre backward's own scratch
    assert ws >= T * (196 + 80) + L.mhc_pre_bwd_workspace_bytes(B.MHC_BF16, T, 4, D)
    assert ws % 16 == 0
    assert L.mhc_layer_bwd_recompute_workspace_bytes(B.MHC_BF16, 0, 4, D) == 0
    assert L.mhc_layer_bwd_recompute_workspace_bytes(B.MHC_BF16, T, 3, D) == 0

    def call(T=16, n=4, D=64, iters=20, ws_ptr=A, ws_bytes=None, dx=A, dphi=A):
        need = L.mhc_layer_bwd_recompute_workspace_bytes(B.MHC_BF16, max(T, 0), 4, D)
        nb = need if ws_bytes is None else ws_bytes
        return L.mhc_layer_bwd_recompute(B.MHC_BF16, A, A, A, A, A, A, A, T, n, D, iters, 1e-6,
                                         dx, A, dphi, A, A, ws_ptr, nb, None)

    assert call(n=5) == B.MHC_ERR_UNSUPPORTED
    assert call(ws_ptr=None) == B.MHC_ERR_INVALID_ARG
    assert call(ws_bytes=1024) == B.MHC_ERR_INVALID_ARG
    assert call(ws_ptr=MIS) == B.MHC_ERR_MISALIGNED
    assert call(dx=None) == B.MHC_ERR_INVALID_ARG
    assert call(iters=B.MAX_ITERS + 1) == B.MHC_ERR_UNSUPPORTED
    assert call(T=0, ws_ptr=None, dx=None, dphi=None) == B.MHC_ERR_INVALID_ARG
    assert call(T=0, ws_ptr=None, dx=None, dphi=MIS) == B.MHC_ERR_MISALIGNED


def test_critical_path_validation(L):
    def crit(dt=B.MHC_BF16, x=A, T=8, n=4, D=64, eps=1e-6, outs=None):
        outs = outs or [A] * 4
        return L.mhc_pre_critical(dt, x, A, A, A, T, n, D, eps, *outs, None)

    assert crit(n=3) == B.MHC_ERR_UNSUPPORTED
    assert crit(D=60) == B.MHC_ERR_UNSUPPORTED
    assert crit(x=None) == B.MHC_ERR_INVALID_ARG
    assert crit(outs=[A, MIS, A, A]) == B.MHC_ERR_MISALIGNED
    assert crit(eps=float("nan")) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_pre_critical(B.MHC_BF16, *([None] * 4), 0, 4, 64, 1e-6, *([None] * 4), None) == B.MHC_OK

    def side(T=8, n=4, iters=20, proj=A, outs=None):
        outs = outs or [A, A]
        return L.mhc_post_res_gates(proj, A, A, T, n, iters, *outs, None)

    assert side(n=2) == B.MHC_ERR_UNSUPPORTED
    assert side(iters=0) == B.MHC_ERR_INVALID_ARG
    assert side(iters=B.MAX_ITERS + 1) == B.MHC_ERR_UNSUPPORTED
    assert side(proj=None) == B.MHC_ERR_INVALID_ARG
    assert side(outs=[A, MIS]) == B.MHC_ERR_MISALIGNED
    assert side(T=-1) == B.MHC_ERR_INVALID_ARG
    assert L.mhc_post_res_gates(None, None, None, 0, 4, 20, None, None, None) == B.MHC_OK
