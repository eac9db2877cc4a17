"""Thin ctypes binding of libmhc_gb300.so (argument marshalling only).

Each function takes CUDA tensors, allocates the outputs with torch (device
memory is PyTorch's job here), and calls the C entry point of the same name on
the current torch stream.  Every step of the layer runs in the library's CUDA
kernels; there is no CPU path.  If the library is missing, the first call
raises: build it with ``python -m mhc_pre_gb300.build`` (or
``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os
from collections import namedtuple

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libmhc_gb300.so")

MHC_OK, MHC_ERR_INVALID_ARG, MHC_ERR_UNSUPPORTED = 0, 1, 2
MHC_ERR_MISALIGNED, MHC_ERR_CUDA, MHC_ERR_TIMEOUT = 3, 4, 5
MHC_F32, MHC_BF16 = 0, 1
MAX_ITERS = 64

EXPORTS = ("mhc_status_string", "mhc_version", "mhc_get_last_device_error",
           "mhc_pre", "mhc_post", "mhc_post_norm", "mhc_post_norm_bwd",
           "mhc_post_pre", "mhc_post_pre_workspace_bytes",
           "mhc_post_bwd", "mhc_kernel_launches",
           "mhc_pre_bwd_workspace_bytes", "mhc_pre_bwd", "mhc_pre_bwd_noalloc",
           "mhc_pre_gates", "mhc_layer_bwd_recompute_workspace_bytes",
           "mhc_layer_bwd_recompute", "mhc_test_force_timeout", "mhc_pre_critical",
           "mhc_post_res_gates")

PreOut = namedtuple("PreOut", "x_in H_pre H_post H_res proj inv_rms")
PostPreOut = namedtuple("PostPreOut", "x_next x_in H_pre H_post H_res proj inv_rms")
PostNormOut = namedtuple("PostNormOut", "x_next inv_rms_y inv_rms_out")
SANDWICH_NORM, BLOCK_NORM = 1, 2
PostBwdOut = namedtuple("PostBwdOut", "dx dy dH_post dH_res")
PreBwdOut = namedtuple("PreBwdOut", "dx dphi db dalpha")
PreGatesOut = namedtuple("PreGatesOut", "H_pre H_post H_res proj inv_rms")
PreCriticalOut = namedtuple("PreCriticalOut", "x_in H_pre proj inv_rms")
PostResGatesOut = namedtuple("PostResGatesOut", "H_post H_res")
LayerBwdOut = namedtuple("LayerBwdOut", "dx dy dphi db dalpha")

_P, _I64, _I, _F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
_SIGS = {
    "mhc_status_string": ([_I], ctypes.c_char_p),
    "mhc_version": ([], ctypes.c_char_p),
    "mhc_get_last_device_error": ([_P], _I),
    "mhc_pre": ([_I, _P, _P, _P, _P, _I64, _I, _I64, _I, _F,
                 _P, _P, _P, _P, _P, _P, _P], _I),
    "mhc_post": ([_I, _P, _P, _P, _P, _I64, _I, _I64, _P, _P], _I),
    "mhc_post_pre": ([_I, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _I, _F,
                      _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
    "mhc_post_pre_workspace_bytes": ([_I, _I64, _I, _I64], ctypes.c_size_t),
    "mhc_post_norm": ([_I, _P, _P, _P, _P, _I, _F, _I64, _I, _I64, _P, _P, _P, _P], _I),
    "mhc_post_norm_bwd": ([_I, _P, _P, _P, _P, _P, _I, _F, _P, _P, _I64, _I, _I64,
                           _P, _P, _P, _P, _P], _I),
    "mhc_post_bwd": ([_I, _P, _P, _P, _P, _P, _I64, _I, _I64,
                      _P, _P, _P, _P, _P], _I),
    "mhc_kernel_launches": ([ctypes.c_char_p, _I, _I64, _I, _I64], _I),
    "mhc_pre_bwd_workspace_bytes": ([_I, _I64, _I, _I64], ctypes.c_size_t),
    "mhc_pre_bwd": ([_I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64,
                     _I, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
    "mhc_pre_bwd_noalloc": ([_I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I,
                             _I64, _I, _P, _P, _P, _P, _P], _I),
    "mhc_pre_gates": ([_I, _P, _P, _P, _P, _I64, _I, _I64, _I, _F,
                       _P, _P, _P, _P, _P, _P], _I),
    "mhc_layer_bwd_recompute_workspace_bytes": ([_I, _I64, _I, _I64], ctypes.c_size_t),
    "mhc_test_force_timeout": ([_I], _I),
    "mhc_pre_critical": ([_I, _P, _P, _P, _P, _I64, _I, _I64, _F, _P, _P, _P, _P, _P], _I),
    "mhc_post_res_gates": ([_P, _P, _P, _I64, _I, _I, _P, _P, _P], _I),
    "mhc_layer_bwd_recompute": ([_I, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _I, _F,
                                 _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P], _I),
}

_lib = None


def _empty(shape, dtype=None, device=None):
    """Allocates every output and workspace buffer this module hands to the
    library.  Plain torch.empty; the guard-band tests put an allocator that
    surrounds each buffer with sentinel bytes in its place."""
    return torch.empty(shape, dtype=dtype, device=device)


class MhcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the library once and declares every exported signature."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: the mHC layer has no CPU path; build the "
            "CUDA library with `python -m mhc_pre_gb300.build`")
    handle = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(handle, name)
        fn.argtypes = args
        fn.restype = res
    if path == LIB_PATH:
        _lib = handle
    return handle


def status_string(status: int) -> str:
    return lib().mhc_status_string(status).decode()


def version() -> str:
    return lib().mhc_version().decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MHC_BF16
    if t.dtype == torch.float32:
        return MHC_F32
    raise TypeError(f"activations must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("the mHC library takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("the mHC library takes contiguous tensors only")
    return t.data_ptr()


def _stream(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _check(status: int, where: str):
    if status != MHC_OK:
        raise MhcError(status, where)


def _f32(t: torch.Tensor, name: str) -> torch.Tensor:
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return t


def mhc_pre(x, phi, b, alpha, iters: int = 20, eps: float = 1e-6):
    """Forward of the read side.  x [T, n, D] (bf16 or f32, CUDA)."""
    T, n, D = x.shape
    G = 2 * n + n * n
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PreOut(_empty((T, D), dtype=x.dtype, device=x.device),
                 _empty((T, n), **f32), _empty((T, n), **f32),
                 _empty((T, n, n), **f32), _empty((T, G), **f32),
                 _empty((T,), **f32))
    st = lib().mhc_pre(_dtype_code(x), _ptr(x), _ptr(_f32(phi, "phi")),
                       _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")), T, n, D,
                       iters, eps, *[_ptr(o) for o in out], _stream(x.device))
    _check(st, "mhc_pre")
    return out


def mhc_pre_gates(x, phi, b, alpha, iters: int = 20, eps: float = 1e-6):
    """mhc_pre without the H_pre mix (no x_in): the gates and the saved state,
    bit for bit as mhc_pre writes them."""
    T, n, D = x.shape
    G = 2 * n + n * n
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PreGatesOut(_empty((T, n), **f32), _empty((T, n), **f32),
                      _empty((T, n, n), **f32), _empty((T, G), **f32),
                      _empty((T,), **f32))
    st = lib().mhc_pre_gates(_dtype_code(x), _ptr(x), _ptr(_f32(phi, "phi")),
                             _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")), T, n, D,
                             iters, eps, *[_ptr(o) for o in out], _stream(x.device))
    _check(st, "mhc_pre_gates")
    return out


def layer_bwd_recompute_workspace_bytes(dtype, T: int, n: int, D: int) -> int:
    code = MHC_BF16 if dtype == torch.bfloat16 else MHC_F32
    return int(lib().mhc_layer_bwd_recompute_workspace_bytes(code, T, n, D))


def mhc_pre_critical(x, phi, b, alpha, eps: float = 1e-6, stream=None):
    """The inference critical path of mhc_pre: x_in, H_pre, proj, inv_rms (no
    Sinkhorn).  ``stream``: a torch.cuda.Stream (default: the current one)."""
    T, n, D = x.shape
    G = 2 * n + n * n
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PreCriticalOut(_empty((T, D), dtype=x.dtype, device=x.device), _empty((T, n), **f32),
                         _empty((T, G), **f32), _empty((T,), **f32))
    s = stream.cuda_stream if stream is not None else _stream(x.device)
    st = lib().mhc_pre_critical(_dtype_code(x), _ptr(x), _ptr(_f32(phi, "phi")), _ptr(_f32(b, "b")),
                                _ptr(_f32(alpha, "alpha")), T, n, D, eps, *[_ptr(o) for o in out], s)
    _check(st, "mhc_pre_critical")
    return out


def mhc_post_res_gates(proj, b, alpha, iters: int = 20, stream=None):
    """H_post and H_res from a saved projection (the side of the critical-path
    split).  ``stream``: a torch.cuda.Stream (default: the current one)."""
    T, G = proj.shape
    n = 4
    f32 = dict(dtype=torch.float32, device=proj.device)
    out = PostResGatesOut(_empty((T, n), **f32), _empty((T, n, n), **f32))
    s = stream.cuda_stream if stream is not None else _stream(proj.device)
    st = lib().mhc_post_res_gates(_ptr(_f32(proj, "proj")), _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")),
                                  T, n, iters, *[_ptr(o) for o in out], s)
    _check(st, "mhc_post_res_gates")
    return out


def mhc_layer_bwd_recompute(g_in, g_next, x, y, phi, b, alpha, iters: int = 20,
                            eps: float = 1e-6, workspace=None):
    """The layer's backward from its inputs x and y alone (the gates and the
    saved state recomputed).  Returns dx, dy, dphi, db, dalpha."""
    T, n, D = x.shape
    G = 2 * n + n * n
    if not (g_in.dtype == g_next.dtype == x.dtype == y.dtype):
        raise TypeError("g_in, g_next, x and y must share a dtype")
    need = layer_bwd_recompute_workspace_bytes(x.dtype, T, n, D)
    if workspace is None:
        workspace = _empty((max(need, 16),), dtype=torch.uint8, device=x.device)
    f32 = dict(dtype=torch.float32, device=x.device)
    dx = _empty(x.shape, x.dtype, x.device)
    dy = _empty(y.shape, y.dtype, y.device)
    dphi = _empty((n * D, G), **f32)
    db = _empty((G,), **f32)
    dalpha = _empty((3,), **f32)
    st = lib().mhc_layer_bwd_recompute(
        _dtype_code(x), _ptr(g_in), _ptr(g_next), _ptr(x), _ptr(y), _ptr(_f32(phi, "phi")),
        _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")), T, n, D, iters, eps, _ptr(dx), _ptr(dy),
        _ptr(dphi), _ptr(db), _ptr(dalpha), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(x.device))
    _check(st, "mhc_layer_bwd_recompute")
    return LayerBwdOut(dx, dy, dphi, db, dalpha)


def mhc_post_pre(x, y, H_post_l, H_res_l, phi, b, alpha, iters: int = 20,
                 eps: float = 1e-6):
    """mhc_post of layer l, then mhc_pre of layer l + 1 on the stored x_next."""
    T, n, D = x.shape
    G = 2 * n + n * n
    if y.dtype != x.dtype:
        raise TypeError("x and y must share a dtype")
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PostPreOut(_empty(x.shape, x.dtype, x.device),
                     _empty((T, D), dtype=x.dtype, device=x.device),
                     _empty((T, n), **f32), _empty((T, n), **f32),
                     _empty((T, n, n), **f32), _empty((T, G), **f32),
                     _empty((T,), **f32))
    nws = int(lib().mhc_post_pre_workspace_bytes(_dtype_code(x), T, n, D))
    ws = _empty((max(nws, 1),), dtype=torch.uint8, device=x.device)
    st = lib().mhc_post_pre(_dtype_code(x), _ptr(x), _ptr(y), _ptr(_f32(H_post_l, "H_post_l")),
                            _ptr(_f32(H_res_l, "H_res_l")), _ptr(_f32(phi, "phi")),
                            _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")), T, n, D, iters, eps,
                            *[_ptr(o) for o in out], _ptr(ws), nws, _stream(x.device))
    _check(st, "mhc_post_pre")
    return out


def mhc_post_norm(x, y, H_post, H_res, flags: int, eps: float = 1e-6):
    """mhc_post with the sandwich (flag 1) and block (flag 2) normalisations."""
    T, n, D = x.shape
    if y.dtype != x.dtype:
        raise TypeError("x and y must share a dtype")
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PostNormOut(_empty(x.shape, x.dtype, x.device), _empty((T,), **f32), _empty((T,), **f32))
    st = lib().mhc_post_norm(_dtype_code(x), _ptr(x), _ptr(y), _ptr(_f32(H_post, "H_post")),
                             _ptr(_f32(H_res, "H_res")), flags, eps, T, n, D, *[_ptr(o) for o in out],
                             _stream(x.device))
    _check(st, "mhc_post_norm")
    return out


def mhc_post_norm_bwd(g_next, x, y, H_post, H_res, flags: int, inv_rms_y, inv_rms_out,
                      eps: float = 1e-6):
    """Gradients of <g_next, x_next> for mhc_post_norm: (dx, dy, dH_post, dH_res)."""
    T, n, D = x.shape
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PostBwdOut(_empty(x.shape, x.dtype, x.device), _empty(y.shape, y.dtype, y.device),
                     _empty((T, n), **f32), _empty((T, n, n), **f32))
    st = lib().mhc_post_norm_bwd(_dtype_code(x), _ptr(g_next), _ptr(x), _ptr(y),
                                 _ptr(_f32(H_post, "H_post")), _ptr(_f32(H_res, "H_res")), flags, eps,
                                 _ptr(_f32(inv_rms_y, "inv_rms_y")), _ptr(_f32(inv_rms_out, "inv_rms_out")),
                                 T, n, D, *[_ptr(o) for o in out], _stream(x.device))
    _check(st, "mhc_post_norm_bwd")
    return out


def mhc_post(x, y, H_post, H_res):
    """x_next [T, n, D] = H_res x + H_post (x) y."""
    T, n, D = x.shape
    if y.dtype != x.dtype:
        raise TypeError("x and y must share a dtype")
    x_next = _empty(x.shape, x.dtype, x.device)
    st = lib().mhc_post(_dtype_code(x), _ptr(x), _ptr(y), _ptr(_f32(H_post, "H_post")),
                        _ptr(_f32(H_res, "H_res")), T, n, D, _ptr(x_next),
                        _stream(x.device))
    _check(st, "mhc_post")
    return x_next


def mhc_post_bwd(g_next, x, y, H_post, H_res):
    """Gradients of <g_next, x_next>: (dx, dy, dH_post, dH_res)."""
    T, n, D = x.shape
    if not (g_next.dtype == x.dtype == y.dtype):
        raise TypeError("g_next, x and y must share a dtype")
    f32 = dict(dtype=torch.float32, device=x.device)
    out = PostBwdOut(_empty(x.shape, x.dtype, x.device), _empty(y.shape, y.dtype, y.device),
                     _empty((T, n), **f32), _empty((T, n, n), **f32))
    st = lib().mhc_post_bwd(_dtype_code(x), _ptr(g_next), _ptr(x), _ptr(y),
                            _ptr(_f32(H_post, "H_post")), _ptr(_f32(H_res, "H_res")),
                            T, n, D, *[_ptr(o) for o in out], _stream(x.device))
    _check(st, "mhc_post_bwd")
    return out


def kernel_launches(op: str, dtype, T: int, n: int, D: int) -> int:
    """Kernels the entry point ``op`` launches for these sizes."""
    code = MHC_BF16 if dtype in (torch.bfloat16, "bf16") else MHC_F32
    return int(lib().mhc_kernel_launches(op.encode(), code, T, n, D))


def pre_bwd_workspace_bytes(dtype, T: int, n: int, D: int) -> int:
    code = MHC_BF16 if dtype == torch.bfloat16 else MHC_F32
    return int(lib().mhc_pre_bwd_workspace_bytes(code, T, n, D))


def mhc_pre_bwd(g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms, dx,
                iters: int = 20, workspace=None):
    """Backward of mhc_pre.  ``dx`` is accumulated in place (dx += pre part)."""
    T, n, D = x.shape
    G = 2 * n + n * n
    if not (g_in.dtype == x.dtype == dx.dtype):
        raise TypeError("g_in, x and dx must share a dtype")
    need = pre_bwd_workspace_bytes(x.dtype, T, n, D)
    if workspace is None:
        workspace = _empty((max(need, 16),), dtype=torch.uint8, device=x.device)
    f32 = dict(dtype=torch.float32, device=x.device)
    dphi = _empty((n * D, G), **f32)
    db = _empty((G,), **f32)
    dalpha = _empty((3,), **f32)
    st = lib().mhc_pre_bwd(_dtype_code(x), _ptr(g_in), _ptr(_f32(dH_post, "dH_post")),
                           _ptr(_f32(dH_res, "dH_res")), _ptr(x), _ptr(_f32(phi, "phi")),
                           _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")),
                           _ptr(_f32(proj, "proj")), _ptr(_f32(inv_rms, "inv_rms")),
                           T, n, D, iters, _ptr(dx), _ptr(dphi), _ptr(db), _ptr(dalpha),
                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(x.device))
    _check(st, "mhc_pre_bwd")
    return PreBwdOut(dx, dphi, db, dalpha)


def mhc_pre_bwd_noalloc(g_in, dH_post, dH_res, x, phi, b, alpha, proj, inv_rms,
                        dx, iters: int = 20):
    """mhc_pre_bwd with the library's fixed scratch array instead of a
    caller workspace (for callers that cannot allocate device memory).
    ``dx`` is accumulated in place; the outputs dphi, db, dalpha are allocated
    here by torch only because this binding returns new tensors."""
    T, n, D = x.shape
    G = 2 * n + n * n
    if not (g_in.dtype == x.dtype == dx.dtype):
        raise TypeError("g_in, x and dx must share a dtype")
    f32 = dict(dtype=torch.float32, device=x.device)
    dphi = _empty((n * D, G), **f32)
    db = _empty((G,), **f32)
    dalpha = _empty((3,), **f32)
    st = lib().mhc_pre_bwd_noalloc(
        _dtype_code(x), _ptr(g_in), _ptr(_f32(dH_post, "dH_post")), _ptr(_f32(dH_res, "dH_res")),
        _ptr(x), _ptr(_f32(phi, "phi")), _ptr(_f32(b, "b")), _ptr(_f32(alpha, "alpha")),
        _ptr(_f32(proj, "proj")), _ptr(_f32(inv_rms, "inv_rms")), T, n, D, iters, _ptr(dx),
        _ptr(dphi), _ptr(db), _ptr(dalpha), _stream(x.device))
    _check(st, "mhc_pre_bwd_noalloc")
    return PreBwdOut(dx, dphi, db, dalpha)


def get_last_device_error(device=None) -> int:
    """Synchronises the current stream and returns the device error status."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    return int(lib().mhc_get_last_device_error(_stream(dev)))
