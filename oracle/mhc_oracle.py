"""Plain float64 reference of the mHC layer, forward and backward.

Test infrastructure only: see the package docstring for who may import it.

Notation (openPangu 2.0 analysis notes, section 5.3):
    h_bar  : the n-stream residual state of one token, shape [n, D]
    x_bar  = RMSNorm(h_bar), taken over the flattened n*D row (K = n*D)
    [r_pre, r_post, r_res] = x_bar @ W_mHC        (G = 2n + n^2 logits)
    H_pre  = sigmoid(r_pre)         in (0, 1)     (n streams -> 1)
    H_post = 2 * sigmoid(r_post)    in (0, 2)     (1 stream  -> n)
    H_res  = Sinkhorn(reshape(r_res, n, n))       (n streams -> n)
The Ascend mHC Triton operator article adds that H_res is doubly stochastic
(non-negative, every row and column summing to 1) and that H_pre / H_post read
n streams into one and write one stream back to n.

Readings where the pages are silent:
  * W_mHC is called ``phi`` here, stored [K, G] with K index k = i*D + d
    (stream-major flattening of h_bar).
  * Each logit group has one scalar scale alpha and every logit a bias b:
    logits = alpha_group * (x_bar @ phi) + b, groups (pre, post, res).
  * RMSNorm has unit weight and eps inside the square root.
  * The res block is reshaped row-major: H_res[i, j] <- logit 2n + i*n + j.
  * One Sinkhorn iteration = normalise rows, then normalise columns, starting
    from exp(L); no epsilon in the denominators.
  * x_in = sum_i H_pre[i] * x[i];  x_next[i] = sum_j H_res[i, j] * x[j]
    + H_post[i] * y, where y is the sublayer output (an independent input).
  * The gradient through Sinkhorn is the exact reverse-mode derivative of the
    unrolled ``iters``-step map.

All arithmetic is float64 on whatever values the caller passes (the tests pass
the same bf16-quantised activations the GPU receives, widened to float64).
"""

from __future__ import annotations

import numpy as np

_F = np.float64


def _f64(a):
    return np.asarray(a, dtype=_F)


def group_of_logit(n: int) -> np.ndarray:
    """Group index (0 = pre, 1 = post, 2 = res) of each of the 2n + n^2 logits.

    Order [r_pre, r_post, r_res] as written in section 5.3 of the openPangu 2.0
    notes.
    """
    return np.array([0] * n + [1] * n + [2] * (n * n), dtype=np.int64)


def rmsnorm_flat(x, eps: float):
    """RMSNorm over the flattened n*D row, unit weight (section 5.3).

    x: [T, n, D].  Returns (x_bar [T, n, D], inv_rms [T]) with
    inv_rms = 1 / sqrt(mean(x^2) + eps).
    """
    x = _f64(x)
    T, n, D = x.shape
    flat = x.reshape(T, n * D)
    ms = np.mean(flat * flat, axis=1)
    inv_rms = 1.0 / np.sqrt(ms + eps)
    return x * inv_rms[:, None, None], inv_rms


def project(x_bar, phi):
    """Projection of the normalised row onto the G gate logits: x_bar @ phi.

    x_bar: [T, n, D]; phi: [n*D, G] (row k = i*D + d).  Returns [T, G].
    """
    x_bar = _f64(x_bar)
    T, n, D = x_bar.shape
    return x_bar.reshape(T, n * D) @ _f64(phi)


def logits_from_proj(proj, alpha, b, n: int):
    """logits = alpha_group * proj + b, groups [pre (n), post (n), res (n^2)]."""
    alpha = _f64(alpha)
    scale = alpha[group_of_logit(n)]
    return _f64(proj) * scale[None, :] + _f64(b)[None, :]


def _sigmoid(v):
    return 1.0 / (1.0 + np.exp(-v))


def gates(logits, n: int):
    """H_pre = sigmoid(r_pre), H_post = 2 sigmoid(r_post) (section 5.3)."""
    logits = _f64(logits)
    return _sigmoid(logits[:, :n]), 2.0 * _sigmoid(logits[:, n:2 * n])


def sinkhorn_iterates(L, iters: int):
    """All intermediate matrices of the Sinkhorn-Knopp map started at exp(L).

    L: [T, n, n].  Returns a list [M0, P1, M1, P2, M2, ..., P_iters, M_iters]
    where P_k = M_{k-1} with rows normalised and M_k = P_k with columns
    normalised.  M_iters is H_res.
    """
    M = np.exp(_f64(L))
    out = [M]
    for _ in range(iters):
        P = M / M.sum(axis=2, keepdims=True)
        M = P / P.sum(axis=1, keepdims=True)
        out.append(P)
        out.append(M)
    return out


def sinkhorn(L, iters: int):
    """H_res = Sinkhorn(exp(L)) after ``iters`` row-then-column rounds."""
    return sinkhorn_iterates(L, iters)[-1]


def sinkhorn_vjp(L, iters: int, dH):
    """Reverse-mode derivative of ``sinkhorn`` with respect to L.

    For Y = X / s with s = row sums of X:   dX = (dY - rowsum(dY * Y)) / s.
    For Y = X / c with c = column sums:     dX = (dY - colsum(dY * Y)) / c.
    For M0 = exp(L):                        dL = dM0 * M0.
    """
    its = sinkhorn_iterates(L, iters)
    g = _f64(dH)
    for k in range(iters, 0, -1):
        P, M = its[2 * k - 1], its[2 * k]
        c = P.sum(axis=1, keepdims=True)          # column sums of P
        g = (g - np.sum(g * M, axis=1, keepdims=True)) / c
        Mprev = its[2 * k - 2]
        s = Mprev.sum(axis=2, keepdims=True)      # row sums of M_{k-1}
        g = (g - np.sum(g * P, axis=2, keepdims=True)) / s
    return g * its[0]


def mhc_pre(x, phi, b, alpha, iters: int, eps: float):
    """Forward of the pre side of one mHC layer for T tokens.

    x: [T, n, D]; phi: [n*D, 2n+n^2]; b: [2n+n^2]; alpha: [3].
    Returns a dict with x_in [T, D], H_pre [T, n], H_post [T, n],
    H_res [T, n, n], proj [T, G] (x_bar @ phi), logits [T, G], inv_rms [T].
    """
    x = _f64(x)
    T, n, D = x.shape
    x_bar, inv_rms = rmsnorm_flat(x, eps)
    proj = project(x_bar, phi)
    logits = logits_from_proj(proj, alpha, b, n)
    H_pre, H_post = gates(logits, n)
    H_res = sinkhorn(logits[:, 2 * n:].reshape(T, n, n), iters)
    x_in = np.einsum("ti,tid->td", H_pre, x)
    return dict(x_in=x_in, H_pre=H_pre, H_post=H_post, H_res=H_res,
                proj=proj, logits=logits, inv_rms=inv_rms)


def mhc_post(x, y, H_post, H_res):
    """x_next[i] = sum_j H_res[i, j] x[j] + H_post[i] y (section 5.3)."""
    x = _f64(x)
    return (np.einsum("tij,tjd->tid", _f64(H_res), x)
            + _f64(H_post)[:, :, None] * _f64(y)[:, None, :])


def round_to_storage(v, dtype: str):
    """The value an activation takes when stored: float32 or bfloat16, each
    round-to-nearest-even from the exact value (the pages compute in fp32 and
    store activations in the tensor's type).  bfloat16 keeps 8 significant
    bits and float32's exponent range; values here are far from its limits.
    """
    v = _f64(v)
    if dtype == "f32":
        return v.astype(np.float32).astype(_F)
    if dtype != "bf16":
        raise ValueError(dtype)
    m, e = np.frexp(v)                      # v = m 2^e, 1/2 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)   # rint: ties to even


def mhc_post_stored(x, y, H_post, H_res, store: str):
    """x_next as an activation of type ``store`` holds it: the exact update
    rounded once to that type.  The pages compute in float32 and store each
    activation in its own type; they fix no order for the float32 sum, so
    the plainest reading is the exact value, rounded once at the store."""
    return round_to_storage(mhc_post(x, y, H_post, H_res), store)


def mhc_post_pre(x, y, H_post_l, H_res_l, phi, b, alpha, iters: int, eps: float,
                 store: str):
    """Layer l's residual update, then layer l + 1's pre forward on the
    stored x_next (the cross-layer fusion of the inference critical path,
    section 11.3 of the openPangu 2.0 notes; each step as in section 5.3).

    ``store`` is the activation type ("bf16" or "f32") x_next is kept in
    (``mhc_post_stored``).  Returns mhc_pre's dict plus x_next (as stored).
    """
    x_next = mhc_post_stored(x, y, H_post_l, H_res_l, store)
    out = mhc_pre(x_next, phi, b, alpha, iters, eps)
    out["x_next"] = x_next
    return out


def mhc_post_bwd(g_next, x, y, H_post, H_res):
    """Gradients of <g_next, mhc_post(x, y, H_post, H_res)>.

    Returns dict dx [T, n, D], dy [T, D], dH_post [T, n], dH_res [T, n, n].
    """
    g = _f64(g_next)
    x = _f64(x)
    y = _f64(y)
    dx = np.einsum("tij,tid->tjd", _f64(H_res), g)
    dy = np.einsum("ti,tid->td", _f64(H_post), g)
    dH_post = np.einsum("tid,td->ti", g, y)
    dH_res = np.einsum("tid,tjd->tij", g, x)
    return dict(dx=dx, dy=dy, dH_post=dH_post, dH_res=dH_res)


SANDWICH_NORM, BLOCK_NORM = 1, 2


def mhc_post_norm(x, y, H_post, H_res, flags: int, eps: float):
    """The residual update with openPangu's stability changes (section 5.4 of
    the openPangu 2.0 notes), each optional (bit of ``flags``):
      SANDWICH_NORM: the sublayer output y is RMS-normalised over D before
        the H_post write-back;
      BLOCK_NORM: the updated multi-stream state is RMS-normalised over its
        flattened n*D row (the extent of the layer's own RMSNorm).
    Unit weights, eps inside the square root.  Returns dict x_next
    [T, n, D], inv_rms_y [T], inv_rms_out [T] (1 where a step is off).
    """
    x, y = _f64(x), _f64(y)
    T = x.shape[0]
    if flags & SANDWICH_NORM:
        inv_rms_y = 1.0 / np.sqrt(np.mean(y * y, axis=1) + eps)
    else:
        inv_rms_y = np.ones(T)
    z = mhc_post(x, y * inv_rms_y[:, None], H_post, H_res)
    if flags & BLOCK_NORM:
        x_next, inv_rms_out = rmsnorm_flat(z, eps)
    else:
        x_next, inv_rms_out = z, np.ones(T)
    return dict(x_next=x_next, inv_rms_y=inv_rms_y, inv_rms_out=inv_rms_out)


def _rmsnorm_vjp(g, u, inv_rms, axes):
    """Reverse mode of u = z * inv_rms(z) (RMSNorm with unit weight over
    ``axes``): dz = inv_rms (g - u <g, u> / N), N the normalised extent."""
    N = int(np.prod([g.shape[a] for a in axes]))
    c = np.sum(g * u, axis=axes, keepdims=True)
    shape = [g.shape[0]] + [1] * (g.ndim - 1)
    return inv_rms.reshape(shape) * (g - u * c / N)


def mhc_post_norm_bwd(g_next, x, y, H_post, H_res, flags: int, eps: float):
    """Gradients of <g_next, x_next> for mhc_post_norm, by the chain rule
    through its steps.  Returns dict dx, dy, dH_post, dH_res."""
    f = mhc_post_norm(x, y, H_post, H_res, flags, eps)
    g = _f64(g_next)
    dz = _rmsnorm_vjp(g, f["x_next"], f["inv_rms_out"], (1, 2)) if flags & BLOCK_NORM else g
    yn = _f64(y) * f["inv_rms_y"][:, None]
    pb = mhc_post_bwd(dz, x, yn, H_post, H_res)
    dy = _rmsnorm_vjp(pb["dy"], yn, f["inv_rms_y"], (1,)) if flags & SANDWICH_NORM else pb["dy"]
    return dict(dx=pb["dx"], dy=dy, dH_post=pb["dH_post"], dH_res=pb["dH_res"])


def mhc_pre_bwd(g_in, dH_post, dH_res, x, phi, b, alpha, iters: int,
                eps: float):
    """Gradients of <g_in, x_in> + (terms reaching H_post, H_res).

    dH_post and dH_res are the upstream gradients of the gates (as returned by
    ``mhc_post_bwd``).  Returns dict dx [T, n, D] (the pre-side part only: the
    H_pre mix plus the path through the projection and RMSNorm), dphi [K, G],
    db [G], dalpha [3], and the per-token intermediates dlogits [T, G] and
    dH_pre [T, n].
    """
    x = _f64(x)
    g_in = _f64(g_in)
    phi = _f64(phi)
    T, n, D = x.shape
    K = n * D
    fwd = mhc_pre(x, phi, b, alpha, iters, eps)
    logits, proj, inv_rms = fwd["logits"], fwd["proj"], fwd["inv_rms"]
    H_pre = fwd["H_pre"]

    # x_in = sum_i H_pre[i] x[i]
    dH_pre = np.einsum("td,tid->ti", g_in, x)
    dx = H_pre[:, :, None] * g_in[:, None, :]

    # gates
    s_pre = _sigmoid(logits[:, :n])
    s_post = _sigmoid(logits[:, n:2 * n])
    dl_pre = dH_pre * s_pre * (1.0 - s_pre)
    dl_post = _f64(dH_post) * 2.0 * s_post * (1.0 - s_post)
    dl_res = sinkhorn_vjp(logits[:, 2 * n:].reshape(T, n, n), iters,
                          _f64(dH_res)).reshape(T, n * n)
    dlogits = np.concatenate([dl_pre, dl_post, dl_res], axis=1)

    # logits = alpha_group * proj + b
    grp = group_of_logit(n)
    db = dlogits.sum(axis=0)
    dalpha = np.array([np.sum((dlogits * proj)[:, grp == g]) for g in range(3)])
    dproj = dlogits * _f64(alpha)[grp][None, :]

    # proj = x_bar @ phi
    x_bar = (x * inv_rms[:, None, None]).reshape(T, K)
    dphi = x_bar.T @ dproj
    dx_bar = dproj @ phi.T                              # [T, K]

    # x_bar = x * s, s = (mean(x^2) + eps)^(-1/2)
    xf = x.reshape(T, K)
    s = inv_rms[:, None]
    dot = np.sum(dx_bar * xf, axis=1, keepdims=True)
    dx_norm = s * dx_bar - (s ** 3) * xf * dot / K
    dx = dx + dx_norm.reshape(T, n, D)
    return dict(dx=dx, dphi=dphi, db=db, dalpha=dalpha, dlogits=dlogits,
                dH_pre=dH_pre)
