"""Pins of the oracle's residual update with openPangu's stability changes
(sandwich normalisation of the sublayer output, block post-normalisation of
the multi-stream state; section 5.4 of the openPangu 2.0 notes).

Pinned by: reduction to mhc_post with both steps off; the exact RMS of a
normalised output; scale invariance (eps = 0); closed forms on constant rows;
and float64 central differences of the backward, every flag combination.
"""

import numpy as np
import pytest

from oracle import mhc_oracle as O

SW, BN = O.SANDWICH_NORM, O.BLOCK_NORM


def _inputs(T=3, n=4, D=8, seed=0):
    r = np.random.default_rng(seed)
    x = r.standard_normal((T, n, D))
    y = r.standard_normal((T, D)) * 3.0
    H_post = 2.0 / (1.0 + np.exp(-r.standard_normal((T, n))))
    H_res = O.sinkhorn(r.standard_normal((T, n, n)), 20)
    return x, y, H_post, H_res


def test_no_step_is_mhc_post():
    x, y, hp, hr = _inputs()
    f = O.mhc_post_norm(x, y, hp, hr, 0, 1e-6)
    np.testing.assert_array_equal(f["x_next"], O.mhc_post(x, y, hp, hr))
    assert np.all(f["inv_rms_y"] == 1.0) and np.all(f["inv_rms_out"] == 1.0)


def test_block_norm_output_has_the_rms_its_eps_allows():
    x, y, hp, hr = _inputs(seed=1)
    eps = 1e-3
    f = O.mhc_post_norm(x, y, hp, hr, BN, eps)
    z = O.mhc_post(x, y, hp, hr)
    ms = np.mean(z.reshape(z.shape[0], -1) ** 2, axis=1)
    got = np.mean(f["x_next"].reshape(z.shape[0], -1) ** 2, axis=1)
    np.testing.assert_allclose(got, ms / (ms + eps), rtol=1e-12)


def test_sandwich_uses_the_normalised_sublayer_output():
    # y scaled by any c > 0 gives the same update when eps = 0, and a
    # constant row y = c maps to a row of ones
    x, y, hp, hr = _inputs(seed=2)
    a = O.mhc_post_norm(x, y, hp, hr, SW, 0.0)["x_next"]
    b = O.mhc_post_norm(x, 7.5 * y, hp, hr, SW, 0.0)["x_next"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    yc = np.full_like(y, -4.0)
    f = O.mhc_post_norm(x, yc, hp, hr, SW, 0.0)
    np.testing.assert_allclose(f["x_next"], O.mhc_post(x, -np.ones_like(y), hp, hr), rtol=1e-12)


def test_block_norm_is_scale_invariant():
    x, y, hp, hr = _inputs(seed=3)
    # block norm alone: scaling x and y together leaves the output unchanged
    a = O.mhc_post_norm(x, y, hp, hr, BN, 0.0)["x_next"]
    b = O.mhc_post_norm(3.0 * x, 3.0 * y, hp, hr, BN, 0.0)["x_next"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    # with the sandwich step too, y's scale drops out on its own; x's does not
    c = O.mhc_post_norm(x, y, hp, hr, BN | SW, 0.0)["x_next"]
    d = O.mhc_post_norm(x, 5.0 * y, hp, hr, BN | SW, 0.0)["x_next"]
    e = O.mhc_post_norm(0.5 * x, y, hp, hr, BN | SW, 0.0)["x_next"]
    np.testing.assert_allclose(c, d, rtol=1e-12, atol=1e-12)
    assert np.max(np.abs(c - e)) > 1e-3


@pytest.mark.parametrize("flags", [0, SW, BN, SW | BN])
def test_backward_matches_central_differences(flags):
    x, y, hp, hr = _inputs(T=2, D=8, seed=4 + flags)
    eps = 1e-3
    g = np.random.default_rng(9).standard_normal(x.shape)
    loss = lambda x_, y_, hp_, hr_: float(np.sum(g * O.mhc_post_norm(x_, y_, hp_, hr_, flags, eps)["x_next"]))
    got = O.mhc_post_norm_bwd(g, x, y, hp, hr, flags, eps)
    h = 1e-6
    for name, arr, idx in (("dx", x, 0), ("dy", y, 1), ("dH_post", hp, 2), ("dH_res", hr, 3)):
        num = np.zeros_like(arr)
        for k in np.ndindex(arr.shape):
            args_p = [x, y, hp, hr]
            args_m = [x, y, hp, hr]
            ap, am = arr.copy(), arr.copy()
            ap[k] += h
            am[k] -= h
            args_p[idx], args_m[idx] = ap, am
            num[k] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(got[name], num, rtol=1e-6, atol=1e-7, err_msg=name)
