"""Pins of the float64 oracle against closed forms and invariants.

None of these re-types the oracle's own formula: each checks a value or a
property that the definitions on the pages (openPangu 2.0 notes, section 5.3;
Ascend mHC Triton operator article, paragraph on H^res / H^pre / H^post) or
plain mathematics fix independently.  A plausible slip in the oracle (a
transposed operand, a wrong flattening order, a swapped logit group, a missing
eps) breaks at least one of them.
"""

import math

import numpy as np
import scipy.special

from oracle import mhc_oracle as O


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------- RMSNorm ---

def test_rmsnorm_constant_row_closed_form():
    # every element c: mean(x^2) = c^2, so x_bar = c / sqrt(c^2 + eps)
    for c, eps in [(3.0, 1e-6), (-0.5, 1e-2), (1e-3, 1e-6)]:
        x = np.full((2, 4, 8), c)
        xb, inv = O.rmsnorm_flat(x, eps)
        np.testing.assert_allclose(xb, c / math.sqrt(c * c + eps), rtol=1e-15)
        np.testing.assert_allclose(inv, 1.0 / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_normalises_over_all_streams():
    # With eps = 0 the flattened n*D row has unit mean square.  If the norm
    # were taken per stream instead, this two-stream row would fail.
    x = np.zeros((1, 2, 4))
    x[0, 0] = [1, 1, 1, 1]
    x[0, 1] = [3, 3, 3, 3]
    xb, inv = O.rmsnorm_flat(x, 0.0)
    assert abs(np.mean(xb ** 2) - 1.0) < 1e-15
    assert abs(inv[0] - 1.0 / math.sqrt(5.0)) < 1e-15
    x = _rng(1).normal(size=(5, 4, 16)) * 7.0
    xb, _ = O.rmsnorm_flat(x, 0.0)
    np.testing.assert_allclose(np.mean(xb.reshape(5, -1) ** 2, axis=1), 1.0,
                               rtol=1e-14)


def test_rmsnorm_scale_invariance():
    x = _rng(2).normal(size=(3, 4, 8))
    a, _ = O.rmsnorm_flat(x, 0.0)
    b, _ = O.rmsnorm_flat(x * 123.0, 0.0)
    c, _ = O.rmsnorm_flat(-x, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-14)
    np.testing.assert_allclose(a, -c, rtol=1e-14)


# ------------------------------------------------------------ projection ---

def test_projection_picks_stream_major_elements():
    # phi[:, g] = e_{k_g} with k = i*D + d picks x_bar[i, d]; catches a
    # transposed phi or a [D, n] flattening.
    n, D = 4, 8
    G = 2 * n + n * n
    x = _rng(3).normal(size=(2, n, D))
    xb, _ = O.rmsnorm_flat(x, 1e-6)
    picks = [(g % n, (3 * g + 1) % D) for g in range(G)]
    phi = np.zeros((n * D, G))
    for g, (i, d) in enumerate(picks):
        phi[i * D + d, g] = 1.0
    p = O.project(xb, phi)
    for g, (i, d) in enumerate(picks):
        np.testing.assert_allclose(p[:, g], xb[:, i, d], rtol=0, atol=0)


def test_logit_groups_alpha_and_bias():
    n = 4
    G = 2 * n + n * n
    grp = O.group_of_logit(n)
    assert list(grp[:4]) == [0] * 4 and list(grp[4:8]) == [1] * 4
    assert list(grp[8:]) == [2] * 16
    proj = np.ones((1, G))
    b = np.arange(G, dtype=float) * 0.1
    lg = O.logits_from_proj(proj, [2.0, 3.0, 5.0], b, n)
    expect = np.array([2.0] * 4 + [3.0] * 4 + [5.0] * 16) + b
    np.testing.assert_allclose(lg[0], expect, rtol=1e-15)
    # zero projection: logits are the bias exactly
    lg0 = O.logits_from_proj(np.zeros((3, G)), [0.7, 0.7, 0.7], b, n)
    np.testing.assert_array_equal(lg0, np.tile(b, (3, 1)))


# ----------------------------------------------------------------- gates ---

def test_gates_match_library_logistic_and_ranges():
    n = 4
    lg = _rng(4).normal(size=(50, 2 * n + n * n)) * 6.0
    hp, hq = O.gates(lg, n)
    np.testing.assert_allclose(hp, scipy.special.expit(lg[:, :n]), rtol=1e-14)
    np.testing.assert_allclose(hq, 2 * scipy.special.expit(lg[:, n:2 * n]),
                               rtol=1e-14)
    assert np.all((hp > 0) & (hp < 1))          # H_pre in (0, 1)
    assert np.all((hq > 0) & (hq < 2))          # H_post in (0, 2)


def test_gates_at_zero_and_symmetry():
    n = 4
    hp, hq = O.gates(np.zeros((1, 24)), n)
    np.testing.assert_array_equal(hp, 0.5)
    np.testing.assert_array_equal(hq, 1.0)
    lg = _rng(5).normal(size=(7, 24))
    a, b = O.gates(lg, n)
    c, d = O.gates(-lg, n)
    np.testing.assert_allclose(a + c, 1.0, rtol=1e-15)
    np.testing.assert_allclose(b + d, 2.0, rtol=1e-15)


# ------------------------------------------------------------- pre / post ---

def test_pre_mix_selects_one_stream():
    # Logits +-40 make H_pre = e_k to within 4e-18, so x_in = x_k.
    n, D = 4, 8
    x = _rng(6).normal(size=(1, n, D))
    for k in range(n):
        phi = np.zeros((n * D, 2 * n + n * n))
        b = np.full(2 * n + n * n, -40.0)
        b[k] = 40.0
        out = O.mhc_pre(x, phi, b, [1.0, 1.0, 1.0], 20, 1e-6)
        np.testing.assert_allclose(out["x_in"][0], x[0, k], rtol=1e-15,
                                   atol=1e-15)


def test_pre_is_homogeneous_in_x_without_eps():
    # eps = 0: the gates see only x / rms(x), so x_in(c x) = c x_in(x).
    n, D = 4, 16
    r = _rng(7)
    x = r.normal(size=(3, n, D))
    phi = r.normal(size=(n * D, 24)) * 0.3
    b = r.normal(size=24) * 0.1
    a = O.mhc_pre(x, phi, b, [0.5, 0.5, 0.5], 20, 0.0)
    c = O.mhc_pre(x * 9.0, phi, b, [0.5, 0.5, 0.5], 20, 0.0)
    np.testing.assert_allclose(c["x_in"], 9.0 * a["x_in"], rtol=1e-13)
    np.testing.assert_allclose(c["H_res"], a["H_res"], rtol=1e-13)


def test_post_identity_and_permutation():
    n, D, T = 4, 8, 3
    r = _rng(8)
    x = r.normal(size=(T, n, D))
    y = r.normal(size=(T, D))
    hq = r.uniform(0, 2, size=(T, n))
    eye = np.tile(np.eye(n), (T, 1, 1))
    out = O.mhc_post(x, y, hq, eye)
    np.testing.assert_allclose(out, x + hq[:, :, None] * y[:, None, :],
                               rtol=1e-15)
    # H_res = permutation matrix P (P[i, perm[i]] = 1): stream i of the
    # output is stream perm[i] of the input.  Catches H_res^T.
    perm = [2, 0, 3, 1]
    P = np.zeros((n, n))
    for i, j in enumerate(perm):
        P[i, j] = 1.0
    out = O.mhc_post(x, y, np.zeros((T, n)), np.tile(P, (T, 1, 1)))
    for i, j in enumerate(perm):
        np.testing.assert_array_equal(out[:, i], x[:, j])


def test_post_preserves_stream_sum_with_unit_column_sums():
    # sum_i (H_res x)_i = sum_j x_j when every column of H_res sums to 1;
    # the column-last Sinkhorn gives exactly that.
    n, D, T = 4, 32, 5
    r = _rng(9)
    x = r.normal(size=(T, n, D))
    y = r.normal(size=(T, D))
    H = O.sinkhorn(r.normal(size=(T, n, n)) * 2.0, 3)
    hq = r.uniform(0, 2, size=(T, n))
    out = O.mhc_post(x, y, hq, H)
    lhs = out.sum(axis=1)
    rhs = x.sum(axis=1) + hq.sum(axis=1)[:, None] * y
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def test_post_bwd_adjoint_identity():
    # <g, post(x, y)> is bilinear: the returned gradients reproduce it
    # exactly (Euler): <g, out> = <dx, x> + <dy, y> split by linearity in
    # (x, y) at fixed H, and = <dH_res, H_res> + <dH_post, H_post> in (H).
    n, D, T = 4, 8, 4
    r = _rng(10)
    x, g = r.normal(size=(T, n, D)), r.normal(size=(T, n, D))
    y = r.normal(size=(T, D))
    hq = r.uniform(0, 2, size=(T, n))
    H = r.uniform(0, 1, size=(T, n, n))
    out = O.mhc_post(x, y, hq, H)
    gr = O.mhc_post_bwd(g, x, y, hq, H)
    total = np.sum(g * out)
    assert abs(total - (np.sum(gr["dx"] * x) + np.sum(gr["dy"] * y))) < 1e-11
    assert abs(total - (np.sum(gr["dH_res"] * H)
                        + np.sum(gr["dH_post"] * hq))) < 1e-11
