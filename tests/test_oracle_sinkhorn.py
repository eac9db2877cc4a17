"""Pins of the oracle's Sinkhorn-Knopp projection.

Facts used (openPangu 2.0 notes, section 5.3: H_res = Sinkhorn(reshape(r_res)),
20 rounds, approximately doubly stochastic; Ascend mHC Triton operator article:
non-negative entries, row and column sums 1) plus textbook properties of
matrix scaling:
  * equal logits give the uniform matrix 1/n;
  * every iterate is D1 exp(L) D2 for positive diagonals D1, D2;
  * the limit is the unique doubly stochastic scaling of exp(L), which an
    independent root finder (scipy) reaches from the marginal equations;
  * for n = 2 that limit has the closed form p = sqrt(ad)/(sqrt(ad)+sqrt(bc));
  * a rank-one exp(L) is uniform after a single round.
"""

import math

import numpy as np
import scipy.optimize

from oracle import mhc_oracle as O


def test_equal_logits_give_uniform():
    for n in (2, 3, 4, 6):
        for c in (0.0, 5.0, -3.0):
            H = O.sinkhorn(np.full((2, n, n), c), 20)
            np.testing.assert_allclose(H, 1.0 / n, rtol=1e-15)


def test_rank_one_is_uniform_after_one_round():
    r = np.random.default_rng(11)
    u, v = r.normal(size=4), r.normal(size=4)
    L = (u[:, None] + v[None, :])[None]          # exp(L) = e^u e^v^T
    np.testing.assert_allclose(O.sinkhorn(L, 1), 0.25, rtol=1e-14)


def test_iterates_are_diagonal_scalings():
    # log(M_k) - L = a_i + c_j, so every 2x2 cross difference vanishes.
    r = np.random.default_rng(12)
    L = r.normal(size=(3, 4, 4)) * 2.0
    for M in O.sinkhorn_iterates(L, 7):
        R = np.log(M) - L
        cross = R[:, :, None, :, None] - R[:, :, None, None, :] \
            - R[:, None, :, :, None] + R[:, None, :, None, :]
        assert np.max(np.abs(cross)) < 1e-12


def test_column_sums_exact_and_rows_converge():
    r = np.random.default_rng(13)
    L = r.normal(size=(200, 4, 4)) * 0.3          # logit spread of the cfgs
    for iters in (1, 5, 20):
        H = O.sinkhorn(L, iters)
        assert np.all(H >= 0)
        np.testing.assert_allclose(H.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    H = O.sinkhorn(L, 20)
    assert np.max(np.abs(H.sum(axis=2) - 1.0)) < 1e-6


def _fixed_point_by_root_finding(A):
    """Doubly stochastic scaling of A from the marginal equations alone."""
    n = A.shape[0]

    def resid(w):
        a = np.concatenate([[0.0], w[:n - 1]])    # gauge: a_0 = 0
        c = w[n - 1:]
        S = np.exp(a)[:, None] * A * np.exp(c)[None, :]
        return np.concatenate([S.sum(axis=1)[1:], S.sum(axis=0)]) - 1.0

    sol = scipy.optimize.root(resid, np.zeros(2 * n - 1), tol=1e-12)
    assert np.max(np.abs(resid(sol.x))) < 1e-13
    a = np.concatenate([[0.0], sol.x[:n - 1]])
    c = sol.x[n - 1:]
    return np.exp(a)[:, None] * A * np.exp(c)[None, :]


def test_limit_matches_independent_root_finder():
    r = np.random.default_rng(14)
    for scale in (0.5, 1.0, 2.0):
        L = r.normal(size=(4, 4)) * scale
        ref = _fixed_point_by_root_finding(np.exp(L))
        H = O.sinkhorn(L[None], 2000)[0]
        np.testing.assert_allclose(H, ref, rtol=0, atol=1e-10)


def test_two_by_two_closed_form():
    # The doubly stochastic scaling of A = [[a, b], [c, d]] is
    # [[p, 1-p], [1-p, p]] with p = sqrt(ad) / (sqrt(ad) + sqrt(bc)):
    # the scaling keeps the cross ratio (ad)/(bc) = p^2 / (1-p)^2.
    for a, b, c, d in [(1.0, 2.0, 3.0, 4.0), (0.2, 5.0, 1.0, 0.7),
                       (9.0, 0.1, 0.3, 2.0), (1.0, 1.0, 1.0, 1.0)]:
        p = math.sqrt(a * d) / (math.sqrt(a * d) + math.sqrt(b * c))
        L = np.log(np.array([[a, b], [c, d]]))[None]
        H = O.sinkhorn(L, 400)[0]
        np.testing.assert_allclose(H, [[p, 1 - p], [1 - p, p]], atol=1e-12)


def test_peaked_permutation_logits():
    perm = [1, 3, 0, 2]
    L = np.zeros((1, 4, 4))
    for i, j in enumerate(perm):
        L[0, i, j] = 12.0
    H = O.sinkhorn(L, 20)[0]
    for i, j in enumerate(perm):
        assert H[i, j] > 1 - 1e-4
    assert abs(H.sum() - 4.0) < 1e-9


def test_row_shift_invariance_and_gradient_rows_sum_to_zero():
    # Adding a constant to a row of L scales a row of exp(L); the first row
    # normalisation removes it, so H is unchanged at any iteration count and
    # the gradient along each row of L sums to zero.
    r = np.random.default_rng(15)
    L = r.normal(size=(5, 4, 4))
    shift = r.normal(size=(5, 4, 1)) * 3.0
    for iters in (1, 5, 20):
        np.testing.assert_allclose(O.sinkhorn(L + shift, iters),
                                   O.sinkhorn(L, iters), rtol=1e-13)
        dL = O.sinkhorn_vjp(L, iters, r.normal(size=(5, 4, 4)))
        assert np.max(np.abs(dL.sum(axis=2))) < 1e-13


def test_vjp_matches_central_differences():
    r = np.random.default_rng(16)
    for n in (2, 4):
        for iters in (1, 3, 20):
            L = r.normal(size=(1, n, n))
            W = r.normal(size=(1, n, n))
            g = O.sinkhorn_vjp(L, iters, W)
            h = 1e-6
            fd = np.zeros_like(L)
            for i in range(n):
                for j in range(n):
                    e = np.zeros_like(L)
                    e[0, i, j] = h
                    fd[0, i, j] = (np.sum(W * O.sinkhorn(L + e, iters))
                                   - np.sum(W * O.sinkhorn(L - e, iters))) / (2 * h)
            np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-9)
