"""Pins of the oracle's cross-layer step (mhc_post of layer l, then mhc_pre of
layer l + 1 on the stored x_next) and of its storage rounding.

The composition itself is two pinned oracle functions; what is new is the
value x_next takes when stored: the exact update rounded once to the storage
type.  The bfloat16 rounding is pinned against PyTorch's own float32 ->
bfloat16 conversion (ties to even), and the stored update against the nearest
bfloat16 of the exact rational value, found by brute force.
"""

import numpy as np
import torch

from oracle import mhc_oracle as O


def _bf16_ref(v32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(v32).to(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(20000), rng.standard_normal(2000) * 1e-3,
                        rng.standard_normal(2000) * 1e4, [0.0, -0.0, 1.0, -2.5]]).astype(np.float32)
    np.testing.assert_array_equal(O.round_to_storage(v, "bf16"), _bf16_ref(v))


def test_bf16_rounding_ties_go_to_even():
    rng = np.random.default_rng(12)
    # bf16 values, then exactly half a bf16 unit above them (representable in float32)
    base = _bf16_ref(rng.standard_normal(5000).astype(np.float32))
    m, e = np.frexp(base)
    half_ulp = np.ldexp(np.ones_like(base), e - 9)          # 2^(e-1) * 2^-8 / 2
    ties = (base + np.sign(base) * half_ulp).astype(np.float32)
    assert np.all(ties.astype(np.float64) == base + np.sign(base) * half_ulp)
    got = O.round_to_storage(ties, "bf16")
    np.testing.assert_array_equal(got, _bf16_ref(ties))
    # the result's last kept bit is 0 (even) wherever the input was a tie
    q = np.rint(np.frexp(got)[0] * 256).astype(np.int64)
    assert np.all(q % 2 == 0)


def test_float32_storage_is_float32_rounding():
    v = np.array([1.0 + 2.0 ** -30, np.pi, -1e-7 / 3.0], dtype=np.float64)
    np.testing.assert_array_equal(O.round_to_storage(v, "f32"),
                                  torch.from_numpy(v).to(torch.float32).double().numpy())


def _layer_inputs(T=5, n=4, D=16, seed=3):
    rng = np.random.default_rng(seed)
    x = _bf16_ref(rng.standard_normal((T, n, D)).astype(np.float32))
    y = _bf16_ref(rng.standard_normal((T, D)).astype(np.float32))
    G = 2 * n + n * n
    phi = rng.standard_normal((n * D, G)) * 0.1
    b = rng.standard_normal(G) * 0.1
    alpha = np.array([0.5, 0.7, 0.9])
    return x, y, phi, b, alpha


def test_identity_update_reduces_to_pre():
    x, y, phi, b, alpha = _layer_inputs()
    T, n, _ = x.shape
    H_res = np.broadcast_to(np.eye(n), (T, n, n)).copy()
    H_post = np.zeros((T, n))
    got = O.mhc_post_pre(x, y, H_post, H_res, phi, b, alpha, 20, 1e-6, "bf16")
    ref = O.mhc_pre(x, phi, b, alpha, 20, 1e-6)
    np.testing.assert_array_equal(got["x_next"], x)       # x is bf16-exact
    for k in ("x_in", "H_pre", "H_post", "H_res", "proj", "inv_rms"):
        np.testing.assert_array_equal(got[k], ref[k])


def _bf16_neighbours(v: float):
    """The bf16 values just below and above the float64 value v (or v itself
    twice when v is a bf16 value), by stepping the 8-bit significand."""
    from fractions import Fraction
    if v == 0.0:
        return 0.0, 0.0
    m, e = np.frexp(v)
    lo = np.floor(m * 256.0) / 256.0
    hi = np.ceil(m * 256.0) / 256.0
    return float(np.ldexp(lo, e)), float(np.ldexp(hi, e))


def test_stored_x_next_is_the_nearest_bf16_of_the_exact_update():
    """Brute force: every stored element is the bf16 value nearest to the
    exact rational update (ties to the even significand), computed with
    Fractions from the float64-exact inputs, not from the oracle's sum."""
    from fractions import Fraction
    x, y, _, _, _ = _layer_inputs(T=4, D=12, seed=8)
    T, n, D = x.shape
    rng = np.random.default_rng(9)
    H_res = rng.random((T, n, n)).astype(np.float32).astype(np.float64) * 0.5
    H_post = rng.random((T, n)).astype(np.float32).astype(np.float64) * 2.0
    got = O.mhc_post_stored(x, y, H_post, H_res, "bf16")
    for t in range(T):
        for i in range(n):
            for d in range(D):
                ex = sum(Fraction(float(H_res[t, i, j])) * Fraction(float(x[t, j, d])) for j in range(n))
                ex += Fraction(float(H_post[t, i])) * Fraction(float(y[t, d]))
                lo, hi = _bf16_neighbours(float(ex))
                lo, hi = min(lo, hi), max(lo, hi)
                dl, dh = abs(Fraction(lo) - ex), abs(Fraction(hi) - ex)
                if dl < dh:
                    want = lo
                elif dh < dl:
                    want = hi
                else:   # a tie: the even significand
                    want = lo if int(np.frexp(lo)[0] * 256) % 2 == 0 else hi
                assert got[t, i, d] == want, (t, i, d, got[t, i, d], want)


def test_stored_x_next_float32_is_one_rounding():
    x, y, _, _, _ = _layer_inputs(T=6, D=16, seed=10)
    T, n, _ = x.shape
    rng = np.random.default_rng(13)
    H_res = rng.random((T, n, n)).astype(np.float32).astype(np.float64)
    H_post = rng.random((T, n)).astype(np.float32).astype(np.float64)
    exact = O.mhc_post(x, y, H_post, H_res)
    got = O.mhc_post_stored(x, y, H_post, H_res, "f32")
    # float32 values within half a float32 unit of the exact update
    assert np.all(got.astype(np.float32).astype(np.float64) == got)
    unit = np.ldexp(1.0, np.frexp(exact)[1] - 24)
    assert np.all(np.abs(got - exact) <= 0.5 * unit)
