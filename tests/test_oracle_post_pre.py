"""Pins of the oracle's cross-layer step (mhc_post of layer l, then mhc_pre of
layer l + 1 on the stored x_next) and of its storage rounding.

The composition itself is two pinned oracle functions; what is new is the
value x_next takes when stored: a float32 sum (one rounding per multiply-add,
pinned against exact rational arithmetic) rounded to bfloat16 (pinned against
PyTorch's own float32 -> bfloat16 conversion, ties to even).
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


def _round_exact_to_f32(fr):
    """Round an exact rational to float32, ties to even, by brute force."""
    from fractions import Fraction
    c = np.float32(float(fr))                  # within one float32 unit of the answer
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(cands, key=lambda v: (abs(Fraction(float(v)) - fr),
                                     int(np.frexp(np.float64(v))[0] * 2 ** 24) % 2))
    return float(best)


def test_fp32_fma_is_one_rounding_of_the_exact_value():
    from fractions import Fraction
    rng = np.random.default_rng(21)
    a, b, c = (rng.standard_normal(3000).astype(np.float32) * s for s in (1.0, 1.0, 1e-3))
    got = O.fp32_fma(a, b, c)
    ref = [_round_exact_to_f32(Fraction(float(p)) * Fraction(float(q)) + Fraction(float(r)))
           for p, q, r in zip(a, b, c)]
    np.testing.assert_array_equal(got, np.array(ref))


def test_stored_x_next_is_the_rounded_update():
    # within one unit of the storage type of the exact update (plus the
    # float32 sum's own rounding), and exactly the bf16 rounding of the exact
    # value wherever that is not near a rounding boundary
    x, y, _, _, _ = _layer_inputs(T=9, D=32, seed=8)
    T, n, _ = x.shape
    rng = np.random.default_rng(9)
    H_res = rng.random((T, n, n)).astype(np.float32).astype(np.float64) * 0.5
    H_post = rng.random((T, n)).astype(np.float32).astype(np.float64) * 2.0
    exact = O.mhc_post(x, y, H_post, H_res)
    # five float32 roundings along the sum, each at most half a unit of a
    # partial sum bounded by the sum of the terms' magnitudes
    mag = O.mhc_post(np.abs(x), np.abs(y), np.abs(H_post), np.abs(H_res))
    fp32_err = (n + 1) * 2.0 ** -24 * mag
    for store, bits in (("bf16", 8), ("f32", 24)):
        got = O.mhc_post_stored(x, y, H_post, H_res, store)
        unit = np.ldexp(1.0, np.frexp(exact)[1] - bits)
        assert np.all(np.abs(got - exact) <= unit + fp32_err)
    direct = O.round_to_storage(exact, "bf16")
    got = O.mhc_post_stored(x, y, H_post, H_res, "bf16")
    m = np.frexp(exact)[0] * 256.0
    far = np.abs(m - np.floor(m) - 0.5) > 1e-4
    np.testing.assert_array_equal(got[far], direct[far])
