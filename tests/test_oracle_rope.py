"""Pins for the oracle's rotary position embedding (oracle/rope.py)."""
import math

import numpy as np

from oracle import rope


def test_hand_worked_d4():
    # d = 4, base 10000: theta = (1, 1/100); position 1 rotates pair (x0, x2) by
    # 1 rad and pair (x1, x3) by 0.01 rad
    x = np.array([1.0, 2.0, 3.0, 4.0])
    got = rope.apply(x, 1, 10000.0)
    c1, s1, c2, s2 = math.cos(1), math.sin(1), math.cos(0.01), math.sin(0.01)
    want = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + 1 * s1, 4 * c2 + 2 * s2]
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-15)


def test_position_zero_is_identity_and_norm_is_kept():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 128))
    np.testing.assert_array_equal(rope.apply(x, np.zeros(5), 1e6), x)
    y = rope.apply(x, rng.integers(0, 200000, 5), 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_dot_products_depend_on_position_difference_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    a = rope.apply(q, 1000, 1e4) @ rope.apply(k, 990, 1e4)
    b = rope.apply(q, 30, 1e4) @ rope.apply(k, 20, 1e4)
    np.testing.assert_allclose(a, b, rtol=1e-11)
    assert abs(a - q @ k) > 1e-6          # and the embedding does act


def test_inverse_frequencies():
    f = rope.inv_freq(128, 1e6)
    assert f[0] == 1.0 and f.shape == (64,)
    np.testing.assert_allclose(f[32], 1e6 ** -0.5, rtol=1e-15)
