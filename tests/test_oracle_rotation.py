"""Pins for the oracle's offline calibration (Technical Summary sections 2.1, 2.2A)."""
import itertools

import numpy as np
import pytest
import scipy.linalg

import golden_io
from oracle import rotation


# --- Hadamard ---------------------------------------------------------------

def test_hadamard_matches_textbook_sylvester():
    for d, h in golden_io.hadamard().items():
        np.testing.assert_array_equal(rotation.hadamard(d) * np.sqrt(d), h)


@pytest.mark.parametrize("d", [2, 8, 32, 64, 128])
def test_hadamard_matches_scipy_and_is_orthogonal(d):
    h = rotation.hadamard(d)
    np.testing.assert_allclose(h, scipy.linalg.hadamard(d) / np.sqrt(d), rtol=0, atol=1e-15)
    assert np.abs(h @ h.T - np.eye(d)).max() <= 1e-15 * d
    np.testing.assert_array_equal(h, h.T)
    assert set(np.unique(np.abs(h) * np.sqrt(d)).round(12)) == {1.0}


def test_hadamard_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        rotation.hadamard(48)


# --- bit reversal -----------------------------------------------------------

def test_bit_reversal_golden():
    for d, br in golden_io.bitrev().items():
        np.testing.assert_array_equal(rotation.bit_reverse(d), br)


@pytest.mark.parametrize("d", [64, 128])
def test_bit_reversal_is_involution_and_matrix_symmetric(d):
    br = rotation.bit_reverse(d)
    np.testing.assert_array_equal(br[br], np.arange(d))
    p = rotation.bit_reversal_matrix(d)
    np.testing.assert_array_equal(p, p.T)
    np.testing.assert_array_equal(p.sum(0), 1)
    x = np.arange(d, dtype=float)
    np.testing.assert_array_equal(x @ p, br.astype(float))   # (xP)_j = x_br(j)


# --- eigenbasis -------------------------------------------------------------

def _haar(rng, d):
    q, r = np.linalg.qr(rng.standard_normal((d, d)))
    return q * np.sign(np.diag(r))


@pytest.mark.parametrize("d", [8, 64, 128])
def test_eigh_planted_spectrum(d):
    rng = np.random.default_rng(1)
    w = _haar(rng, d)
    lam = 0.93 ** np.arange(d) + 0.01
    c = w @ np.diag(lam) @ w.T
    ev, u = rotation.sorted_eigh(c)
    np.testing.assert_allclose(ev, lam, rtol=1e-12, atol=1e-14)
    assert np.all(np.diff(ev) < 0)
    # same basis up to the sign of each column
    dots = np.abs(np.sum(u * w, axis=0))
    np.testing.assert_allclose(dots, 1.0, atol=1e-9)
    assert np.linalg.norm(c @ u - u * ev) <= 1e-10 * np.linalg.norm(c)
    assert np.abs(u.T @ u - np.eye(d)).max() <= 1e-12
    np.testing.assert_allclose(ev, np.sort(np.linalg.eigvalsh(c))[::-1], rtol=1e-12, atol=1e-14)


def test_eigh_canonical_sign_and_diagonal_case():
    c = np.diag([1.0, 5.0, 3.0, 2.0])
    ev, u = rotation.sorted_eigh(c)
    np.testing.assert_array_equal(ev, [5.0, 3.0, 2.0, 1.0])
    # a diagonal matrix returns a permutation matrix with +1 entries
    np.testing.assert_array_equal(u, np.eye(4)[:, [1, 2, 3, 0]])
    rng = np.random.default_rng(3)
    a = rng.standard_normal((16, 16))
    _, u = rotation.sorted_eigh(a @ a.T)
    for col in range(16):
        i = np.argmax(np.abs(u[:, col]))
        assert u[i, col] > 0


# --- covariances ------------------------------------------------------------

def test_query_covariance_brute_force():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((5, 2, 3))
    ref = np.zeros((3, 3))
    for n, g in itertools.product(range(5), range(2)):
        for a in range(3):
            for b in range(3):
                ref[a, b] += q[n, g, a] * q[n, g, b]
    np.testing.assert_allclose(rotation.query_covariance(q), ref / 10, rtol=1e-14)


def _score_cov_loops(q, k, v):
    n, g, d = q.shape
    acc = np.zeros((d, d))
    for h in range(g):
        for i in range(n):
            logits = [sum(q[i, h, c] * k[m, c] for c in range(d)) / np.sqrt(d) for m in range(i + 1)]
            mx = max(logits)
            w = [np.exp(x - mx) for x in logits]
            tot = sum(w)
            o = [sum(w[m] / tot * v[m, c] for m in range(i + 1)) for c in range(d)]
            for a in range(d):
                for b in range(d):
                    acc[a, b] += o[a] * o[b]
    return acc / (n * g)


def test_score_covariance_brute_force_and_blocking():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((6, 2, 4))
    k = rng.standard_normal((6, 4))
    v = rng.standard_normal((6, 4))
    ref = _score_cov_loops(q, k, v)
    np.testing.assert_allclose(rotation.score_covariance(q, k, v), ref, rtol=1e-12)
    np.testing.assert_allclose(rotation.score_covariance(q, k, v, block=1), ref, rtol=1e-12)


def test_score_covariance_closed_forms():
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, 5))
    q = rng.standard_normal((1, 1, 5))
    k = rng.standard_normal((1, 5))
    # one token: S = [1], C_S = v^T v
    np.testing.assert_allclose(rotation.score_covariance(q, k, v), v.T @ v, rtol=1e-14)
    # identical keys: causal attention is uniform, so O_n = mean(V[:n+1])
    n = 7
    v = rng.standard_normal((n, 5))
    k = np.tile(rng.standard_normal(5), (n, 1))
    q = rng.standard_normal((n, 1, 5))
    o = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(rotation.score_covariance(q, k, v), o.T @ o / n, rtol=1e-12)


# --- composite rotation and clip ---------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
def test_composite_rotation_structure(d):
    rng = np.random.default_rng(7)
    a = rng.standard_normal((3 * d, d)) * np.exp(rng.standard_normal(d))
    c = a.T @ a / (3 * d)
    r = rotation.composite_rotation(c, d, rotation.OSCAR)
    assert np.abs(r.T @ r - np.eye(d)).max() <= 1e-9
    # undoing P_br and H leaves the sorted eigenbasis of C
    _, u = rotation.sorted_eigh(c)
    u_back = r @ rotation.bit_reversal_matrix(d).T @ rotation.hadamard(d).T
    np.testing.assert_allclose(u_back, u, atol=1e-12)
    # the first rotated channel carries the top eigen-direction spread by H:
    # column j of R is U @ H[:, br(j)]
    br = rotation.bit_reverse(d)
    np.testing.assert_allclose(r[:, 5], u @ rotation.hadamard(d)[:, br[5]], atol=1e-13)
    np.testing.assert_array_equal(rotation.composite_rotation(None, d, rotation.IDENTITY), np.eye(d))
    np.testing.assert_array_equal(rotation.composite_rotation(None, d, rotation.HADAMARD_ONLY),
                                  rotation.hadamard(d))


def test_percentile_golden():
    for p, expected, vals in golden_io.percentiles():
        assert rotation.clip_threshold(vals[:, None], np.eye(1), p) == pytest.approx(expected, rel=1e-12)


def test_clip_is_percentile_of_abs_rotated_entries():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((200, 8))
    r = _haar(rng, 8)
    y = np.sort(np.abs(x @ r).ravel())
    h = (y.size - 1) * 0.999
    lo = int(np.floor(h))
    ref = y[lo] + (h - lo) * (y[lo + 1] - y[lo])
    assert rotation.clip_threshold(x, r, 99.9) == pytest.approx(ref, rel=1e-13)
