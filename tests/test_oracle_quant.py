"""Pins for the oracle's rotate + clip + INT2 quantiser (Technical Summary 2.2B)."""
import numpy as np
import pytest

import golden_io
from oracle import quant, rotation


def test_hand_worked_groups():
    for clip, s, z, vals, codes in golden_io.quant_groups():
        c, s16, z16 = quant.quantize(vals[None, :], clip)
        np.testing.assert_array_equal(c[0], codes)
        assert float(s16[0, 0]) == s
        assert float(z16[0, 0]) == z


def test_codes_are_nearest_level():
    """Away from exact ties, RNE((y_c - z)/s) clamped is the level nearest to y_c."""
    rng = np.random.default_rng(0)
    y = rng.standard_normal((300, 128)) * np.exp(rng.standard_normal(128))
    clip = 2.5
    codes, s16, z16 = quant.quantize(y, clip)
    yc = quant.clipped(y, clip).astype(np.float64).reshape(300, 4, 32)
    lv = (np.arange(4)[None, None, None, :] * s16.astype(np.float64)[..., None, None]
          + z16.astype(np.float64)[..., None, None])
    dist = np.abs(yc[..., None] - lv)
    best = dist.argmin(-1)
    srt = np.sort(dist, -1)
    clear = (srt[..., 1] - srt[..., 0]) > 1e-5 * (s16.astype(np.float64)[..., None] + 1e-30)
    got = codes.reshape(300, 4, 32)
    assert np.all(got[clear] == best[clear])
    assert clear.mean() > 0.99


def test_codes_range_and_reconstruction_bound():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((500, 64)) * 3
    clip = 5.0
    codes, s16, z16 = quant.quantize(y, clip)
    assert codes.max() <= 3 and codes.min() >= 0
    yh = quant.dequantize(codes, s16, z16)
    s = np.repeat(s16.astype(np.float64), 32, axis=-1)
    z = np.repeat(z16.astype(np.float64), 32, axis=-1)
    unclipped = np.abs(y) < clip
    err = np.abs(quant.clipped(y, clip) - yh)
    bound = s / 2 + 2.0 ** -11 * (np.abs(z) + 3 * s) + 1e-12
    assert np.all(err[unclipped] <= bound[unclipped])


def test_scale_zero_are_fp16_roundings():
    rng = np.random.default_rng(2)
    y = rng.standard_normal((50, 64))
    codes, s16, z16 = quant.quantize(y, 10.0)
    g = y.astype(np.float32).reshape(50, 2, 32)
    mn, mx = g.min(-1), g.max(-1)
    np.testing.assert_array_equal(z16, mn.astype(np.float16))
    np.testing.assert_array_equal(s16, ((mx - mn) / np.float32(3)).astype(np.float16))


def test_clipping_and_constant_groups():
    y = np.zeros((1, 64))
    y[0, :32] = 7.0                 # constant group
    y[0, 32:] = np.linspace(-9, 9, 32)
    codes, s16, z16 = quant.quantize(y, 4.0)
    assert float(s16[0, 0]) == 0 and np.all(codes[0, :32] == 0) and float(z16[0, 0]) == 4.0
    assert float(z16[0, 1]) == -4.0
    assert codes[0, 32] == 0 and codes[0, 63] == 3


def test_flags_cover_only_near_boundary_entries():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 64)).astype(np.float32)
    r = np.linalg.qr(rng.standard_normal((64, 64)))[0].astype(np.float32)
    elem, grp = quant.near_boundary_flags(x, r, 2.0, kappa=2.0 ** -16)
    # a rigorous worst-case bound: a minority of groups sits near an fp16 step
    assert elem.mean() < 0.01 and grp.mean() < 0.25
    # a kernel-like perturbation inside the bound flips only flagged entries
    y = quant.rotate(x, r)
    eps = 2.0 ** -16 * (np.abs(x.astype(np.float64)) @ np.abs(r.astype(np.float64)))
    pert = y + eps * rng.uniform(-1, 1, y.shape)
    c0, s0, z0 = quant.quantize(y, 2.0)
    c1, s1, z1 = quant.quantize(pert, 2.0)
    gmask = np.repeat(grp, 32, axis=-1)
    ok = ~(elem | gmask)
    assert np.all(c0[ok] == c1[ok])
    assert np.all(s0[~grp] == s1[~grp]) and np.all(z0[~grp] == z1[~grp])
    # with kappa = 0 nothing but exact ties would be flagged
    e0, g0 = quant.near_boundary_flags(x, r, 2.0, kappa=0.0)
    assert e0.mean() < 1e-3 and g0.mean() < 1e-3


@pytest.mark.parametrize("d", [64, 128])
def test_identity_and_signed_permutation_rotations_are_exact(d):
    """Exact rotations give y exactly, so no entry needs a flag (kappa = 0)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((32, d)).astype(np.float32)
    perm = rng.permutation(d)
    r = np.zeros((d, d), np.float32)
    r[np.arange(d), perm] = rng.choice([-1.0, 1.0], d)
    y = quant.rotate(x, r)
    np.testing.assert_array_equal(y[:, perm], x * r[np.arange(d), perm][None, :])


# ------------------------------------------------------------ INT4 variant (levels 15)

def test_int4_grid_values_are_their_own_codes():
    """A group spanning [0, 15] with fp16-exact entries has s16 = 1 and z16 = 0,
    so every integer entry is its own code and half-integers round to even."""
    vals = np.concatenate([np.arange(16.0), np.arange(16.0)[::-1]])
    vals[5], vals[6], vals[7], vals[20] = 0.5, 1.5, 2.5, 14.5
    codes, s16, z16 = quant.quantize(vals[None, :], 100.0, levels=quant.INT4_MAX_CODE)
    assert float(s16[0, 0]) == 1.0 and float(z16[0, 0]) == 0.0
    want = np.rint(vals).astype(np.uint8)      # numpy rint is round-half-even
    np.testing.assert_array_equal(codes[0], want)
    assert list(codes[0, [5, 6, 7, 20]]) == [0, 2, 2, 14]


def test_int4_range_scale_and_reconstruction_bound():
    rng = np.random.default_rng(11)
    y = rng.standard_normal((400, 128)) * np.exp(rng.standard_normal(128))
    clip = 3.0
    codes, s16, z16 = quant.quantize(y, clip, levels=15)
    assert codes.max() <= 15 and codes.min() >= 0 and codes.max() > 3
    g = quant.clipped(y, clip).reshape(400, 4, 32)
    np.testing.assert_array_equal(s16, ((g.max(-1) - g.min(-1)) / np.float32(15)).astype(np.float16))
    yh = quant.dequantize(codes, s16, z16)
    s = np.repeat(s16.astype(np.float64), 32, axis=-1)
    z = np.repeat(z16.astype(np.float64), 32, axis=-1)
    err = np.abs(quant.clipped(y, clip) - yh)
    bound = s / 2 + 2.0 ** -11 * (np.abs(z) + 15 * s) + 1e-12
    assert np.all(err <= bound)
    # sixteen levels: the worst error is about a fifth of the four-level one
    c2, s2, z2 = quant.quantize(y, clip)
    e2 = np.abs(quant.clipped(y, clip) - quant.dequantize(c2, s2, z2))
    assert err.max() < 0.3 * e2.max()


def test_int4_flags_cover_only_near_boundary_entries():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((64, 64)).astype(np.float32)
    r = np.linalg.qr(rng.standard_normal((64, 64)))[0].astype(np.float32)
    elem, grp = quant.near_boundary_flags(x, r, 2.0, kappa=2.0 ** -16, levels=15)
    y = quant.rotate(x, r)
    eps = 2.0 ** -16 * (np.abs(x.astype(np.float64)) @ np.abs(r.astype(np.float64)))
    for seed in range(3):
        pert = y + eps * np.random.default_rng(seed).uniform(-1, 1, y.shape)
        c0, s0, z0 = quant.quantize(y, 2.0, levels=15)
        c1, s1, z1 = quant.quantize(pert, 2.0, levels=15)
        ok = ~(elem | np.repeat(grp, 32, axis=-1))
        assert np.all(c0[ok] == c1[ok])
        assert np.all(np.abs(c0.astype(int) - c1.astype(int))[~np.repeat(grp, 32, axis=-1)] <= 1)
    # finer levels put more entries near a decision boundary than INT2 does
    e2, _ = quant.near_boundary_flags(x, r, 2.0, kappa=2.0 ** -16)
    assert elem.mean() >= e2.mean() and elem.mean() < 0.05


def test_nonfinite_groups_are_zero_groups():
    """Reading for non-finite values: a group whose fp32 rotated values are not
    all finite is stored as s = z = 0 with every code 0; the other groups of the
    same vector are quantised as if it were absent."""
    rng = np.random.default_rng(5)
    y = rng.standard_normal((3, 128))
    y[0, 40] = np.nan            # group 1 of row 0
    y[1, 127] = np.inf           # group 3 of row 1
    y[2, 0] = 1e39               # finite in fp64, infinite in fp32: group 0 of row 2
    codes, s16, z16 = quant.quantize(y, 2.5)
    bad = np.zeros((3, 4), bool)
    bad[0, 1] = bad[1, 3] = bad[2, 0] = True
    np.testing.assert_array_equal(quant.nonfinite_groups(y), bad)
    for r, g in zip(*np.nonzero(bad)):
        assert s16[r, g] == 0 and z16[r, g] == 0
        assert not codes[r, 32 * g:32 * g + 32].any()
    for r in range(3):
        for g in range(4):
            if bad[r, g]:
                continue
            c1, s1, z1 = quant.quantize(y[r, 32 * g:32 * g + 32][None], 2.5)
            np.testing.assert_array_equal(codes[r, 32 * g:32 * g + 32], c1[0])
            assert s16[r, g] == s1[0, 0] and z16[r, g] == z1[0, 0]


def test_nonfinite_input_poisons_the_whole_rotated_row():
    """IEEE arithmetic: one NaN or infinity in x makes every entry of x R
    non-finite, whatever R (an infinity times a zero entry is NaN), so every
    group of that token-head becomes a zero group; other rows are untouched."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 64))
    x[0, 3] = np.inf
    x[1, 60] = np.nan
    for r in (np.eye(64), rotation.hadamard(64)):
        y = quant.rotate(x, r)
        assert np.isnan(y[:2]).all()
        np.testing.assert_allclose(y[2], x[2] @ r, rtol=1e-15, atol=1e-15)
        # direct IEEE evaluation agrees on which entries are finite
        with np.errstate(invalid="ignore"):
            direct = np.array([[np.sum(x[i] * r[:, j]) for j in range(64)] for i in range(2)])
        assert not np.isfinite(direct).any()
        codes, s16, z16 = quant.quantize(y, 1.0)
        assert not codes[:2].any() and not s16[:2].any() and not z16[:2].any()
