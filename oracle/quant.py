"""Rotate, clip and INT2-quantise one token's key or value vector.

[Summary 2.2B] ("the historical middle context is stored in INT2 after
applying the fixed OSCAR rotation and clipping"), [Summary 1] (INT2 = four
levels).  The pages fix neither group size nor scale format; the readings taken
are: asymmetric quantisation over groups of 32 consecutive rotated channels,
fp16 scale s and fp16 zero z per group (z = group minimum, as in KIVI, which the
index page lists among the method's sources), codes chosen by
round-half-to-even, min/max taken after clipping, and codes computed from the
fp16-rounded s and z so that dequantisation matches what is stored.

Decision precision.  The rotated value y is defined exactly (fp64 here); the
integer decision (clip, group range, s, z, code) is then taken in fp32, the
precision of the library's kernels, step by step:
    y32  = fp32(y)
    yc   = min(max(y32, -c), c)
    mn, mx = min, max of yc over the group
    s16  = fp16( fp32( fp32(mx - mn) / 3 ) ),   z16 = fp16(mn)
    code = 0 if s16 == 0 else clamp(rint( fp32( fp32(yc - z16) / s16 ) ), 0, 3)
Dequantisation is y_hat = code * s16 + z16.

Non-finite values (a reading: the pages are silent).  Under IEEE arithmetic a
NaN or an infinity anywhere in x makes every entry of y = x R non-finite (an
infinity times a zero entry of R is NaN, otherwise it stays infinite or meets
another one of opposite sign), so ``rotate`` returns a row of NaN for such an
x.  A group whose fp32 values y32 are not all finite is stored as a zero group:
s16 = z16 = 0 and every code 0 (its dequantised values are 0, and the library
reports it in its status word).

INT4 variant (a format variant beside the pages' INT2, for the comparison the
pages draw with INT4 caches in [Summary 4]): the same steps with 16 levels, i.e.
the divisor 3 and the top code 3 become 15 (``levels`` = largest code).
"""
from __future__ import annotations

import numpy as np

GROUP = 32
INT2_MAX_CODE = 3     # 4 levels
INT4_MAX_CODE = 15    # 16 levels


def rotate(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    """y = x R in fp64 (x holds bf16 values, R fp32 values; each product is
    exact).  A row of x with a non-finite entry gives a row of NaN (see above)."""
    x = np.asarray(x, np.float64)
    bad = ~np.isfinite(x).all(axis=-1)
    y = np.where(bad[..., None], 0.0, x) @ np.asarray(r, np.float64)
    return np.where(bad[..., None], np.nan, y)


def quantize(y: np.ndarray, clip: float, group: int = GROUP, levels: int = INT2_MAX_CODE):
    """Quantise rotated vectors y [..., d] to codes 0..levels.  Returns (codes
    uint8 [..., d], s16 float16 [..., d/group], z16 float16 [..., d/group])."""
    with np.errstate(over="ignore", invalid="ignore"):
        y32 = np.asarray(y).astype(np.float32)
    c = np.float32(clip)
    shp = y32.shape
    d = shp[-1]
    ng = d // group
    # groups with a non-finite value are stored as zero groups
    bad = ~np.isfinite(y32.reshape(shp[:-1] + (ng, group))).all(axis=-1)
    y32 = np.where(np.repeat(bad, group, axis=-1).reshape(shp), np.float32(0), y32)
    yc = np.minimum(np.maximum(y32, -c), c)
    g = yc.reshape(shp[:-1] + (ng, group))
    mn = np.where(bad, np.float32(0), g.min(axis=-1))
    mx = np.where(bad, np.float32(0), g.max(axis=-1))
    s32 = np.float32(mx - mn) / np.float32(levels)
    s16 = s32.astype(np.float32).astype(np.float16)
    z16 = mn.astype(np.float16)
    with np.errstate(divide="ignore", invalid="ignore"):
        num = (g - z16.astype(np.float32)[..., None]).astype(np.float32)
        t = (num / s16.astype(np.float32)[..., None]).astype(np.float32)
        code = np.clip(np.rint(t), 0, levels)
    code = np.where((s16 == 0)[..., None], 0, code)
    return code.reshape(shp).astype(np.uint8), s16, z16


def nonfinite_groups(y: np.ndarray, group: int = GROUP) -> np.ndarray:
    """bool [..., d/group]: groups ``quantize`` stores as zero groups."""
    with np.errstate(over="ignore", invalid="ignore"):
        y32 = np.asarray(y).astype(np.float32)
    shp = y32.shape
    return ~np.isfinite(y32.reshape(shp[:-1] + (shp[-1] // group, group))).all(axis=-1)


def dequantize(codes: np.ndarray, s16: np.ndarray, z16: np.ndarray, group: int = GROUP) -> np.ndarray:
    """y_hat = code * s + z (fp64)."""
    c = np.asarray(codes, np.float64)
    shp = c.shape
    ng = shp[-1] // group
    c = c.reshape(shp[:-1] + (ng, group))
    yh = c * np.asarray(s16, np.float64)[..., None] + np.asarray(z16, np.float64)[..., None]
    return yh.reshape(shp)


def clipped(y: np.ndarray, clip: float) -> np.ndarray:
    y32 = np.asarray(y).astype(np.float32)
    c = np.float32(clip)
    return np.minimum(np.maximum(y32, -c), c)


def near_boundary_flags(x: np.ndarray, r: np.ndarray, clip: float, kappa: float,
                        group: int = GROUP, levels: int = INT2_MAX_CODE):
    """Entries whose decision may legitimately differ from a kernel whose fp32
    rotated value y' satisfies |y' - y| <= kappa * sum_i |x_i| |R_ij|.

    Returns (elem_flags bool [..., d], group_flags bool [..., d/group]).  A
    flagged group may differ in s16, z16 and every code; a flagged element may
    differ by one code.  Unflagged entries must agree exactly.
    """
    x = np.asarray(x, np.float64)
    r = np.asarray(r, np.float64)
    y = x @ r
    eps = kappa * (np.abs(x) @ np.abs(r))
    c = float(np.float32(clip))
    elem = np.abs(np.abs(y) - c) <= eps
    # an entry clipped with margin is exactly +-c on both sides
    eps_c = np.where(np.abs(y) - c > eps, 0.0, eps)
    codes, s16, z16 = quantize(y, clip, group, levels)
    yc = clipped(y, clip).astype(np.float64)
    shp = y.shape
    ng = shp[-1] // group
    gshape = shp[:-1] + (ng, group)
    gy = yc.reshape(gshape)
    ge = eps_c.reshape(gshape)
    # the kernel's group min / max lie in these intervals
    mn_lo, mn_hi = (gy - ge).min(-1), (gy + ge).min(-1)
    mx_lo, mx_hi = (gy - ge).max(-1), (gy + ge).max(-1)
    # z16 = fp16(mn): flag if the fp16 rounding can change inside the interval
    gflag = mn_lo.astype(np.float16) != mn_hi.astype(np.float16)
    # s16 = fp16(fp32(fp32(mx - mn)/levels)): the two fp32 steps add a few ulps
    s_lo = np.maximum((mx_lo - mn_hi) / levels * (1 - 2.0 ** -21), 0.0)
    s_hi = (mx_hi - mn_lo) / levels * (1 + 2.0 ** -21)
    gflag |= s_lo.astype(np.float16) != s_hi.astype(np.float16)
    # code: t = (yc - z16)/s16 near a half-integer
    s = s16.astype(np.float64)
    z = z16.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (gy - z[..., None]) / s[..., None]
        delta = eps_c.reshape(gy.shape) / s[..., None] + 2.0 ** -20 * (np.abs(t) + 1.0)
        frac = t - np.floor(t)
        near_half = np.abs(frac - 0.5) <= delta
    near_half = np.where((s == 0)[..., None], False, near_half)
    elem |= near_half.reshape(shp)
    return elem, gflag
