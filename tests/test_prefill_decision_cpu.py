"""The tensor-core prefill's fast code decision, restated in float32 and checked
against the oracle's quantiser (Technical Summary 2.2B: rotate, clip, quantise).

The kernel's fast path, per group of 32 rotated values y:
  - min and max over the raw values, then only those two clipped (clipping is
    monotone, so they equal the extremes of the clipped group);
  - s16 = fp16(fp32(mx - mn) / top), z16 = fp16(mn), as the definition;
  - t = (y - z16) times (a reciprocal of s16 that may be off by up to two ulp,
    times fp32(1/top)), saturated to [0, 1]; the quotient top * t is rounded by
    one fused multiply-add with 1.5 * 2^23 (the code is then the low mantissa
    bits), and a second fused multiply-add gives its distance from that integer;
  - the group goes to the correctly rounded division whenever a clamped
    quotient lies within 6.4e-5 of a half-integer.
A fused multiply-add a * b + c of float32 values is restated as the float64
product and sum rounded once to float32 (the product of a float32 t and a
small integer top is exact in float64, and so is its sum with 1.5 * 2^23).
Wherever a group is not flagged, every code must equal the definition's, for
values inside and beyond the clip threshold alike."""
import numpy as np
import pytest

from oracle import quant

MAGIC = np.float32(12582912.0)           # 1.5 * 2^23
MARGIN = np.float32(0.5) - np.float32(6.4e-5)


def fast_decide(y, clip, top, rng):
    y = np.asarray(y, np.float32)
    c = np.float32(clip)
    mn = np.minimum(np.maximum(y.min(axis=1), -c), c)
    mx = np.minimum(np.maximum(y.max(axis=1), -c), c)
    s16 = (np.float32(mx - mn) / np.float32(top)).astype(np.float32).astype(np.float16)
    z16 = mn.astype(np.float16)
    sf = s16.astype(np.float32)
    zf = z16.astype(np.float32)
    live = sf != 0
    with np.errstate(divide="ignore"):
        inv = np.where(live, np.float32(1.0) / np.where(live, sf, np.float32(1.0)), np.float32(0.0))
    # an approximate reciprocal: the correctly rounded one moved by up to two ulp
    steps = rng.integers(-2, 3, size=inv.shape).astype(np.int32)
    inv = np.where(live, (inv.view(np.int32) + steps).view(np.float32), np.float32(0.0))
    inv_top = (inv * np.float32(1.0 / top)).astype(np.float32)
    q = ((y - zf[:, None]).astype(np.float32) * inv_top[:, None]).astype(np.float32)
    t = np.minimum(np.maximum(q, np.float32(0.0)), np.float32(1.0)).astype(np.float32)
    kt = t.astype(np.float64) * float(top)                    # exact
    m = (kt + float(MAGIC)).astype(np.float32)                 # one rounding
    codes = (m.view(np.uint32) & np.uint32(0xF)).astype(np.uint8)
    r = (m - MAGIC).astype(np.float32)                         # exact
    dist = (kt - r.astype(np.float64)).astype(np.float32)      # one rounding
    near = (np.abs(dist) > MARGIN).any(axis=1) & live
    return codes, s16, z16, near


def groups(rng, n):
    """Groups of 32 values: ordinary spreads over many magnitudes, outliers far
    beyond the clip threshold, ranges small enough for a subnormal fp16 scale,
    constant groups, and groups entirely beyond the threshold."""
    clip = 3.0
    base = rng.standard_normal((n, 32)) * np.exp(rng.uniform(-6, 2, (n, 1)))
    kind = rng.integers(0, 5, n)
    y = base.copy()
    out = kind == 1
    y[out, rng.integers(0, 32, out.sum())] = rng.choice([-1, 1], out.sum()) * rng.uniform(3.5, 40, out.sum())
    tiny = kind == 2
    y[tiny] = rng.uniform(-1, 1, (tiny.sum(), 1)) + rng.standard_normal((tiny.sum(), 32)) * 1e-6
    const = kind == 3
    y[const] = rng.uniform(-2, 2, (const.sum(), 1))
    beyond = kind == 4
    y[beyond] = rng.choice([-1, 1], (beyond.sum(), 1)) * rng.uniform(3.2, 9, (beyond.sum(), 32))
    return y.astype(np.float32), clip


@pytest.mark.parametrize("top", [quant.INT2_MAX_CODE, quant.INT4_MAX_CODE])
def test_fast_decision_equals_definition_where_unflagged(top):
    rng = np.random.default_rng(top)
    y, clip = groups(rng, 20000)
    codes, s16, z16, near = fast_decide(y, clip, top, rng)
    ref_codes, ref_s, ref_z = quant.quantize(y[:, None, :].reshape(-1, 32), clip, levels=top)
    np.testing.assert_array_equal(s16.view(np.uint16), ref_s.reshape(-1).view(np.uint16))
    np.testing.assert_array_equal(z16.view(np.uint16), ref_z.reshape(-1).view(np.uint16))
    keep = ~near
    np.testing.assert_array_equal(codes[keep], ref_codes[keep])
    # the exact path stays the rare one on such data
    assert near.mean() < 0.05, near.mean()


def test_clamp_then_round_equals_round_then_clamp():
    """Rounding a quotient clamped to integer bounds gives the clamped rounded
    quotient, ties included (round-half-even on both sides)."""
    q = np.concatenate([np.linspace(-3, 20, 200001, dtype=np.float32),
                        np.arange(-2, 19, dtype=np.float32) + np.float32(0.5)])
    for top in (3, 15):
        a = (np.minimum(np.maximum(q, 0), top).astype(np.float32) + MAGIC).view(np.uint32) & 0xF
        b = np.clip(np.rint(q), 0, top).astype(np.uint32)
        np.testing.assert_array_equal(a, b)
