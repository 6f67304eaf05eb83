"""GPU parity on the method's edge cases: magnitudes far from the unit-scale
workloads, groups whose range is zero (constant, all-zero or fully clipped
inputs), a tiny clip threshold, and non-finite inputs.

"Technical Summary: OSCAR ...", section 2.2A.4 (the clip) and section 2.2B
(INT2 storage after rotation and clipping).  Stored pools are compared with the
oracle's placement (bit for bit where the rotation is exact), the kernels'
traced rotated values feed the decision check under the OSCAR rotation, and
attention is compared with the oracle's attention over the stored pools at the
parity tolerances (rel-L2 5e-3; max-abs 1e-2 beyond the bf16 store's rounding).
"""
import dataclasses

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth
from oracle import cache as ocache, quant

pytestmark = pytest.mark.gpu

W8 = synth.QWEN3_8B_32K


def _scaled(inst, fk=1.0, fv=1.0, fq=1.0):
    """The instance with keys, values and queries (calibration sets included)
    multiplied by fk, fv, fq and rounded to bf16 again."""
    r = synth.bf16_round

    def each(lst, f):
        return [[r(np.asarray(x) * np.float32(f)) for x in hs] for hs in lst]
    return dataclasses.replace(
        inst, k=each(inst.k, fk), v=each(inst.v, fv), q=r(inst.q * np.float32(fq)),
        calib_q=[r(c * np.float32(fq)) for c in inst.calib_q],
        calib_k=[r(c * np.float32(fk)) for c in inst.calib_k],
        calib_v=[r(c * np.float32(fv)) for c in inst.calib_v])


def _identity(d, hkv, ck=9.0, cv=4.0):
    eye = [np.eye(d, dtype=np.float32) for _ in range(hkv)]
    return ocache.Rotations(eye, list(eye), [np.float32(ck)] * hkv, [np.float32(cv)] * hkv)


def _exact_pools_equal(cache, exp):
    got2, gotb = H.pools(cache)
    np.testing.assert_array_equal(got2[exp.int2_defined], exp.int2[exp.int2_defined])
    np.testing.assert_array_equal(gotb[exp.bf16_defined], exp.bf16[exp.bf16_defined])


@pytest.mark.parametrize("fk,fv,fq", [(1e-3, 1, 1), (1e2, 1, 1), (1, 1e-3, 1), (1, 1e2, 1),
                                      (1, 1, 1e-3), (1, 1, 1e2), (1e-3, 1e-3, 1e-3),
                                      (1e2, 1e2, 1e2)])
def test_magnitude_sweep(fk, fv, fq):
    """Keys, values and queries scaled by 1e-3 or 1e2 (rotations and clips
    calibrated on the scaled data): the prefill's decisions stay exact given
    its rotated values, and decode attention stays within the parity
    tolerances, for the call and for the fused step."""
    t = H.torch()
    L = H.lib()
    lens = [2000, 700]
    inst = _scaled(synth.draw_instance(W8, n_calib=512, seq_lens=lens), fk, fv, fq)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=128)
    y, where = H.prefill_trace(cache, inst)
    rows = {b: (np.arange(n), y[s:s + n]) for b, (s, n) in where.items()}
    st = H.check_traced(cache, pp, inst, rot, rows, H.kappa_tc(W8.head_dim), lens=lens, sink=4,
                        window=128)
    got = H.decode(cache, inst.q, lens)
    ref = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=128, gqa=W8.gqa)
    err, rel = H.check_close(got, ref, f"decode at scale k{fk} v{fv} q{fq}")
    H.report(f"magnitude[k{fk},v{fv},q{fq}]", max_abs=err, rel_l2=rel,
             beyond_bf16_rounding=H.LAST_CHECK["excess"], **st)
    assert np.isfinite(got).all()
    assert H.status(cache) == 0


def _edge_tokens(inst, d, hkv, clip_k):
    """Plant zero-range groups in sequence 0 (INT2 positions 10..15): an
    all-zero token, a constant token, a group entirely beyond the clip, a group
    alternating beyond +-clip, and a group constant inside one 32-channel block
    while the rest of the token varies."""
    k = [x.copy() for x in inst.k[0]]
    v = [x.copy() for x in inst.v[0]]
    for h in range(hkv):
        for a in (k[h], v[h]):
            a[10] = 0.0
            a[11] = 1.5
            a[12, 0:32] = 4.0 * clip_k
            a[13, 32:64] = np.where(np.arange(32) % 2 == 0, 8.0 * clip_k, -8.0 * clip_k)
            a[14, 64:96] = -0.75
            a[15, :] = synth.bf16_round(np.linspace(-3.0, 3.0, d).astype(np.float32))
    return dataclasses.replace(inst, k=[k] + inst.k[1:], v=[v] + inst.v[1:])


@pytest.mark.parametrize("misalign", [False, True])
@pytest.mark.parametrize("clip", [9.0, 1e-3])
def test_zero_range_and_clipped_groups(misalign, clip):
    """With an exact (identity) rotation every stored byte is fixed: zero-range
    groups store s = 0 and codes 0 with z the group's value, fully clipped
    groups store z = +-clip; with a tiny clip almost every value is clipped.
    Prefill (tensor-core or CUDA-core kernel), then ten append steps, then
    decode against the oracle over the stored pools."""
    t = H.torch()
    L = H.lib()
    d, hkv = W8.head_dim, W8.num_kv_heads
    lens1 = np.array([300, 260])
    steps = 10
    lens0 = lens1 - steps
    inst = _edge_tokens(synth.draw_instance(W8, n_calib=32, seq_lens=lens1), d, hkv, 9.0)
    rot = _identity(d, hkv, clip, clip)
    cache, pp = H.make_cache(inst, rot, window=128, lens=lens0, growth=steps)
    H.prefill(cache, inst, lens=lens0, misalign=misalign)
    _exact_pools_equal(cache, H.expected(inst, rot, pp, window=128, lens=lens0))
    for s in range(steps):
        cur = lens0 + s + 1
        kn = np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        vn = np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        L.oscar_quantize_append(cache, H.bf16_tensor(kn), H.bf16_tensor(vn),
                                t.from_numpy(cur.astype(np.int32)).to(H.DEV))
    exp = H.expected(inst, rot, pp, window=128, lens=lens1)
    _exact_pools_equal(cache, exp)
    # the planted groups really are zero-range ones
    c, s16, z16 = quant.quantize(quant.rotate(inst.k[0][0][10:13], rot.rk[0]), rot.ck[0])
    assert (s16[:2] == 0).all() and s16[2, 0] == 0
    got = H.decode(cache, inst.q, lens1)
    ref = H.attention_from_pools(cache, pp, inst.q, lens1, rot, sink=4, window=128, gqa=W8.gqa)
    H.check_close(got, ref, f"decode over zero-range groups, clip {clip}")
    assert H.status(cache) == 0


def _plant_nonfinite(inst, positions):
    """NaN and infinities at the given positions of sequence 0 (KV heads 0, 1)."""
    k = [x.copy() for x in inst.k[0]]
    v = [x.copy() for x in inst.v[0]]
    pa, pb, pc = positions
    k[0][pa, 5] = np.nan
    v[0][pb, 70] = np.inf
    k[1][pc, 127] = -np.inf
    v[1][pc, 0] = np.nan
    return dataclasses.replace(inst, k=[k] + inst.k[1:], v=[v] + inst.v[1:])


@pytest.mark.parametrize("misalign", [False, True])
@pytest.mark.parametrize("rotation", ["identity", "oscar"])
def test_nonfinite_inputs_become_zero_groups(misalign, rotation):
    """A NaN or an infinity in an INT2 token's key or value: every group of that
    token-head is stored as a zero group and OSCAR_DEVERR_NONFINITE is set; the
    other tokens are placed as usual, and attention over the cache stays finite
    and matches the oracle over the stored pools.  A token that leaves the
    window carrying a NaN through the append is handled the same way."""
    t = H.torch()
    L = H.lib()
    d, hkv = W8.head_dim, W8.num_kv_heads
    lens1 = np.array([400, 333])
    lens0 = lens1 - 3
    W = 128
    # positions 30, 31 are INT2 from the prefill on; 270 is a BF16 token at the
    # prefill's length 397 and leaves the window at length 399 (second step)
    inst = _plant_nonfinite(synth.draw_instance(W8, n_calib=256, seq_lens=lens1), (30, 31, 270))
    rot = _identity(d, hkv) if rotation == "identity" else H.oracle_rotations(
        synth.draw_instance(W8, n_calib=256, seq_lens=[16]))
    cache, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=3)
    H.prefill(cache, inst, lens=lens0, misalign=misalign)
    assert H.status(cache) & L.DEVERR_NONFINITE
    cache.status.zero_()
    for s in range(3):
        cur = lens0 + s + 1
        kn = np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        vn = np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        L.oscar_quantize_append(cache, H.bf16_tensor(kn), H.bf16_tensor(vn),
                                t.from_numpy(cur.astype(np.int32)).to(H.DEV))
        t.cuda.synchronize()
        if cur[0] - 1 - W == 270:   # the planted token left the window in this step
            assert H.status(cache) & L.DEVERR_NONFINITE
    # every group of the planted token-heads is a zero group
    for b, h, pos in ((0, 0, 30), (0, 0, 31), (0, 1, 270)):
        kc, ks, kz, vc, vs, vz = H.stored_int2(cache, pp, b, h, [pos], d)
        x_k = np.asarray(inst.k[b][h][pos])
        x_v = np.asarray(inst.v[b][h][pos])
        if not np.isfinite(x_k).all():
            assert not kc.any() and not ks.view(np.uint16).any() and not kz.view(np.uint16).any()
        if not np.isfinite(x_v).all():
            assert not vc.any() and not vs.view(np.uint16).any() and not vz.view(np.uint16).any()
    exp = H.expected(inst, rot, pp, window=W, lens=lens1,
                     kappa=None if rotation == "identity" else H.kappa_tc(d))
    if rotation == "identity":
        _exact_pools_equal(cache, exp)
    else:
        H.compare_pools(cache, exp)
    got = H.decode(cache, inst.q, lens1)
    assert np.isfinite(got).all()
    ref = H.attention_from_pools(cache, pp, inst.q, lens1, rot, sink=4, window=W, gqa=W8.gqa)
    H.check_close(got, ref, f"decode over zero groups ({rotation})")


def test_nan_in_bf16_window_reaches_only_its_heads():
    """A NaN in a BF16 (recent-window) token is stored as given; the output of
    the query heads that read its KV head is NaN, every other output matches
    the oracle over the stored pools."""
    d, hkv, G = W8.head_dim, W8.num_kv_heads, W8.gqa
    lens = np.array([500, 300])
    inst = synth.draw_instance(W8, n_calib=128, seq_lens=lens)
    k = [x.copy() for x in inst.k[0]]
    k[3][lens[0] - 5, 17] = np.nan           # inside the recent window of sequence 0
    inst = dataclasses.replace(inst, k=[k] + inst.k[1:])
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=128)
    H.prefill(cache, inst)
    assert H.status(cache) == 0              # BF16 tokens are stored as given
    got = H.decode(cache, inst.q, lens)
    nan_cols = np.arange(3 * G, 4 * G)
    assert np.isnan(got[0, nan_cols]).all()
    keep = np.ones(got.shape[:2], bool)
    keep[0, nan_cols] = False
    assert np.isfinite(got[keep]).all()
    ref = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=128, gqa=G)
    H.check_close(got[keep], ref[keep], "decode beside a NaN in the window")
