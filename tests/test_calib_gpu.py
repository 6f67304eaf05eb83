"""GPU parity of the calibration calls (C_Q, C_S, clip) against the oracle's
definitions in fp64, on the synthetic calibration recipe.

Tolerances follow from the arithmetic stated in include/oscar.h:
- C_Q: bf16 products are exact in fp32; each fp32 accumulator sums at most 128
  rows before it is flushed into a compensated pair, so
  |dC_ij| <= 128 * 2^-23 * A_ij with A = (1/(nG)) sum |x_i||x_j|; 2^-15 A is used.
- C_S: probabilities carried as a bf16 pair (2^-17 relative), ex2.approx
  (about 2^-22), O stored as a bf16 pair (2^-17), fp32 logits over d exact
  products, and the Gram bound above on O; by Cauchy-Schwarz A_ij <=
  sqrt(C_ii C_jj), so |dC_ij| <= 1e-4 sqrt(C_ii C_jj) is used.
- clip: for an exact rotation (identity, signed permutation) y is exact in
  fp32 and the selected order statistics are the oracle's, so the clip equals
  the oracle's up to the final fp32 rounding (1 ulp); for a full R each |y|
  moves by at most gamma_d max_{t,j} sum_i |x_ti||R_ij|, and so does the
  interpolated percentile.
"""
import dataclasses

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth
from oracle import rotation

pytestmark = pytest.mark.gpu


def _workload(hq, hkv, d, seed=0):
    return dataclasses.replace(synth.QWEN3_8B_32K if d == 128 else synth.TINY, num_q_heads=hq,
                               num_kv_heads=hkv, head_dim=d, seed=seed)


def _calib(hq, hkv, d, n, seed=0):
    inst = synth.draw_instance(_workload(hq, hkv, d, seed), n_calib=n, seq_lens=[1])
    G = hq // hkv
    q = np.zeros((n, hq, d), np.float32)
    for h in range(hkv):
        q[:, h * G:(h + 1) * G] = inst.calib_q[h]
    k = np.stack(inst.calib_k, axis=1)
    v = np.stack(inst.calib_v, axis=1)
    return inst, q, k, v


def _workspace(hkv, hq, d, n):
    t = H.torch()
    L = H.lib()
    nbytes = L.oscar_calibration_workspace_size(hkv, hq, d, n)
    assert nbytes > 0
    return t.empty(nbytes // 4 + 64, dtype=t.float32, device=H.DEV)


SHAPES = [  # (hq, hkv, d, n)
    (4, 1, 64, 2048),      # the tiny workload's calibration size
    (32, 8, 128, 1000),    # 8B shape, ragged against chunks and 64-row stages
    (2, 2, 128, 77),       # G = 1
    (16, 1, 64, 33),       # G = 16
    (8, 1, 128, 1),        # one token
]


@pytest.mark.parametrize("hq,hkv,d,n", SHAPES)
def test_query_covariance_matches_oracle(hq, hkv, d, n):
    t = H.torch()
    L = H.lib()
    inst, q, _, _ = _calib(hq, hkv, d, n)
    c = t.full((hkv, d, d), float("nan"), dtype=t.float64, device=H.DEV)
    L.oscar_query_covariance_device(H.bf16_tensor(q), hkv, c, _workspace(hkv, hq, d, n))
    got = c.cpu().numpy()
    for h in range(hkv):
        x = np.asarray(inst.calib_q[h], np.float64)
        ref = rotation.query_covariance(x)
        ax = np.abs(x.reshape(-1, d))
        bound = 2.0 ** -15 * (ax.T @ ax) / ax.shape[0] + 1e-300
        err = np.abs(got[h] - ref)
        assert np.all(err <= bound), (h, float(np.max(err / bound)))


@pytest.mark.parametrize("hq,hkv,d,n", [
    (4, 1, 64, 300),       # tiny shape
    (8, 2, 128, 700),      # G = 4 at d = 128, ragged against 32-token tiles and 64-key tiles
    (2, 2, 128, 130),      # G = 1: 128-token tiles, two key tiles in one CTA
    (16, 1, 64, 70),       # G = 16: 8-token tiles
    (4, 1, 64, 1),         # one token: O = v_0 for every head
])
def test_score_covariance_matches_oracle(hq, hkv, d, n):
    t = H.torch()
    L = H.lib()
    inst, q, k, v = _calib(hq, hkv, d, n, seed=1)
    c = t.full((hkv, d, d), float("nan"), dtype=t.float64, device=H.DEV)
    L.oscar_score_covariance_device(H.bf16_tensor(q), H.bf16_tensor(k), H.bf16_tensor(v), c,
                                    _workspace(hkv, hq, d, n))
    got = c.cpu().numpy()
    for h in range(hkv):
        ref = rotation.score_covariance(inst.calib_q[h], inst.calib_k[h], inst.calib_v[h])
        dg = np.sqrt(np.diag(ref))
        bound = 1e-4 * np.outer(dg, dg) + 1e-300
        err = np.abs(got[h] - ref)
        assert np.all(err <= bound), (h, float(np.max(err / bound)))
        if n == 1:
            v0 = np.asarray(inst.calib_v[h][0], np.float64)
            np.testing.assert_allclose(got[h], np.outer(v0, v0), rtol=1e-5, atol=1e-12)


def _clip_device(x, r, pct):
    t = H.torch()
    L = H.lib()
    n, hkv, d = x.shape
    out = t.full((hkv,), float("nan"), dtype=t.float32, device=H.DEV)
    rt = t.from_numpy(np.ascontiguousarray(r, np.float32)).to(H.DEV)
    L.oscar_clip_threshold_device(H.bf16_tensor(x), rt, pct, out, _workspace(hkv, hkv, d, n))
    return out.cpu().numpy()


def _ulp_diff(a, b):
    return abs(int(np.float32(a).view(np.int32)) - int(np.float32(b).view(np.int32)))


@pytest.mark.parametrize("d,hkv,n", [(64, 1, 2048), (128, 8, 1000), (128, 2, 3), (64, 1, 1)])
@pytest.mark.parametrize("pct", [99.9, 50.0, 0.0, 100.0])
def test_clip_exact_rotations_select_the_oracle_order_statistics(d, hkv, n, pct):
    inst, _, k, _ = _calib(hkv, hkv, d, n, seed=2)
    rng = np.random.default_rng(5)
    rots = []
    for h in range(hkv):
        if h % 2 == 0:
            rots.append(np.eye(d, dtype=np.float32))
        else:   # signed permutation: exact in fp32
            p = np.zeros((d, d), np.float32)
            p[np.arange(d), rng.permutation(d)] = rng.choice([-1.0, 1.0], d)
            rots.append(p)
    r = np.stack(rots)
    got = _clip_device(k, r, pct)
    for h in range(hkv):
        ref = rotation.clip_threshold(k[:, h], r[h], pct)
        assert _ulp_diff(got[h], ref) <= 1, (h, got[h], ref)


def test_clip_with_many_ties():
    # integer-valued data: long runs of equal |y|, so the two order statistics
    # fall inside and at the end of runs of equals
    rng = np.random.default_rng(3)
    n, hkv, d = 997, 2, 64
    x = rng.integers(-4, 5, size=(n, hkv, d)).astype(np.float32)
    r = np.stack([np.eye(d, dtype=np.float32)] * hkv)
    for pct in (99.9, 12.5, 33.3, 99.99, 100.0):
        got = _clip_device(x, r, pct)
        for h in range(hkv):
            ref = rotation.clip_threshold(x[:, h], r[h], pct)
            assert _ulp_diff(got[h], ref) <= 1, (pct, h, got[h], ref)


@pytest.mark.parametrize("d,hkv,n", [(64, 1, 2048), (128, 8, 1500)])
def test_clip_full_rotation_within_fp32_bound(d, hkv, n):
    inst, _, k, v = _calib(hkv * 4, hkv, d, n, seed=4)
    rot = H.oracle_rotations(inst)
    gamma = d * 2.0 ** -24 / (1 - d * 2.0 ** -24)
    for x, rs in ((k, rot.rk), (v, rot.rv)):
        r = np.stack([np.asarray(a, np.float32) for a in rs])
        got = _clip_device(x, r, 99.9)
        for h in range(hkv):
            ref = rotation.clip_threshold(x[:, h], r[h], 99.9)
            bound = gamma * float(np.max(np.abs(x[:, h]).astype(np.float64) @ np.abs(r[h])))
            bound += abs(ref) * 2.0 ** -23
            assert abs(float(got[h]) - ref) <= bound, (h, float(got[h]), ref, bound)


def test_full_size_calibration_8b_shape():
    """The 8B layer at the calibration size the bench times (32/8 heads, d = 128):
    C_Q at n = 8192 against the oracle for every KV head; C_S at n = 2048 for
    two KV heads (the oracle's causal attention is O(n^2) in fp64); the clips of
    K under the oracle's R for every head."""
    t = H.torch()
    L = H.lib()
    hq, hkv, d = 32, 8, 128
    inst, q, k, v = _calib(hq, hkv, d, 8192, seed=0)
    ws = _workspace(hkv, hq, d, 8192)
    c = t.empty((hkv, d, d), dtype=t.float64, device=H.DEV)
    L.oscar_query_covariance_device(H.bf16_tensor(q), hkv, c, ws)
    got = c.cpu().numpy()
    for h in range(hkv):
        x = np.asarray(inst.calib_q[h], np.float64)
        ax = np.abs(x.reshape(-1, d))
        bound = 2.0 ** -15 * (ax.T @ ax) / ax.shape[0]
        assert np.all(np.abs(got[h] - rotation.query_covariance(x)) <= bound), h
    n = 2048
    ws2 = _workspace(hkv, hq, d, n)
    L.oscar_score_covariance_device(H.bf16_tensor(q[:n]), H.bf16_tensor(k[:n]),
                                    H.bf16_tensor(v[:n]), c, ws2)
    got = c.cpu().numpy()
    for h in (0, 5):
        ref = rotation.score_covariance(inst.calib_q[h][:n], inst.calib_k[h][:n], inst.calib_v[h][:n])
        dg = np.sqrt(np.diag(ref))
        assert np.all(np.abs(got[h] - ref) <= 1e-4 * np.outer(dg, dg)), h
    rot = H.oracle_rotations(inst, n_calib=1024)
    r = np.stack([np.asarray(a, np.float32) for a in rot.rk])
    clip = _clip_device(k, r, 99.9)
    gamma = d * 2.0 ** -24 / (1 - d * 2.0 ** -24)
    for h in range(hkv):
        ref = rotation.clip_threshold(k[:, h], r[h], 99.9)
        bound = gamma * float(np.max(np.abs(k[:, h]).astype(np.float64) @ np.abs(r[h])))
        assert abs(float(clip[h]) - ref) <= bound + abs(ref) * 2.0 ** -23, h
