"""Pins for the oracle's mixed-cache decode attention (Technical Summary 2.2B)."""
import math

import numpy as np
import pytest

from int2_rotated_kv_gb300 import synth
from oracle import attention, cache, layout, quant, rotation


def _rand(rng, *shape):
    return synth.bf16_round(rng.standard_normal(shape).astype(np.float32))


def test_vectorised_matches_loops():
    rng = np.random.default_rng(0)
    q, k, v = _rand(rng, 3, 64), _rand(rng, 37, 64), _rand(rng, 37, 64)
    np.testing.assert_allclose(attention.softmax_attention(q, k, v),
                               attention.softmax_attention_loops(q, k, v), rtol=1e-12, atol=1e-13)


def test_single_token_and_uniform_attention():
    rng = np.random.default_rng(1)
    q, k, v = _rand(rng, 2, 64), _rand(rng, 1, 64), _rand(rng, 1, 64)
    np.testing.assert_allclose(attention.softmax_attention(q, k, v), np.repeat(v, 2, 0), rtol=1e-15)
    k = np.zeros((9, 64))
    v = _rand(rng, 9, 64)
    np.testing.assert_allclose(attention.softmax_attention(q, k, v)[0], v.astype(np.float64).mean(0), rtol=1e-12)


def test_region_rule():
    L, S, W = 200, 4, 64
    m = cache.is_int2(np.arange(L), L, S, W)
    assert not m[:S].any() and not m[L - W:].any() and m[S:L - W].all()
    assert not cache.is_int2(np.arange(60), 60, S, W).any()     # L <= S + W: all BF16


def test_all_bf16_window_reduces_to_plain_attention():
    w = synth.TINY
    inst = synth.draw_instance(w, n_calib=64, seq_lens=[50])
    rot = cache.Rotations([np.eye(64, dtype=np.float32)], [np.eye(64, dtype=np.float32)],
                          [np.float32(100)], [np.float32(100)])
    out = attention.mixed_decode(inst.q, inst.k, inst.v, inst.seq_lens, rot, sink=4, window=64,
                                 gqa=4)
    ref = np.stack([attention.softmax_attention_loops(inst.q[0], inst.k[0][0], inst.v[0][0])])
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


def test_brute_force_tiny_mixed_cache():
    """L = 40 with S = 4, W = 8: tokens 4..31 are INT2; rebuild them by hand
    (rotate, quantise, dequantise, rotate back) and attend with loops."""
    rng = np.random.default_rng(2)
    d, L, S, W = 64, 40, 4, 8
    k, v, q = _rand(rng, L, d), _rand(rng, L, d), _rand(rng, 2, d)
    r = rotation.composite_rotation(np.cov(rng.standard_normal((256, d)).T), d).astype(np.float32)
    ck, cv = np.float32(2.5), np.float32(2.0)
    ke, ve = k.astype(np.float64).copy(), v.astype(np.float64).copy()
    for t in range(S, L - W):
        for x, c, dst in ((k, ck, ke), (v, cv, ve)):
            y = np.array([sum(float(x[t, i]) * float(r[i, j]) for i in range(d)) for j in range(d)])
            codes, s, z = quant.quantize(y[None], c)
            yh = quant.dequantize(codes, s, z)[0]
            dst[t] = [sum(yh[j] * float(r[i, j]) for j in range(d)) for i in range(d)]
    ref = attention.softmax_attention_loops(q, ke, ve)
    rot = cache.Rotations([r], [r], [ck], [cv])
    out = attention.mixed_decode(q[None], [[k]], [[v]], [L], rot, sink=S, window=W, gqa=2)[0]
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-11)


def test_pre_post_rotation_form_equals_definition():
    """(q R_K) . y_hat^T = q . (y_hat R_K^T)^T and (sum p y_hat) R_V^T = sum p (y_hat R_V^T):
    the kernel's algebra reaches the definition by associativity, R need not be
    orthogonal."""
    rng = np.random.default_rng(3)
    d, n = 64, 30
    rk = rng.standard_normal((d, d)).astype(np.float32)
    rv = rng.standard_normal((d, d)).astype(np.float32)
    x = _rand(rng, n, d)
    q = _rand(rng, 4, d)
    ck = kc = np.float32(50.0)
    yk = quant.dequantize(*quant.quantize(quant.rotate(x, rk), ck))
    yv = quant.dequantize(*quant.quantize(quant.rotate(x[::-1], rv), kc))
    kt, vt = yk @ rk.T.astype(np.float64), yv @ rv.T.astype(np.float64)
    ref = attention.softmax_attention(q, kt, vt)
    logits = (q @ rk.astype(np.float64)) @ yk.T / math.sqrt(d)
    p = np.exp(logits - logits.max(1, keepdims=True))
    alt = (p @ yv) @ rv.T.astype(np.float64) / p.sum(1, keepdims=True)
    np.testing.assert_allclose(alt, ref, rtol=1e-10, atol=1e-12)


def test_orthogonal_rotation_without_quantisation_changes_nothing():
    rng = np.random.default_rng(4)
    d = 128
    r = rotation.composite_rotation(np.diag(np.arange(d, 0, -1.0)), d)
    q, k, v = _rand(rng, 4, d), _rand(rng, 50, d), _rand(rng, 50, d)
    a = attention.softmax_attention(q @ r, k @ r, v @ r) @ r.T
    np.testing.assert_allclose(a, attention.softmax_attention(q, k, v), rtol=1e-10, atol=1e-12)


def test_expected_pools_roundtrip_and_prefix_sharing():
    """Pools written for two sequences sharing their first two pages hold the
    same bytes on the shared pages, and unpack back to the quantiser's output."""
    rng = np.random.default_rng(5)
    d, S, W, H = 64, 4, 16, 1
    L0, L1 = 70, 85
    shared_k, shared_v = _rand(rng, 32, d), _rand(rng, 32, d)
    k = [[np.concatenate([shared_k, _rand(rng, L0 - 32, d)])],
         [np.concatenate([shared_k, _rand(rng, L1 - 32, d)])]]
    v = [[np.concatenate([shared_v, _rand(rng, L0 - 32, d)])],
         [np.concatenate([shared_v, _rand(rng, L1 - 32, d)])]]
    r = np.linalg.qr(rng.standard_normal((d, d)))[0].astype(np.float32)
    rot = cache.Rotations([r], [r], [np.float32(3)], [np.float32(3)])
    it = np.array([[0, 1, 2, 3, 4, 5], [0, 1, 6, 7, 8, 9]], np.int32)
    bt = np.array([[0, -1, -1, 1, 2, -1], [0, -1, -1, -1, 3, 4]], np.int32)
    exp = cache.expected_pools(k, v, [L0, L1], rot, sink=S, window=W, d=d, hkv=H,
                               int2_table=it, bf16_table=bt, num_int2_pages=10,
                               num_bf16_pages=5)
    blk = layout.int2_block_bytes(d)
    kc, ks, kz, vc, vs, vz = layout.unpack_int2_block(exp.int2[blk:2 * blk], d)
    codes, s, z = quant.quantize(quant.rotate(shared_k[16:32], r), 3)
    np.testing.assert_array_equal(kc, codes)
    np.testing.assert_array_equal(ks, s)
    assert exp.int2_defined[blk:2 * blk].all()          # page 1: tokens 16..31, all INT2
    tb = layout.tables(d)
    np.testing.assert_array_equal(exp.int2_defined[:blk], tb['owner'] >= S)   # page 0: sink slots unused
    bk, bv = layout.unpack_bf16_block(exp.bf16[:32 * d], d)
    np.testing.assert_array_equal(bk[:S], synth.bf16_bits(shared_k[:S]))


# --------------------------------------------------------- several query rows

def test_multiquery_single_row_at_the_end_is_decode():
    """One row per sequence at position L - 1 is exactly the decode attention."""
    inst = synth.draw_instance(synth.TINY, n_calib=128, seq_lens=[300, 200])
    rot = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    q4 = inst.q[:, None]
    got = attention.mixed_multiquery(q4, inst.k, inst.v, inst.seq_lens,
                                     [[L - 1] for L in inst.seq_lens], rot, sink=4, window=64,
                                     gqa=4)
    ref = attention.mixed_decode(inst.q, inst.k, inst.v, inst.seq_lens, rot, sink=4, window=64,
                                 gqa=4)
    np.testing.assert_array_equal(got[:, 0], ref)


def test_multiquery_all_bf16_is_causal_attention_by_loops():
    """Identity rotation with the window covering the context: row m attends to
    tokens 0 .. q_pos (causal), checked against explicit loops."""
    rng = np.random.default_rng(5)
    L, d, G, M = 40, 8, 2, 4
    k = [[rng.standard_normal((L, d))]]
    v = [[rng.standard_normal((L, d))]]
    q = rng.standard_normal((1, M, G, d))
    pos = [[36, 37, 38, 39]]
    eye = np.eye(d, dtype=np.float32)
    rot = cache.Rotations([eye], [eye], [np.float32(1)], [np.float32(1)])
    got = attention.mixed_multiquery(q, k, v, [L], pos, rot, sink=0, window=L, gqa=G)
    for m in range(M):
        n = pos[0][m] + 1
        ref = attention.softmax_attention_loops(q[0, m], k[0][0][:n], v[0][0][:n])
        np.testing.assert_allclose(got[0, m], ref, rtol=1e-12, atol=1e-12)


def test_multiquery_ignores_tokens_after_the_row():
    """Changing tokens after a row's position changes nothing for that row."""
    inst = synth.draw_instance(synth.TINY, n_calib=128, seq_lens=[300])
    rot = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    q = np.stack([inst.q[0], inst.q[0]])[None]          # two rows, same query
    pos = [[250, 299]]
    a = attention.mixed_multiquery(q, inst.k, inst.v, [300], pos, rot, sink=4, window=64, gqa=4)
    k2 = [[inst.k[0][0].copy()]]
    v2 = [[inst.v[0][0].copy()]]
    k2[0][0][260:] += 3.0
    v2[0][0][260:] -= 2.0
    b = attention.mixed_multiquery(q, k2, v2, [300], pos, rot, sink=4, window=64, gqa=4)
    np.testing.assert_array_equal(a[0, 0], b[0, 0])      # row at 250 does not see 260..
    assert np.abs(a[0, 1] - b[0, 1]).max() > 1e-3       # row at 299 does


def test_fidelity_report_special_cases():
    """The fidelity report's pins (the pages print no number for it): with no
    INT2 token every variant reproduces all-BF16 attention exactly; with keys
    and values already on a four-level grid (every group spanning 0..3, so
    s = 1, z = 0 and every code exact) the unrotated cache loses nothing; a
    quantised cache that does lose information shows a positive error."""
    w = synth.TINY
    inst = synth.draw_instance(w, n_calib=128, seq_lens=[60])       # 60 <= 4 + 64: all BF16
    rep = attention.fidelity_report(inst, sink=4, window=64)
    for name, _ in attention.FIDELITY_VARIANTS:
        assert rep[name] == {"out_rel_l2": 0.0, "k_rel_l2": 0.0, "v_rel_l2": 0.0}
    inst = synth.draw_instance(w, n_calib=128, seq_lens=[300])
    rng = np.random.default_rng(9)
    grid = []
    for _ in range(2):
        a = rng.integers(0, 4, size=(300, 64)).astype(np.float32)
        a[:, 0::32] = 0.0
        a[:, 1::32] = 3.0                     # every group spans exactly [0, 3]
        grid.append([a])
    inst_g = __import__("dataclasses").replace(inst, k=[grid[0]], v=[grid[1]])
    eye = [np.eye(64, dtype=np.float32)]
    rot_id = cache.Rotations(eye, eye, [np.float32(3.0)], [np.float32(3.0)])
    rep = attention.fidelity_report(inst_g, sink=4, window=64, rotations={"unrotated": rot_id})
    assert rep["unrotated"] == {"out_rel_l2": 0.0, "k_rel_l2": 0.0, "v_rel_l2": 0.0}
    rep = attention.fidelity_report(inst, sink=4, window=64, rotations={"unrotated": rot_id})
    assert rep["unrotated"]["k_rel_l2"] > 0.1 and rep["unrotated"]["out_rel_l2"] > 0.0
    for name, _ in attention.FIDELITY_VARIANTS:
        assert 0.0 < rep[name]["v_rel_l2"] < 1.0
