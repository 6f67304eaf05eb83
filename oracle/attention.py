"""Decode attention over the mixed BF16 / INT2 cache, by the plain definition.

[Summary 2.2B] (mixed-precision layout; the kernel unpacks, dequantises,
inverse-rotates and attends), [Abstract] ("custom INT2 attention kernel").
The oracle does not follow any kernel algebra: it rebuilds every INT2 token in
the original basis, k~ = y_hat_K R_K^T and v~ = y_hat_V R_V^T, keeps BF16
tokens as stored, and evaluates softmax(q K~^T / sqrt(d)) V~ in fp64.  (Softmax
scale 1/sqrt(d) is the reading taken; the pages do not state it.)
"""
from __future__ import annotations

import math

import numpy as np

from . import cache, quant, rotation


def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None):
    """out[g] = sum_t softmax_t(q_g . k_t * scale) v_t, fp64.  q [G,d], k,v [L,d]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    logits = q @ k.T * scale
    logits -= logits.max(axis=-1, keepdims=True)
    p = np.exp(logits)
    return (p @ v) / p.sum(axis=-1, keepdims=True)


def softmax_attention_loops(q, k, v, scale=None):
    """Same quantity with explicit Python loops (tiny inputs only)."""
    G, d = len(q), len(q[0])
    L = len(k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = []
    for g in range(G):
        logits = []
        for t in range(L):
            acc = 0.0
            for j in range(d):
                acc += float(q[g][j]) * float(k[t][j])
            logits.append(acc * scale)
        mx = max(logits)
        w = [math.exp(x - mx) for x in logits]
        tot = sum(w)
        row = []
        for j in range(d):
            acc = 0.0
            for t in range(L):
                acc += w[t] * float(v[t][j])
            row.append(acc / tot)
        out.append(row)
    return np.array(out)


def reconstruct(x: np.ndarray, r: np.ndarray, clip: float,
                levels: int = quant.INT2_MAX_CODE) -> np.ndarray:
    """Stored INT2 (or INT4: levels 15) form of tokens x [n, d], mapped back to
    the original basis: dequantise(quantise(x R)) R^T."""
    codes, s, z = quant.quantize(quant.rotate(x, r), clip, levels=levels)
    return quant.dequantize(codes, s, z) @ np.asarray(r, np.float64).T


def effective_kv(k: np.ndarray, v: np.ndarray, L: int, sink: int, window: int,
                 rk, rv, ck: float, cv: float, levels: int = quant.INT2_MAX_CODE):
    """Keys/values as the cache holds them for a sequence of length L."""
    k = np.asarray(k[:L], np.float64).copy()
    v = np.asarray(v[:L], np.float64).copy()
    m = cache.is_int2(np.arange(L), L, sink, window)
    if m.any():
        k[m] = reconstruct(k[m], rk, ck, levels)
        v[m] = reconstruct(v[m], rv, cv, levels)
    return k, v


def mixed_decode(q: np.ndarray, k: list, v: list, lens, rot: "cache.Rotations", *,
                 sink: int, window: int, gqa: int, levels: int = quant.INT2_MAX_CODE) -> np.ndarray:
    """out [B, Hq, d] for decode queries q [B, Hq, d]; query head hq reads KV
    head hq // gqa; k[b][h], v[b][h] are [L_b, d].  levels 15: the INT4 variant."""
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(lens[b])
        for h in range(Hq // gqa):
            ke, ve = effective_kv(k[b][h], v[b][h], L, sink, window,
                                  rot.rk[h], rot.rv[h], rot.ck[h], rot.cv[h], levels)
            out[b, h * gqa:(h + 1) * gqa] = softmax_attention(q[b, h * gqa:(h + 1) * gqa], ke, ve)
    return out


def mixed_multiquery(q: np.ndarray, k: list, v: list, lens, q_pos, rot: "cache.Rotations", *,
                     sink: int, window: int, gqa: int) -> np.ndarray:
    """Several query rows per sequence over the mixed cache (a chunk of new
    tokens, or tokens to verify): out [B, M, Hq, d] for q [B, M, Hq, d].  The
    cache holds L_b tokens in the form a sequence of length L_b stores them
    (BF16 sink and recent window, INT2 in between); row m of sequence b attends
    to the stored tokens at positions 0 .. q_pos[b][m] (causal)."""
    B, M, Hq, d = q.shape
    out = np.zeros((B, M, Hq, d))
    for b in range(B):
        L = int(lens[b])
        for h in range(Hq // gqa):
            ke, ve = effective_kv(k[b][h], v[b][h], L, sink, window,
                                  rot.rk[h], rot.rv[h], rot.ck[h], rot.cv[h])
            for m in range(M):
                n = int(q_pos[b][m]) + 1
                out[b, m, h * gqa:(h + 1) * gqa] = softmax_attention(q[b, m, h * gqa:(h + 1) * gqa],
                                                                     ke[:n], ve[:n])
    return out


def bf16_decode(q: np.ndarray, k: list, v: list, lens, *, gqa: int) -> np.ndarray:
    """All-BF16 cache: plain softmax attention over the stored bf16 values."""
    B, Hq, d = q.shape
    out = np.zeros((B, Hq, d))
    for b in range(B):
        L = int(lens[b])
        for h in range(Hq // gqa):
            out[b, h * gqa:(h + 1) * gqa] = softmax_attention(q[b, h * gqa:(h + 1) * gqa],
                                                              k[b][h][:L], v[b][h][:L])
    return out


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def calibrate(calib_q, calib_k, calib_v, variant: int, percentile: float = 99.9):
    """Per KV head rotations and clips from calibration data [Summary 2.2A]."""
    rk, rv, ck, cv = [], [], [], []
    for h in range(len(calib_k)):
        d = calib_k[h].shape[1]
        cq = rotation.query_covariance(calib_q[h]) if variant == rotation.OSCAR else None
        cs = (rotation.score_covariance(calib_q[h], calib_k[h], calib_v[h])
              if variant == rotation.OSCAR else None)
        r_k = rotation.composite_rotation(cq, d, variant).astype(np.float32)
        r_v = rotation.composite_rotation(cs, d, variant).astype(np.float32)
        rk.append(r_k)
        rv.append(r_v)
        ck.append(np.float32(rotation.clip_threshold(calib_k[h], r_k, percentile)))
        cv.append(np.float32(rotation.clip_threshold(calib_v[h], r_v, percentile)))
    return cache.Rotations(rk, rv, ck, cv)


FIDELITY_VARIANTS = (("oscar", rotation.OSCAR), ("hadamard_only", rotation.HADAMARD_ONLY),
                     ("unrotated", rotation.IDENTITY))


def fidelity_report(inst, *, sink: int, window: int, rotations: dict | None = None) -> dict:
    """How far the mixed cache moves attention from the all-BF16 cache, for the
    three rotations the pages compare: OSCAR, Hadamard only and none
    ([Summary 1], [Summary 4], [Abstract]).  Per variant:
      out_rel_l2  rel-L2 of the decode output against all-BF16 attention;
      k_rel_l2, v_rel_l2  rel-L2 of the INT2 tokens' reconstructed keys and
      values (original basis) against the stored bf16 ones.
    ``rotations`` optionally maps a variant name to its Rotations (default:
    ``calibrate`` on the instance's calibration sets).  The pages print no
    number for this synthetic setting, so only its special cases are pinned
    (no INT2 token gives zero error; values already on the four-level grid
    are reproduced exactly without rotation)."""
    w = inst.workload
    ref = bf16_decode(inst.q, inst.k, inst.v, inst.seq_lens, gqa=w.gqa)
    out = {}
    for name, var in FIDELITY_VARIANTS:
        rot = (rotations or {}).get(name) or calibrate(inst.calib_q, inst.calib_k, inst.calib_v, var)
        o = mixed_decode(inst.q, inst.k, inst.v, inst.seq_lens, rot, sink=sink, window=window,
                         gqa=w.gqa)
        dk = nk = dv = nv = 0.0
        for b, L in enumerate(inst.seq_lens):
            L = int(L)
            m = cache.is_int2(np.arange(L), L, sink, window)
            for h in range(w.num_kv_heads):
                ke, ve = effective_kv(inst.k[b][h], inst.v[b][h], L, sink, window,
                                      rot.rk[h], rot.rv[h], rot.ck[h], rot.cv[h])
                k0 = np.asarray(inst.k[b][h][:L], np.float64)[m]
                v0 = np.asarray(inst.v[b][h][:L], np.float64)[m]
                dk += float(((ke[m] - k0) ** 2).sum())
                nk += float((k0 ** 2).sum())
                dv += float(((ve[m] - v0) ** 2).sum())
                nv += float((v0 ** 2).sum())
        out[name] = {"out_rel_l2": rel_l2(o, ref),
                     "k_rel_l2": float(np.sqrt(dk / nk)) if nk > 0 else 0.0,
                     "v_rel_l2": float(np.sqrt(dv / nv)) if nv > 0 else 0.0}
    return out
