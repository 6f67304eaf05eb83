"""Offline calibration: covariances, eigenbasis, Hadamard, bit reversal, clip.

[Summary 2.1] and [Summary 2.2A] (steps 1-4); [Abstract] ("fixed rotations and
clipping thresholds").  Convention: activations are row vectors and a rotation
acts on the right, y = x R, so the inverse is x = y R^T for orthogonal R.
"""
from __future__ import annotations

import numpy as np

OSCAR, HADAMARD_ONLY, IDENTITY = 0, 1, 2


def query_covariance(q: np.ndarray) -> np.ndarray:
    """C_Q = (1/N) sum_n q_n^T q_n  [Summary 2.1 (keys), 2.2A.1].

    ``q`` is [N, G, d]: the G query heads that read one KV head are pooled (the
    pages are silent on grouped-query attention; pooling is the reading taken),
    so the normaliser is N*G.
    """
    q = np.asarray(q, dtype=np.float64)
    n = q.shape[0] * q.shape[1]
    flat = q.reshape(n, q.shape[-1])
    return flat.T @ flat / n


def causal_scores(qh: np.ndarray, k: np.ndarray) -> np.ndarray:
    """Post-softmax causal attention probabilities S (N x N) for one query head,
    scale 1/sqrt(d).  S in C_S is read as these probabilities [Summary 2.1]."""
    n, d = k.shape
    logits = (np.asarray(qh, np.float64) @ np.asarray(k, np.float64).T) / np.sqrt(d)
    mask = np.tril(np.ones((n, n), dtype=bool))
    logits = np.where(mask, logits, -np.inf)
    logits -= logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    return p / p.sum(axis=1, keepdims=True)


def score_covariance(q: np.ndarray, k: np.ndarray, v: np.ndarray, block: int = 1024) -> np.ndarray:
    """C_S = (1/N) V^T S^T S V  [Summary 2.1 (values), 2.2A.1].

    ``q`` [N, G, d], ``k``/``v`` [N, d] of one calibration sequence.  For each
    query head h, O_h = S_h V; C_S = (1/(N G)) sum_h O_h^T O_h.  Rows of S are
    formed ``block`` at a time only to bound memory; each row is the plain
    causal softmax.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    n, g, d = q.shape
    acc = np.zeros((d, d))
    for h in range(g):
        for r0 in range(0, n, block):
            r1 = min(n, r0 + block)
            logits = q[r0:r1, h, :] @ k[:r1].T / np.sqrt(d)
            rows = np.arange(r0, r1)[:, None]
            cols = np.arange(r1)[None, :]
            logits = np.where(cols <= rows, logits, -np.inf)
            logits -= logits.max(axis=1, keepdims=True)
            p = np.exp(logits)
            p /= p.sum(axis=1, keepdims=True)
            o = p @ v[:r1]
            acc += o.T @ o
    return acc / (n * g)


def sorted_eigh(c: np.ndarray):
    """Eigen-decomposition of a symmetric C [Summary 2.2A.2].

    Columns of U sorted by descending eigenvalue.  Sign convention (the pages are
    silent): the entry of largest magnitude in each column is positive, ties to
    the lowest row index.  Returns (eigenvalues, U).
    """
    c = np.asarray(c, np.float64)
    w, u = np.linalg.eigh(0.5 * (c + c.T))
    order = np.argsort(-w, kind="stable")
    w, u = w[order], u[:, order].copy()
    for col in range(u.shape[1]):
        i = int(np.argmax(np.abs(u[:, col])))
        if u[i, col] < 0:
            u[:, col] = -u[:, col]
    return w, u


def hadamard(d: int) -> np.ndarray:
    """Normalised Sylvester Hadamard matrix, H_ij = (-1)^popcount(i & j) / sqrt(d)
    [Summary 2.2A.3, H_Had].  Natural (Sylvester) order is the reading taken."""
    if d <= 0 or d & (d - 1):
        raise ValueError("d must be a power of two")
    i = np.arange(d)
    parity = np.zeros((d, d), dtype=np.int64)
    x = i[:, None] & i[None, :]
    while np.any(x):
        parity ^= x & 1
        x = x >> 1
    return np.where(parity == 1, -1.0, 1.0) / np.sqrt(d)


def bit_reverse(d: int) -> np.ndarray:
    """br(i): i with its log2(d) bits reversed [Summary 2.2A.3, P_br]."""
    nb = d.bit_length() - 1
    if 1 << nb != d:
        raise ValueError("d must be a power of two")
    out = np.zeros(d, dtype=np.int64)
    for i in range(d):
        r = 0
        for b in range(nb):
            if i >> b & 1:
                r |= 1 << (nb - 1 - b)
        out[i] = r
    return out


def bit_reversal_matrix(d: int) -> np.ndarray:
    """P_br with P[i, br(i)] = 1, so (x P)_j = x_{br(j)}."""
    p = np.zeros((d, d))
    p[np.arange(d), bit_reverse(d)] = 1.0
    return p


def composite_rotation(c: np.ndarray | None, d: int, variant: int = OSCAR) -> np.ndarray:
    """R = U H_Had P_br  [Summary 2.2A.3 formula: R_K = U_Q H P_br, R_V = U_S H P_br].

    Variants used only for the fidelity comparison the pages describe
    ([Summary 1], [Summary 4]): Hadamard-only R = H, unrotated R = I.
    """
    if variant == IDENTITY:
        return np.eye(d)
    if variant == HADAMARD_ONLY:
        return hadamard(d)
    _, u = sorted_eigh(c)
    return u @ hadamard(d) @ bit_reversal_matrix(d)


def clip_threshold(x_calib: np.ndarray, r: np.ndarray, percentile: float = 99.9) -> float:
    """Clip c = percentile(|x_calib R|) over all N*d entries [Summary 2.2A.4].

    One threshold per (layer, KV head, K or V).  Percentile rule (pages silent):
    linear interpolation between order statistics (Hyndman-Fan type 7, numpy's
    default ``method='linear'``).
    """
    y = np.abs(np.asarray(x_calib, np.float64) @ np.asarray(r, np.float64))
    return float(np.percentile(y.ravel(), percentile, method="linear"))
