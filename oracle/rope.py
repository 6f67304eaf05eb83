"""Rotary position embedding, as the decode step applies it to a new token's
query and key before they meet the cache (the fused step of a serving
pipeline).  The pages name fused kernel pipelines ([Abstract]) and the models
they serve (Qwen3, [Summary 4]); the embedding itself is that family's:
rotary over the whole head dimension d, channel i paired with i + d/2 (the
"rotate half" arrangement), angle m * theta_i at position m with
theta_i = base^(-2i/d), i in [0, d/2).

For each pair (a, b) = (x_i, x_{i+d/2}):
    a' = a cos(m theta_i) - b sin(m theta_i)
    b' = b cos(m theta_i) + a sin(m theta_i)
computed here in fp64.
"""
from __future__ import annotations

import numpy as np


def inv_freq(d: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d), i = 0 .. d/2 - 1 (fp64)."""
    return float(base) ** (-2.0 * np.arange(d // 2, dtype=np.float64) / d)


def apply(x: np.ndarray, positions, base: float) -> np.ndarray:
    """Rotate x [..., d] at positions [...] (broadcast over the leading axes)."""
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(positions, np.float64)[..., None] * inv_freq(d, base)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)
