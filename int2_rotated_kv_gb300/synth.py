"""Seeded synthetic workloads for the mixed-precision INT2 KV-cache path.

This module only draws random inputs and describes workload shapes.  It holds
none of the method's arithmetic: no covariance, eigenbasis, Hadamard, bit
reversal, clipping, quantisation, packing or attention.  Both the fp64 oracle's
tests and the GPU path's tests and benchmark take their inputs from here, so
the two sides always see the same bf16 values.

Distribution (per KV head; the OSCAR pages evaluate Qwen3 models whose keys
carry strong channel-wise outliers -- Technical Summary section 1 -- and the
workloads below copy those shapes with synthetic numbers):

* per-channel std  sigma_c = exp(0.5 * N(0,1))  (lognormal(0, 0.5));
* keys   K = N(0,1) * sigma_c; on ``k_outliers`` channels chosen without
  replacement the value is multiplied by ``k_outlier_mult`` and then
  ``k_offset`` (+3) is added (the "+3 mean offset" is read as belonging to the
  outlier channels);
* values V = N(0,1) * sigma'_c (fresh sigma); ``v_outliers`` channels x6;
* queries q = z diag(sqrt(lambda)) W^T with lambda_i = 0.9**i and W a Haar
  orthogonal matrix (QR of a Gaussian, column signs fixed so diag(R) > 0); the
  G query heads of a KV head share this covariance;
* every value is rounded once to bf16 (round to nearest even).

Streams: ``numpy.random.default_rng(seed).spawn(4)`` gives, in order, the
per-head parameter stream, the calibration stream, the context stream and the
query stream.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PAGE = 16          # tokens per KV page
GROUP = 32         # channels per quantisation group


# ----------------------------------------------------------------------------
# bf16 helpers (storage format only)
# ----------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.astype(np.uint32).view(np.float32).reshape(np.shape(x))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of bf16-representable float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def bf16_from_bits(u: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# Workload descriptions
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context: int | tuple[int, int]      # fixed length or inclusive uniform range
    sink: int = 4
    window: int = 128
    n_calib: int = 8192
    k_outliers: int = 4
    k_outlier_mult: float = 15.0
    k_offset: float = 3.0
    v_outliers: int = 2
    v_outlier_mult: float = 6.0
    shared_prefix: int = 0
    layers: int = 1
    seed: int = 0

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def seq_lens(self) -> np.ndarray:
        """Per-sequence context lengths (the current decode token included)."""
        if isinstance(self.context, tuple):
            lo, hi = self.context
            rng = np.random.default_rng([self.seed, 7])
            return rng.integers(lo, hi + 1, size=self.batch).astype(np.int64)
        return np.full(self.batch, int(self.context), dtype=np.int64)


TINY = Workload("tiny_d64_g4_L512", batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64,
                context=512, window=64, n_calib=2048)
QWEN3_8B_32K = Workload("qwen3_8b_32k_b1", batch=1, num_q_heads=32, num_kv_heads=8,
                        head_dim=128, context=32768, layers=36)
QWEN3_4B_PREFIX = Workload("qwen3_4b_b64_prefix2048", batch=64, num_q_heads=32, num_kv_heads=8,
                           head_dim=128, context=(4096, 8192), shared_prefix=2048)
QWEN3_32B_128K = Workload("qwen3_32b_128k_b1", batch=1, num_q_heads=64, num_kv_heads=8,
                          head_dim=128, context=131072, k_outliers=8, k_outlier_mult=25.0)
QWEN3_8B_BUDGET = Workload("qwen3_8b_4k_budget40GB", batch=1, num_q_heads=32, num_kv_heads=8,
                           head_dim=128, context=4096, layers=36)

WORKLOADS = {w.name: w for w in (TINY, QWEN3_8B_32K, QWEN3_4B_PREFIX, QWEN3_32B_128K,
                                 QWEN3_8B_BUDGET)}


# ----------------------------------------------------------------------------
# Per-head distribution parameters
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class HeadParams:
    sigma_k: np.ndarray
    sigma_v: np.ndarray
    k_out: np.ndarray
    v_out: np.ndarray
    q_basis: np.ndarray        # Haar orthogonal W (d x d)
    q_std: np.ndarray          # sqrt(lambda_i), lambda_i = 0.9**i


def haar_orthogonal(rng: np.random.Generator, d: int) -> np.ndarray:
    a = rng.standard_normal((d, d))
    q, r = np.linalg.qr(a)
    return q * np.sign(np.diag(r))[None, :]


def head_params(rng: np.random.Generator, w: Workload) -> HeadParams:
    d = w.head_dim
    sigma_k = np.exp(0.5 * rng.standard_normal(d))
    sigma_v = np.exp(0.5 * rng.standard_normal(d))
    k_out = rng.choice(d, w.k_outliers, replace=False)
    v_out = rng.choice(d, w.v_outliers, replace=False)
    basis = haar_orthogonal(rng, d)
    q_std = np.sqrt(0.9 ** np.arange(d))
    return HeadParams(sigma_k, sigma_v, np.sort(k_out), np.sort(v_out), basis, q_std)


def draw_kv(rng: np.random.Generator, p: HeadParams, w: Workload, n: int):
    """n tokens of one KV head: (K, V) float32 [n, d] holding bf16 values."""
    d = w.head_dim
    k = rng.standard_normal((n, d)) * p.sigma_k[None, :]
    k[:, p.k_out] = k[:, p.k_out] * w.k_outlier_mult + w.k_offset
    v = rng.standard_normal((n, d)) * p.sigma_v[None, :]
    v[:, p.v_out] = v[:, p.v_out] * w.v_outlier_mult
    return bf16_round(k.astype(np.float32)), bf16_round(v.astype(np.float32))


def draw_q(rng: np.random.Generator, p: HeadParams, w: Workload, n: int):
    """n query positions x G heads of one KV group: float32 [n, G, d] bf16 values."""
    z = rng.standard_normal((n, w.gqa, w.head_dim))
    q = (z * p.q_std[None, None, :]) @ p.q_basis.T
    return bf16_round(q.astype(np.float32))


@dataclasses.dataclass
class Instance:
    """One drawn workload: calibration sets, per-sequence context and queries."""
    workload: Workload
    params: list            # HeadParams per KV head
    calib_q: list           # per KV head [N, G, d]
    calib_k: list           # per KV head [N, d]
    calib_v: list
    seq_lens: np.ndarray    # [B]
    k: list                 # k[b][h] -> [L_b, d] float32 (bf16 values)
    v: list
    q: np.ndarray           # [B, Hq, d] decode queries (query head = h*G + g)
    new_k: np.ndarray | None = None   # optional next-token K/V for append tests [B, Hkv, d]
    new_v: np.ndarray | None = None


def draw_instance(w: Workload, *, n_calib: int | None = None, seq_lens=None,
                  with_next_token: bool = False) -> Instance:
    """Draw a full instance of ``w`` on the host (numpy).

    ``n_calib`` / ``seq_lens`` override the workload's sizes (small tests).
    Tokens of the shared prefix are drawn once per KV head and reused by every
    sequence, as a prefix cache hit would make them.
    """
    root = np.random.default_rng(w.seed)
    s_params, s_calib, s_ctx, s_query = root.spawn(4)
    H, G, d = w.num_kv_heads, w.gqa, w.head_dim
    params = [head_params(r, w) for r in s_params.spawn(H)]
    n_cal = w.n_calib if n_calib is None else n_calib
    cq, ck, cv = [], [], []
    for h, r in enumerate(s_calib.spawn(H)):
        kk, vv = draw_kv(r, params[h], w, n_cal)
        cq.append(draw_q(r, params[h], w, n_cal))
        ck.append(kk)
        cv.append(vv)
    lens = w.seq_lens() if seq_lens is None else np.asarray(seq_lens, dtype=np.int64)
    B = len(lens)
    prefix_rng, *seq_rngs = s_ctx.spawn(B + 1)
    prefix = []
    if w.shared_prefix:
        for h, r in enumerate(prefix_rng.spawn(H)):
            prefix.append(draw_kv(r, params[h], w, w.shared_prefix))
    ks, vs = [], []
    for b in range(B):
        kb, vb = [], []
        for h, r in enumerate(seq_rngs[b].spawn(H)):
            n_own = int(lens[b]) - (w.shared_prefix if w.shared_prefix else 0)
            kk, vv = draw_kv(r, params[h], w, max(n_own, 0))
            if w.shared_prefix:
                kk = np.concatenate([prefix[h][0], kk])[: lens[b]]
                vv = np.concatenate([prefix[h][1], vv])[: lens[b]]
            kb.append(kk)
            vb.append(vv)
        ks.append(kb)
        vs.append(vb)
    q = np.zeros((B, H * G, d), dtype=np.float32)
    qr = s_query.spawn(B * H + 1)
    for b in range(B):
        for h in range(H):
            q[b, h * G:(h + 1) * G] = draw_q(qr[b * H + h], params[h], w, 1)[0]
    inst = Instance(w, params, cq, ck, cv, lens, ks, vs, q)
    if with_next_token:
        r = qr[-1]
        nk = np.zeros((B, H, d), np.float32)
        nv = np.zeros((B, H, d), np.float32)
        for b in range(B):
            for h in range(H):
                a, c = draw_kv(r, params[h], w, 1)
                nk[b, h], nv[b, h] = a[0], c[0]
        inst.new_k, inst.new_v = nk, nv
    return inst


def dense_tokens(inst: Instance):
    """Flatten an instance's context into the token-major arrays the prefill
    call takes: k/v [T, Hkv, d], seq_ids [T], positions [T]."""
    B = len(inst.seq_lens)
    H, d = inst.workload.num_kv_heads, inst.workload.head_dim
    T = int(inst.seq_lens.sum())
    k = np.empty((T, H, d), np.float32)
    v = np.empty((T, H, d), np.float32)
    sid = np.empty(T, np.int32)
    pos = np.empty(T, np.int32)
    o = 0
    for b in range(B):
        L = int(inst.seq_lens[b])
        for h in range(H):
            k[o:o + L, h] = inst.k[b][h]
            v[o:o + L, h] = inst.v[b][h]
        sid[o:o + L] = b
        pos[o:o + L] = np.arange(L)
        o += L
    return k, v, sid, pos


def pages_needed(L: int) -> int:
    return (int(L) + PAGE - 1) // PAGE


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def budget_batch(bytes_per_seq: int, budget: float) -> int:
    return int(math.floor(budget / bytes_per_seq))


# ----------------------------------------------------------------------------
# Large workloads, drawn on the GPU
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class DeviceInstance:
    """A workload whose context is drawn on the GPU (torch), for sizes the host
    generator would take minutes on.  Per-head parameters and calibration sets
    come from the same seeded host streams as ``draw_instance``; context and
    queries follow the same per-channel recipe from a seeded torch stream, so
    values differ from ``draw_instance`` but the distribution does not.

    Prefill lists hold tokens [0, L_b - 1) of every sequence (token-major
    k/v [T, Hkv, d] bf16, seq_ids, positions); tokens of a shared prefix are
    listed once, under sequence 0.  k_new/v_new are token L_b - 1 and q the
    decode query at that position."""
    workload: Workload
    params: list
    calib_q: list
    calib_k: list
    calib_v: list
    seq_lens: np.ndarray
    k_tok: object
    v_tok: object
    seq_ids: object
    positions: object
    k_new: object
    v_new: object
    q: object


def _device_kv(gen, p: HeadParams, w: Workload, n: int, device):
    import torch
    d = w.head_dim
    sk = torch.as_tensor(p.sigma_k, dtype=torch.float32, device=device)
    sv = torch.as_tensor(p.sigma_v, dtype=torch.float32, device=device)
    k = torch.randn((n, d), generator=gen, device=device) * sk
    ko = torch.as_tensor(p.k_out, device=device)
    k[:, ko] = k[:, ko] * w.k_outlier_mult + w.k_offset
    v = torch.randn((n, d), generator=gen, device=device) * sv
    vo = torch.as_tensor(p.v_out, device=device)
    v[:, vo] = v[:, vo] * w.v_outlier_mult
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def draw_device(w: Workload, seq_lens, device, *, n_calib: int | None = None,
                seed: int = 0) -> DeviceInstance:
    import torch
    root = np.random.default_rng(w.seed)
    s_params, s_calib, _, _ = root.spawn(4)
    H, G, d = w.num_kv_heads, w.gqa, w.head_dim
    params = [head_params(r, w) for r in s_params.spawn(H)]
    n_cal = w.n_calib if n_calib is None else n_calib
    cq, ck, cv = [], [], []
    for h, r in enumerate(s_calib.spawn(H)):
        kk, vv = draw_kv(r, params[h], w, n_cal)
        cq.append(draw_q(r, params[h], w, n_cal))
        ck.append(kk)
        cv.append(vv)
    lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(lens)
    gen = torch.Generator(device=device)
    gen.manual_seed(1_000_003 * (w.seed + 1) + seed)
    P = w.shared_prefix
    prefix = [_device_kv(gen, params[h], w, P, device) for h in range(H)] if P else None
    ks, vs, sids, poss = [], [], [], []
    for b in range(B):
        n = int(lens[b]) - 1                      # tokens already in the cache
        first = P if (P and b > 0) else 0         # shared prefix listed under sequence 0 only
        own = max(n - P, 0) if P else n
        kb = torch.empty((n - first, H, d), dtype=torch.bfloat16, device=device)
        vb = torch.empty_like(kb)
        for h in range(H):
            k_own, v_own = _device_kv(gen, params[h], w, own, device)
            if P and b == 0:
                kb[:, h] = torch.cat([prefix[h][0], k_own])[:n]
                vb[:, h] = torch.cat([prefix[h][1], v_own])[:n]
            else:
                kb[:, h] = k_own[: n - first]
                vb[:, h] = v_own[: n - first]
        ks.append(kb)
        vs.append(vb)
        sids.append(torch.full((n - first,), b, dtype=torch.int32, device=device))
        poss.append(torch.arange(first, n, dtype=torch.int32, device=device))
    k_new = torch.empty((B, H, d), dtype=torch.bfloat16, device=device)
    v_new = torch.empty_like(k_new)
    q = torch.empty((B, H * G, d), dtype=torch.bfloat16, device=device)
    for h in range(H):
        a, c = _device_kv(gen, params[h], w, B, device)
        k_new[:, h], v_new[:, h] = a, c
        z = torch.randn((B, G, d), generator=gen, device=device)
        std = torch.as_tensor(params[h].q_std, dtype=torch.float32, device=device)
        basis = torch.as_tensor(params[h].q_basis, dtype=torch.float32, device=device)
        q[:, h * G:(h + 1) * G] = ((z * std) @ basis.T).to(torch.bfloat16)
    return DeviceInstance(w, params, cq, ck, cv, lens, torch.cat(ks), torch.cat(vs),
                          torch.cat(sids), torch.cat(poss), k_new, v_new, q)
