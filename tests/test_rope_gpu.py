"""GPU parity of the fused decode step with rotary position embedding
(oscar_decode_step_rope) against the oracle (oracle/rope.py).

The cache is prefilled with keys the oracle rotated at their positions and
rounded to bf16 (the activation precision); each step hands the kernel the raw
query and raw new key.  Checked per step:
- the output against the oracle's attention, over the stored pools, of the
  oracle-rotated bf16 query;
- the output against the plain fused step fed the oracle-rotated inputs;
- afterwards, the new keys' BF16 slots within one bf16 ulp of the oracle's
  rotated keys (the kernel rotates in fp32: cos/sin and products may round the
  other way at a bf16 boundary), every other pool byte as the oracle places it.
"""
import copy

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth
from oracle import rope

pytestmark = pytest.mark.gpu

BASE = 1.0e6     # the Qwen3 rotary base


def _bf16(x):
    """fp64 -> nearest bf16 (via the nearest fp32; ties to even)."""
    return synth.bf16_round(np.asarray(x, np.float32))


def _rotated_instance(inst):
    """The instance with every key rotated at its position, rounded to bf16."""
    r = copy.copy(inst)
    r.k = [[_bf16(rope.apply(kh, np.arange(len(kh)), BASE)) for kh in kb] for kb in inst.k]
    return r


@pytest.mark.parametrize("wl,lens0,steps,W", [
    (synth.TINY, [200, 140, 66], 4, 64),
    (synth.QWEN3_8B_32K, [2000, 1503, 133], 3, 128),
    (synth.TINY, [100000], 2, 64),                 # angles far beyond 2 pi
])
def test_rope_step_matches_oracle(wl, lens0, steps, W):
    t = H.torch()
    L = H.lib()
    lens0 = np.array(lens0)
    lens1 = lens0 + steps
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens1)
    rot = H.oracle_rotations(inst)
    rinst = _rotated_instance(inst)
    cache, pp = H.make_cache(rinst, rot, window=W, lens=lens0, growth=steps)
    plain, _ = H.make_cache(rinst, rot, window=W, lens=lens0, growth=steps)
    H.prefill(cache, rinst, lens=lens0)
    H.prefill(plain, rinst, lens=lens0)
    B, hkv, G = len(lens0), wl.num_kv_heads, wl.gqa
    q = H.bf16_tensor(inst.q)
    max_len = int(lens1.max())
    ws = t.zeros(L.oscar_decode_workspace_size(cache, B, max_len) // 4 + 64, dtype=t.float32,
                 device=H.DEV)
    for st in range(steps):
        cur = lens0 + st + 1
        pos = cur - 1
        kn = np.stack([[inst.k[b][h][pos[b]] for h in range(hkv)] for b in range(B)])
        vn = np.stack([[inst.v[b][h][pos[b]] for h in range(hkv)] for b in range(B)])
        lt = t.from_numpy(cur.astype(np.int32)).to(H.DEV)
        out = t.zeros(inst.q.shape, dtype=t.bfloat16, device=H.DEV)
        L.oscar_decode_step_rope(cache, q, H.bf16_tensor(kn), H.bf16_tensor(vn), lt, max_len, BASE,
                                 out, ws)
        q_r = _bf16(rope.apply(inst.q, pos[:, None], BASE))
        k_r = _bf16(rope.apply(kn, pos[:, None], BASE))
        out_p = t.zeros_like(out)
        L.oscar_decode_step(plain, H.bf16_tensor(q_r), H.bf16_tensor(k_r), H.bf16_tensor(vn), lt,
                            max_len, out_p, ws)
        t.cuda.synchronize()
        got = H.from_bf16(out)
        ref = H.attention_from_pools(cache, pp, q_r, cur, rot, sink=4, window=W, gqa=G)
        H.check_close(got, ref, f"rope step {st} vs oracle over stored pools")
        H.check_close(got, H.from_bf16(out_p), f"rope step {st} vs step on rotated inputs")
    assert H.status(cache) == 0 and H.status(plain) == 0
    # pools: everything but the new keys exactly as the oracle places the rotated tokens
    old = {b: [p_ for p_ in range(int(lens1[b])) if p_ < lens0[b]] for b in range(B)}
    exp = H.ocache.expected_pools(rinst.k, rinst.v, lens1, rot, sink=4, window=W, d=wl.head_dim,
                                  hkv=hkv, int2_table=pp.int2_table, bf16_table=pp.bf16_table,
                                  num_int2_pages=pp.num_int2_pages, num_bf16_pages=pp.num_bf16_pages,
                                  kappa=H.kappa(wl.head_dim), tokens=old)
    H.compare_pools(cache, exp)   # bytes outside flagged near-boundary entries are exact
    # the new keys: within one bf16 ulp of the oracle's rotated key
    new = {b: list(range(int(lens0[b]), int(lens1[b]))) for b in range(B)}
    expn = H.ocache.expected_pools(rinst.k, rinst.v, lens1, rot, sink=4, window=W, d=wl.head_dim,
                                   hkv=hkv, int2_table=pp.int2_table, bf16_table=pp.bf16_table,
                                   num_int2_pages=pp.num_int2_pages,
                                   num_bf16_pages=pp.num_bf16_pages, tokens=new)
    _, gotb = H.pools(cache)
    sel = expn.bf16_defined
    ulps = np.abs(gotb[sel].view(np.int16).astype(np.int32) - expn.bf16[sel].view(np.int16).astype(np.int32))
    assert ulps.max() <= 1 and (ulps > 0).mean() < 0.02, (int(ulps.max()), float((ulps > 0).mean()))


def test_rope_argument_checks():
    L = H.lib()
    wl = synth.TINY
    inst = synth.draw_instance(wl, n_calib=32, seq_lens=[100])
    rot = H.oracle_rotations(inst)
    cache, _ = H.make_cache(inst, rot, window=64)
    t = H.torch()
    z = t.zeros((1, 4, 64), dtype=t.bfloat16, device=H.DEV)
    kv = t.zeros((1, 1, 64), dtype=t.bfloat16, device=H.DEV)
    lt = t.tensor([100], dtype=t.int32, device=H.DEV)
    ws = t.empty(1 << 20, dtype=t.float32, device=H.DEV)
    for bad in (1.0, 0.5, float("inf"), float("nan")):
        with pytest.raises(L.OscarError):
            L.oscar_decode_step_rope(cache, z, kv, kv, lt, 100, bad, z, ws)
