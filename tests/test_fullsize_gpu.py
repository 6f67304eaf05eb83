"""Parity at the benchmark's full sizes, in the launch configuration it times:
the cache holds L - 1 tokens (bulk prefill), then one fused decode step
(oscar_decode_step: append of token L - 1 and attention at length L).

Qwen3-8B shape at L = 32768 is compared in full against the oracle's
attention over the stored pools; Qwen3-32B shape at L = 131072 on two sampled
KV heads (16 of its 64 query heads).  Every INT2 group of the context is
checked through the traced prefill (rotation within its bound, decisions equal
to the oracle's quantiser of the kernel's values), the leaving token through a
traced append on a copy of the pre-step pools, and stored pools are compared
with the oracle's placement on sampled pages, including the page that received
the token leaving the window.  Rotations come from the oracle's calibration on
1024 tokens (the parity does not depend on their quality)."""
import dataclasses

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth

pytestmark = pytest.mark.gpu


def _full_step(wl, heads):
    t = H.torch()
    L = H.lib()
    Lc = int(wl.context)
    inst = synth.draw_instance(wl, n_calib=1024, seq_lens=[Lc])
    rot = H.oracle_rotations(inst)
    W = wl.window
    d, hkv = wl.head_dim, wl.num_kv_heads
    lens0 = np.array([Lc - 1])
    cache, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=1)
    # the bulk prefill, traced: every INT2 group of the context is checked
    y, where = H.prefill_trace(cache, inst, lens=lens0)
    st = H.check_traced(cache, pp, inst, rot, {0: (np.arange(Lc - 1), y)}, H.kappa_tc(d),
                        lens=lens0, sink=4, window=W)
    del y
    # the step's append, traced on a copy of the pools: the token leaving the window
    kn = H.bf16_tensor(np.stack([[inst.k[0][h][Lc - 1] for h in range(hkv)]]))
    vn = H.bf16_tensor(np.stack([[inst.v[0][h][Lc - 1] for h in range(hkv)]]))
    lt = t.tensor([Lc], dtype=t.int32, device=H.DEV)
    twin = dataclasses.replace(cache, int2_pool=cache.int2_pool.clone(),
                               bf16_pool=cache.bf16_pool.clone())
    ya = t.full((1, hkv, 2, d), float("nan"), dtype=t.float32, device=H.DEV)
    L.oscar_quantize_append_trace(twin, kn, vn, lt, ya)
    q = H.bf16_tensor(inst.q)
    out = t.zeros(inst.q.shape, dtype=t.bfloat16, device=H.DEV)
    ws = t.zeros(L.oscar_decode_workspace_size(cache, 1, Lc) // 4 + 64, dtype=t.float32, device=H.DEV)
    L.oscar_decode_step(cache, q, kn, vn, lt, Lc, out, ws)
    t.cuda.synchronize()
    assert H.status(cache) == 0 and H.status(twin) == 0
    got2, gotb = H.pools(cache)
    twin2, twinb = H.pools(twin)
    # the fused step's append writes what the plain append writes
    np.testing.assert_array_equal(got2, twin2)
    np.testing.assert_array_equal(gotb, twinb)
    left = Lc - 1 - W
    sa = H.check_traced(cache, pp, inst, rot, {0: (np.array([left]), ya.cpu().numpy())}, H.kappa(d),
                        lens=[Lc], sink=4, window=W, pools_=got2)
    H.report(f"fullsize[{wl.name}]", prefill=st, append=sa)
    assert st["straddling_groups"] <= max(2, 0.005 * st["groups"])
    got = H.from_bf16(out)
    ref = H.attention_from_pools(cache, pp, inst.q, [Lc], rot, sink=4, window=W, gqa=wl.gqa,
                                 heads=heads)
    cols = np.concatenate([np.arange(h * wl.gqa, (h + 1) * wl.gqa)
                           for h in (range(hkv) if heads is None else heads)])
    H.check_close(got[:, cols], ref[:, cols], f"{wl.name} full-size step")
    # pools on sampled pages against the oracle's placement from the exact x R:
    # the first INT2 page, the page of the token that just left the window, the
    # last page, and a seeded sample in between
    rng = np.random.default_rng(7)
    n_pages = (Lc + 15) // 16
    sample = {0, 1, left // 16, (Lc - 1) // 16, *rng.choice(n_pages, 24, replace=False).tolist()}
    toks = sorted(t_ for pg in sample for t_ in range(16 * pg, min(16 * pg + 16, Lc)))
    exp = H.ocache.expected_pools(inst.k, inst.v, [Lc], rot, sink=4, window=W, d=d,
                                  hkv=hkv, int2_table=pp.int2_table, bf16_table=pp.bf16_table,
                                  num_int2_pages=pp.num_int2_pages, num_bf16_pages=pp.num_bf16_pages,
                                  kappa=H.kappa_tc(d), tokens={0: toks})
    H.compare_pools(cache, exp)


def test_qwen3_8b_32k_full_step():
    _full_step(synth.QWEN3_8B_32K, heads=None)


def test_qwen3_32b_128k_full_step_sampled_heads():
    _full_step(synth.QWEN3_32B_128K, heads=[0, 5])
