"""Pins for test infrastructure that turns stored pools back into attention."""
import types

import numpy as np

import gpu_harness as H
from int2_rotated_kv_gb300 import pages, synth
from oracle import attention, cache as ocache


def test_attention_from_pools_reproduces_the_oracle():
    """Pools packed by the oracle, read back and attended, give exactly the
    oracle's mixed-cache attention (both are fp64 over the same stored values)."""
    import torch
    wl = synth.TINY
    lens = np.array([300, 77, 66])
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    pp = pages.plan(lens, 4, 64, permute_seed=5)
    exp = ocache.expected_pools(inst.k, inst.v, lens, rot, sink=4, window=64, d=wl.head_dim,
                                hkv=wl.num_kv_heads, int2_table=pp.int2_table,
                                bf16_table=pp.bf16_table, num_int2_pages=pp.num_int2_pages,
                                num_bf16_pages=pp.num_bf16_pages)
    cache = types.SimpleNamespace(int2_pool=torch.from_numpy(exp.int2.copy()),
                                  bf16_pool=torch.from_numpy(exp.bf16.view(np.int16).copy()).view(torch.bfloat16))
    got = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=64, gqa=wl.gqa)
    ref = attention.mixed_decode(inst.q, inst.k, inst.v, lens, rot, sink=4, window=64, gqa=wl.gqa)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_attention_from_pools_drops_whole_pages():
    """Leaving out a logical page removes exactly its 16 tokens from the softmax."""
    import torch
    wl = synth.TINY
    lens = np.array([300])
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    pp = pages.plan(lens, 4, 64)
    exp = ocache.expected_pools(inst.k, inst.v, lens, rot, sink=4, window=64, d=wl.head_dim,
                                hkv=1, int2_table=pp.int2_table, bf16_table=pp.bf16_table,
                                num_int2_pages=pp.num_int2_pages, num_bf16_pages=pp.num_bf16_pages)
    cache = types.SimpleNamespace(int2_pool=torch.from_numpy(exp.int2.copy()),
                                  bf16_pool=torch.from_numpy(exp.bf16.view(np.int16).copy()).view(torch.bfloat16))
    got = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=64, gqa=4, drop={0: [5]})
    ke, ve = attention.effective_kv(inst.k[0][0], inst.v[0][0], 300, 4, 64, rot.rk[0], rot.rv[0],
                                    rot.ck[0], rot.cv[0])
    keep = np.ones(300, bool)
    keep[80:96] = False
    ref = attention.softmax_attention(inst.q[0, 0:4], ke[keep], ve[keep])
    np.testing.assert_allclose(got[0, 0:4], ref, rtol=1e-12, atol=1e-12)


def test_attention_from_pools_upto_matches_multiquery_oracle():
    """A visibility limit per sequence reproduces the oracle's multi-row attention."""
    import torch
    wl = synth.TINY
    lens = np.array([300, 250])
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    pp = pages.plan(lens, 4, 64)
    exp = ocache.expected_pools(inst.k, inst.v, lens, rot, sink=4, window=64, d=wl.head_dim,
                                hkv=1, int2_table=pp.int2_table, bf16_table=pp.bf16_table,
                                num_int2_pages=pp.num_int2_pages, num_bf16_pages=pp.num_bf16_pages)
    cache = types.SimpleNamespace(int2_pool=torch.from_numpy(exp.int2.copy()),
                                  bf16_pool=torch.from_numpy(exp.bf16.view(np.int16).copy()).view(torch.bfloat16))
    pos = np.array([[120, 299], [7, 249]])
    q = np.stack([inst.q, inst.q], axis=1)                    # [B, M, Hq, d]
    ref = attention.mixed_multiquery(q, inst.k, inst.v, lens, pos, rot, sink=4, window=64, gqa=4)
    for m in range(2):
        got = H.attention_from_pools(cache, pp, q[:, m], lens, rot, sink=4, window=64, gqa=4,
                                     upto=pos[:, m])
        np.testing.assert_allclose(got, ref[:, m], rtol=1e-12, atol=1e-12)


def test_attention_from_pools_reads_int4_pools():
    """The INT4 variant: oracle-packed two-plane pools read back and attended
    give exactly the oracle's attention with sixteen-level codes."""
    import torch
    wl = synth.TINY
    lens = np.array([300, 90])
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    pp = pages.plan(lens, 4, 64, permute_seed=2)
    exp = ocache.expected_pools(inst.k, inst.v, lens, rot, sink=4, window=64, d=wl.head_dim,
                                hkv=1, int2_table=pp.int2_table, bf16_table=pp.bf16_table,
                                num_int2_pages=pp.num_int2_pages, num_bf16_pages=pp.num_bf16_pages,
                                bits=4)
    cache = types.SimpleNamespace(int2_pool=torch.from_numpy(exp.int2.copy()), code_bits=4,
                                  bf16_pool=torch.from_numpy(exp.bf16.view(np.int16).copy()).view(torch.bfloat16))
    got = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=64, gqa=4)
    ref = attention.mixed_decode(inst.q, inst.k, inst.v, lens, rot, sink=4, window=64, gqa=4,
                                 levels=15)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # and sixteen levels sit closer to all-BF16 attention than four do
    bf = attention.bf16_decode(inst.q, inst.k, inst.v, lens, gqa=4)
    int2 = attention.mixed_decode(inst.q, inst.k, inst.v, lens, rot, sink=4, window=64, gqa=4)
    assert attention.rel_l2(ref, bf) < attention.rel_l2(int2, bf)
