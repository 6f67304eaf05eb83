"""GPU parity of split-K decode attention over the mixed cache (and of the
same-design BF16 baseline) against the oracle's plain-definition attention,
computed from the codes the cache actually stores: the parity rule for the
attention output.  The stored codes themselves are checked against the
oracle's quantiser in test_quantize_gpu.py (bit-exact except flagged
near-boundary entries, where one step either way is allowed)."""
import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth
from oracle import attention, cache as ocache

pytestmark = pytest.mark.gpu


def _run(wl, lens, W, *, n_calib=512, shared=0, permute=None, max_len=None, variant=0):
    inst = synth.draw_instance(wl, n_calib=n_calib, seq_lens=lens)
    rot = H.oracle_rotations(inst, variant=variant)
    cache, pp = H.make_cache(inst, rot, window=W, shared=shared, permute=permute, max_len=max_len)
    H.prefill(cache, inst)
    out = H.decode(cache, inst.q, inst.seq_lens, max_len=max_len)
    return inst, rot, cache, pp, out


@pytest.mark.parametrize("wl,lens,W", [
    (synth.TINY, [512], 64),                                   # the tiny workload itself
    (synth.TINY, [37, 69, 70, 83, 1500], 64),                  # all-BF16, boundary, ragged
    (synth.QWEN3_8B_32K, [4133, 129, 133, 2048 + 132], 128),   # G=4, d=128, several splits
    (synth.QWEN3_32B_128K, [5000, 1], 128),                    # G=8, L=1 edge
])
def test_decode_matches_oracle(wl, lens, W):
    inst, rot, cache, pp, out = _run(wl, lens, W)
    ref = H.attention_from_pools(cache, pp, inst.q, inst.seq_lens, rot, sink=4, window=W,
                                 gqa=wl.gqa)
    H.check_close(out, ref, f"{wl.name} {lens}")
    assert H.status(cache) == 0


def _ragged(n, lo, hi, seed):
    return [int(x) for x in np.random.default_rng(seed).integers(lo, hi, size=n)]


@pytest.mark.parametrize("wl,lens,W", [
    # more (row, query head) pairs per KV head than a wave of combine CTAs, two
    # or three splits each: the row-parallel merge (d = 128, and d = 64 with one
    # KV head)
    (synth.QWEN3_8B_32K, _ragged(44, 150, 1300, 1), 128),
    (synth.TINY, _ragged(80, 70, 700, 2), 64),
    # many pairs with more splits each (G = 8, six sequences): the merge that
    # runs the pairs of a CTA one after another
    (synth.QWEN3_32B_128K, _ragged(6, 2500, 3500, 3), 128),
])
def test_many_pairs_per_kv_head(wl, lens, W):
    inst, rot, cache, pp, out = _run(wl, lens, W, n_calib=256)
    ref = H.attention_from_pools(cache, pp, inst.q, inst.seq_lens, rot, sink=4, window=W,
                                 gqa=wl.gqa)
    H.check_close(out, ref, f"{wl.name} {len(lens)} sequences")
    assert H.status(cache) == 0


@pytest.mark.parametrize("g", [1, 2, 16])
def test_small_gqa_groups(g):
    wl = synth.Workload("g%d" % g, batch=2, num_q_heads=2 * g, num_kv_heads=2, head_dim=128,
                        context=3000, n_calib=256)
    inst, rot, cache, pp, out = _run(wl, [3000, 1777], 128)
    ref = H.attention_from_pools(cache, pp, inst.q, inst.seq_lens, rot, sink=4, window=128, gqa=g)
    H.check_close(out, ref)


def test_decode_from_oracle_packed_pools():
    """Pools written by the oracle (no GPU quantiser involved) decode to the
    oracle's attention: isolates the attention kernels."""
    t = H.torch()
    wl = synth.QWEN3_8B_32K
    lens = [1800, 950]
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=128, permute=3)
    exp = H.expected(inst, rot, pp, window=128)
    cache.int2_pool.copy_(t.from_numpy(exp.int2).to(H.DEV))
    cache.bf16_pool.copy_(t.from_numpy(exp.bf16.view(np.int16)).view(t.bfloat16).to(H.DEV))
    out = H.decode(cache, inst.q, inst.seq_lens)
    ref = attention.mixed_decode(inst.q, inst.k, inst.v, inst.seq_lens, rot, sink=4, window=128,
                                 gqa=wl.gqa)
    H.check_close(out, ref)


def test_split_count_and_placement_invariance():
    wl = synth.QWEN3_8B_32K
    lens = [3000, 2100]
    inst, rot, cache, pp, out = _run(wl, lens, 128)
    # a larger max_seq_len changes the split plan (pages per split)
    out2 = H.decode(cache, inst.q, inst.seq_lens, max_len=16 * pp.max_pages)
    assert np.abs(out2 - out).max() <= 2 * 2.0 ** -8 * max(1.0, np.abs(out).max())
    # the same data at permuted physical pages gives identical bits
    _, _, _, _, out3 = _run(wl, lens, 128, permute=11)
    np.testing.assert_array_equal(out3, out)


def test_prefix_sharing_equals_private_copies():
    wl = synth.QWEN3_4B_PREFIX
    lens = [2200, 2600, 2400]
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    c1, pp1 = H.make_cache(inst, rot, window=128, shared=wl.shared_prefix)
    assert pp1.int2_table[0, 5] == pp1.int2_table[2, 5]          # shared page ids
    H.prefill(c1, inst)
    o1 = H.decode(c1, inst.q, inst.seq_lens)
    c2, pp2 = H.make_cache(inst, rot, window=128, shared=0)
    H.prefill(c2, inst)
    o2 = H.decode(c2, inst.q, inst.seq_lens)
    np.testing.assert_array_equal(o1, o2)
    ref = H.attention_from_pools(c1, pp1, inst.q, inst.seq_lens, rot, sink=4, window=128,
                                 gqa=wl.gqa)
    H.check_close(o1, ref)


@pytest.mark.parametrize("wl,lens", [(synth.TINY, [512, 17]),
                                     (synth.QWEN3_8B_32K, [3071, 1])])
def test_bf16_baseline_matches_oracle(wl, lens):
    inst = synth.draw_instance(wl, n_calib=32, seq_lens=lens)
    rot = ocache.Rotations([np.eye(wl.head_dim, dtype=np.float32)] * wl.num_kv_heads,
                           [np.eye(wl.head_dim, dtype=np.float32)] * wl.num_kv_heads,
                           [np.float32(1)] * wl.num_kv_heads, [np.float32(1)] * wl.num_kv_heads)
    # every token BF16: window covers the whole context
    big = int(max(lens))
    cache, _ = H.make_cache(inst, rot, window=big, sink=0)
    H.prefill(cache, inst)
    out = H.decode(cache, inst.q, inst.seq_lens, bf16_only=True)
    ref = attention.bf16_decode(inst.q, inst.k, inst.v, inst.seq_lens, gqa=wl.gqa)
    H.check_close(out, ref)


def test_bad_lengths_are_reported_not_faulted():
    wl = synth.TINY
    inst, rot, cache, pp, _ = _run(wl, [300, 200], 64)
    t = H.torch()
    L = H.lib()
    lens = t.tensor([300, 10_000], dtype=t.int32, device=H.DEV)    # beyond max_seq_len
    q = H.bf16_tensor(inst.q)
    o = t.zeros((2, 4, 64), dtype=t.bfloat16, device=H.DEV)
    ws = t.zeros(L.oscar_decode_workspace_size(cache, 2, 300) // 4 + 64, dtype=t.float32,
                 device=H.DEV)
    L.oscar_decode_attention(cache, q, lens, 300, o, ws)
    t.cuda.synchronize()
    assert H.status(cache) & L.DEVERR_SEQ_LEN
    assert float(o[1].float().abs().max()) == 0.0
    ref = H.attention_from_pools(cache, pp, inst.q[:1], [300], rot, sink=4, window=64, gqa=4)
    H.check_close(H.from_bf16(o)[:1], ref)


def test_bad_page_id_is_masked_and_reported():
    """An INT2 page id beyond the pool is skipped (its tokens drop out of the
    softmax) and reported; the other tokens are attended as usual."""
    t = H.torch()
    wl = synth.QWEN3_8B_32K
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=[2500])
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=128)
    H.prefill(cache, inst)
    bad_page = 37
    tbl = pp.int2_table.copy()
    tbl[0, bad_page] = pp.num_int2_pages + 3
    cache.int2_page_table = t.from_numpy(tbl).to(H.DEV)
    out = H.decode(cache, inst.q, inst.seq_lens)
    assert H.status(cache) & H.lib().DEVERR_PAGE_ID
    ref = H.attention_from_pools(cache, pp, inst.q, [2500], rot, sink=4, window=128, gqa=wl.gqa,
                                 drop={0: [bad_page]})
    H.check_close(out, ref)
