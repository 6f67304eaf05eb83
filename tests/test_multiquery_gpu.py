"""GPU parity of several query rows per sequence over the mixed cache (chunked
prefill / verification): against the single-row decode and against the oracle's
attention over the stored codes with each row's causal limit.  Rows of one
sequence share a CTA (8 / G of them), so G = 1, 2 and 4 are covered, with row
counts that leave a partial last group."""
import dataclasses

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth

pytestmark = pytest.mark.gpu


def _setup(wl, lens, W):
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=W)
    H.prefill(cache, inst)
    return inst, rot, cache, pp


def _run(cache, q_rows, lens, pos, max_len):
    t = H.torch()
    L = H.lib()
    B, M = pos.shape
    q = H.bf16_tensor(q_rows)
    lt = t.from_numpy(np.asarray(lens, np.int32)).to(H.DEV)
    pt = t.from_numpy(pos.astype(np.int32)).to(H.DEV)
    out = t.zeros(q_rows.shape, dtype=t.bfloat16, device=H.DEV)
    ws = t.zeros(L.oscar_multiquery_workspace_size(cache, B, M, max_len) // 4 + 64,
                 dtype=t.float32, device=H.DEV)
    L.oscar_multiquery_attention(cache, q, lt, pt, max_len, out, ws)
    t.cuda.synchronize()
    return H.from_bf16(out)


def test_single_row_at_the_end_equals_decode():
    wl = synth.QWEN3_8B_32K
    lens = [2600, 900]
    inst, rot, cache, pp = _setup(wl, lens, 128)
    pos = np.array([[L - 1] for L in lens])
    got = _run(cache, inst.q[:, None], lens, pos, max(lens))
    ref = H.decode(cache, inst.q, lens)
    np.testing.assert_array_equal(got[:, 0], ref)


@pytest.mark.parametrize("wl,lens,W", [(synth.TINY, [512, 300], 64),
                                       (synth.QWEN3_8B_32K, [3000, 1400], 128)])
def test_rows_match_oracle_over_stored_codes(wl, lens, W):
    inst, rot, cache, pp = _setup(wl, lens, W)
    rng = np.random.default_rng(9)
    # the last 4 positions (a chunk), one deep inside the INT2 region, one in the sink
    pos = np.array([[L - 4, L - 3, L - 2, L - 1, L // 3, 2] for L in lens])
    M = pos.shape[1]
    q_rows = np.stack([synth.bf16_round(rng.standard_normal(inst.q.shape).astype(np.float32))
                       for _ in range(M)], axis=1)
    got = _run(cache, q_rows, lens, pos, max(lens))
    for m in range(M):
        ref = H.attention_from_pools(cache, pp, q_rows[:, m], lens, rot, sink=4, window=W,
                                     gqa=wl.gqa, upto=pos[:, m])
        H.check_close(got[:, m], ref, f"row {m}")
    assert H.status(cache) == 0


def test_position_outside_the_cache_is_reported():
    wl = synth.TINY
    lens = [300]
    inst, rot, cache, pp = _setup(wl, lens, 64)
    pos = np.array([[299, 300]])                      # 300 is past the cache
    got = _run(cache, np.stack([inst.q, inst.q], axis=1), lens, pos, 300)
    assert H.status(cache) & H.lib().DEVERR_SEQ_LEN
    assert np.abs(got[0, 1]).max() == 0.0
    ref = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=64, gqa=4)
    H.check_close(got[:, 0], ref)


@pytest.mark.parametrize("g,M", [(1, 11), (2, 5), (4, 3), (1, 8)])
def test_packed_rows_match_oracle(g, M):
    """G query heads per KV head leave 8 - G of the tile's query columns to other
    rows of the sequence: 8 / G rows share each page read.  Positions spread over
    the sink, the INT2 region and the window, in no order."""
    wl = dataclasses.replace(synth.TINY, num_q_heads=g)
    lens = [700, 260]
    inst, rot, cache, pp = _setup(wl, lens, 64)
    rng = np.random.default_rng(20 + g)
    pos = np.stack([rng.permutation(np.concatenate([[L - 1, 1, L // 2], rng.integers(0, L, M)]))[:M]
                    for L in lens])
    q_rows = np.stack([synth.bf16_round(rng.standard_normal(inst.q.shape).astype(np.float32))
                       for _ in range(M)], axis=1)
    got = _run(cache, q_rows, lens, pos, max(lens))
    for m in range(M):
        ref = H.attention_from_pools(cache, pp, q_rows[:, m], lens, rot, sink=4, window=64,
                                     gqa=g, upto=pos[:, m])
        H.check_close(got[:, m], ref, f"G={g} row {m}")
    assert H.status(cache) == 0


def test_multiquery_workspace_grows_with_packing():
    """Fewer CTA units per sequence give each more splits, so the multi-row call
    asks for its own workspace size (at least the per-row decode's)."""
    wl = synth.QWEN3_8B_32K
    inst, rot, cache, pp = _setup(wl, [3000], 128)
    L = H.lib()
    assert L.oscar_multiquery_workspace_size(cache, 1, 16, 3000) >= \
        L.oscar_decode_workspace_size(cache, 16, 3000) > 0
    assert L.oscar_multiquery_workspace_size(cache, 1, 1, 3000) == L.oscar_decode_workspace_size(cache, 1, 3000)
