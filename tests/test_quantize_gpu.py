"""GPU parity of the rotate + clip + INT2-quantise + pack path (prefill and
decode-append) against the oracle's expected page pools."""
import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth
from oracle import cache as ocache, layout

pytestmark = pytest.mark.gpu


def _exact_rotations(d, hkv, kind, seed=0):
    rng = np.random.default_rng(seed)
    rk, rv = [], []
    for _ in range(hkv):
        for dst in (rk, rv):
            if kind == "identity":
                dst.append(np.eye(d, dtype=np.float32))
            else:
                perm = rng.permutation(d)
                r = np.zeros((d, d), np.float32)
                r[np.arange(d), perm] = rng.choice([-1.0, 1.0], d)
                dst.append(r)
    return ocache.Rotations(rk, rv, [np.float32(9.0)] * hkv, [np.float32(4.0)] * hkv)


@pytest.mark.parametrize("kind", ["identity", "signed_permutation"])
@pytest.mark.parametrize("wl,lens", [(synth.TINY, [512]), (synth.QWEN3_8B_32K, [300, 977])])
def test_prefill_exact_rotation_is_bit_exact(kind, wl, lens):
    """With an exact rotation every entry of the pools is fixed: no flags at all."""
    inst = synth.draw_instance(wl, n_calib=32, seq_lens=lens)
    W = 64 if wl.head_dim == 64 else 128
    rot = _exact_rotations(wl.head_dim, wl.num_kv_heads, kind)
    cache, pp = H.make_cache(inst, rot, window=W)
    H.prefill(cache, inst)
    exp = H.expected(inst, rot, pp, window=W)
    got2, gotb = H.pools(cache)
    assert np.array_equal(got2[exp.int2_defined], exp.int2[exp.int2_defined])
    assert np.array_equal(gotb[exp.bf16_defined], exp.bf16[exp.bf16_defined])
    assert H.status(cache) == 0


@pytest.mark.parametrize("wl,lens,W", [(synth.TINY, [512], 64),
                                       (synth.QWEN3_8B_32K, [1000, 2077, 131], 128),
                                       (synth.QWEN3_32B_128K, [700], 128),
                                       # ~86 tiles of 128 tokens: every CTA of the bulk
                                       # prefill wraps its ring and both accumulators
                                       (synth.QWEN3_8B_32K, [6000, 5000], 128)])
def test_prefill_oscar_rotation_matches_oracle(wl, lens, W):
    inst = synth.draw_instance(wl, n_calib=512, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=W)
    H.prefill(cache, inst)
    exp = H.expected(inst, rot, pp, window=W, kappa=H.kappa(wl.head_dim))
    diff, flagged = H.compare_pools(cache, exp)
    token_heads = exp.int2_defined.sum() // (3 * wl.head_dim // 4)
    groups = token_heads * 2 * (wl.head_dim // 32)
    print(f"flagged groups {exp.n_flag_groups}/{groups}, flagged elements {exp.n_flag_elems}, "
          f"differing flagged bytes {diff}/{flagged}")
    # the flags come from a worst-case fp32 error bound; the kernel's actual
    # disagreements are far rarer than the flags
    assert exp.n_flag_groups <= 0.3 * groups
    assert diff <= 0.05 * flagged + 8
    assert H.status(cache) == 0


def test_append_steps_match_prefill_definition():
    """Prefill to L0, then append tokens one step at a time up to L1: the pools
    hold what the oracle places for length L1 (tokens that left the window are
    INT2, the window is BF16)."""
    t = H.torch()
    wl = synth.TINY
    L0, L1, W = 80, 133, 64
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=[L1, L1 - 7])
    rot = H.oracle_rotations(inst)
    lens1 = np.array([L1, L1 - 7])
    lens0 = lens1 - (L1 - L0)
    cache, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=L1 - L0)
    H.prefill(cache, inst, lens=lens0)
    L = H.lib()
    hkv, d = wl.num_kv_heads, wl.head_dim
    for step in range(L1 - L0):
        cur = lens0 + step + 1
        kn = np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        vn = np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        L.oscar_quantize_append(cache, H.bf16_tensor(kn), H.bf16_tensor(vn),
                                t.from_numpy(cur.astype(np.int32)).to(H.DEV))
    exp = H.expected(inst, rot, pp, window=W, lens=lens1, kappa=H.kappa(d))
    diff, flagged = H.compare_pools(cache, exp)
    assert diff <= flagged
    assert H.status(cache) == 0


def test_bad_page_ids_are_skipped_and_reported():
    """A page id beyond the pool is skipped by the kernel's own bounds check and
    reported in the status word; valid pages are still written."""
    t = H.torch()
    wl = synth.TINY
    inst = synth.draw_instance(wl, n_calib=64, seq_lens=[200])
    rot = _exact_rotations(64, 1, "identity")
    cache, pp = H.make_cache(inst, rot, window=64)
    tbl = pp.int2_table.copy()
    tbl[0, 3] = pp.num_int2_pages + 5          # out of range on purpose (checked in-kernel)
    cache.int2_page_table = t.from_numpy(tbl).to(H.DEV)
    H.prefill(cache, inst)
    assert H.status(cache) & H.lib().DEVERR_PAGE_ID
    got2, _ = H.pools(cache)
    exp = H.expected(inst, rot, pp, window=64)
    blk = layout.int2_block_bytes(64)
    ok = exp.int2_defined.copy()
    ok[pp.int2_table[0, 3] * blk:(pp.int2_table[0, 3] + 1) * blk] = False
    assert np.array_equal(got2[ok], exp.int2[ok])
