"""GPU parity of the INT4 cache variant (code_bits = 4: codes 0..15 kept as two
2-bit planes) against the oracle with sixteen levels: prefill on the
tensor-core and the CUDA-core paths, decode-step append, decode attention over
the stored pools, and the fused step."""
import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth
from oracle import attention, cache as ocache

pytestmark = pytest.mark.gpu


def _identity(d, hkv):
    eye = [np.eye(d, dtype=np.float32)] * hkv
    return ocache.Rotations(eye, eye, [np.float32(9.0)] * hkv, [np.float32(4.0)] * hkv)


@pytest.mark.parametrize("misalign", [False, True])
@pytest.mark.parametrize("wl,lens", [(synth.TINY, [512]), (synth.QWEN3_8B_32K, [300, 977])])
def test_int4_prefill_exact_rotation_is_bit_exact(wl, lens, misalign):
    """Identity rotation: y is exact, so every byte of the INT4 pools is fixed."""
    inst = synth.draw_instance(wl, n_calib=32, seq_lens=lens)
    W = 64 if wl.head_dim == 64 else 128
    rot = _identity(wl.head_dim, wl.num_kv_heads)
    cache, pp = H.make_cache(inst, rot, window=W, bits=4)
    H.prefill(cache, inst, misalign=misalign)
    exp = H.expected(inst, rot, pp, window=W, bits=4)
    got2, gotb = H.pools(cache)
    assert np.array_equal(got2[exp.int2_defined], exp.int2[exp.int2_defined])
    assert np.array_equal(gotb[exp.bf16_defined], exp.bf16[exp.bf16_defined])
    assert H.status(cache) == 0


@pytest.mark.parametrize("misalign", [False, True])
@pytest.mark.parametrize("wl,lens,W", [(synth.TINY, [512], 64),
                                       (synth.QWEN3_8B_32K, [1000, 2077, 131], 128)])
def test_int4_prefill_oscar_rotation_matches_oracle(wl, lens, W, misalign):
    """As the INT2 test: every group's decisions equal the oracle's sixteen-level
    quantiser of the kernel's traced rotated values, the rotation lies within
    its bound, and the pools differ from the exact-x R placement only inside
    flagged groups where the two values straddle a decision."""
    inst = synth.draw_instance(wl, n_calib=512, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=W, bits=4)
    y, where = H.prefill_trace(cache, inst, misalign=misalign)
    d = wl.head_dim
    kappa = H.kappa(d) if misalign else H.kappa_tc(d)
    rows = {b: (np.arange(n), y[s:s + n]) for b, (s, n) in where.items()}
    st = H.check_traced(cache, pp, inst, rot, rows, kappa, lens=inst.seq_lens, sink=4, window=W,
                        bits=4)
    exp = H.expected(inst, rot, pp, window=W, kappa=kappa, bits=4)
    H.compare_pools(cache, exp)
    H.report(f"int4 prefill[{wl.name},{lens},misalign={misalign}]", **st)
    # sixteen levels put four times as many decision boundaries in a group
    assert st["straddling_groups"] <= max(2, 0.02 * st["groups"])
    assert H.status(cache) == 0


def test_int4_append_steps_match_prefill_definition():
    t = H.torch()
    wl = synth.TINY
    L0, L1, W = 80, 133, 64
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=[L1, L1 - 7])
    rot = H.oracle_rotations(inst)
    lens1 = np.array([L1, L1 - 7])
    lens0 = lens1 - (L1 - L0)
    cache, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=L1 - L0, bits=4)
    H.prefill(cache, inst, lens=lens0)
    L = H.lib()
    hkv = wl.num_kv_heads
    for step in range(L1 - L0):
        cur = lens0 + step + 1
        kn = np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        vn = np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)] for b in range(2)])
        L.oscar_quantize_append(cache, H.bf16_tensor(kn), H.bf16_tensor(vn),
                                t.from_numpy(cur.astype(np.int32)).to(H.DEV))
    exp = H.expected(inst, rot, pp, window=W, lens=lens1, kappa=H.kappa(wl.head_dim), bits=4)
    H.compare_pools(cache, exp)
    assert H.status(cache) == 0


@pytest.mark.parametrize("wl,lens,W", [(synth.TINY, [512, 300], 64),
                                       (synth.QWEN3_8B_32K, [5000, 1503, 133], 128),
                                       (synth.QWEN3_32B_128K, [3000], 128)])
def test_int4_decode_matches_oracle_over_stored_pools(wl, lens, W):
    inst = synth.draw_instance(wl, n_calib=512, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=W, bits=4)
    H.prefill(cache, inst)
    got = H.decode(cache, inst.q, inst.seq_lens)
    ref = H.attention_from_pools(cache, pp, inst.q, inst.seq_lens, rot, sink=4, window=W,
                                 gqa=wl.gqa)
    H.check_close(got, ref, f"INT4 decode {wl.name}")
    assert H.status(cache) == 0


def test_int4_is_closer_to_bf16_than_int2():
    """Sixteen levels reconstruct the history better: the INT4 cache's output
    is nearer all-BF16 attention than the INT2 cache's, on the same tokens."""
    wl = synth.QWEN3_8B_32K
    lens = [4000, 2500]
    inst = synth.draw_instance(wl, n_calib=512, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    bf = attention.bf16_decode(inst.q, inst.k, inst.v, inst.seq_lens, gqa=wl.gqa)
    err = {}
    for bits in (2, 4):
        cache, pp = H.make_cache(inst, rot, window=128, bits=bits)
        H.prefill(cache, inst)
        err[bits] = attention.rel_l2(H.decode(cache, inst.q, inst.seq_lens), bf)
    assert err[4] < 0.5 * err[2], err


def test_int4_fused_step_equals_append_then_decode():
    t = H.torch()
    L = H.lib()
    wl = synth.QWEN3_8B_32K
    lens0 = np.array([2000, 1503, 133])
    steps, W = 3, 128
    lens1 = lens0 + steps
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens1)
    rot = H.oracle_rotations(inst)
    fused, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=steps, bits=4)
    split, _ = H.make_cache(inst, rot, window=W, lens=lens0, growth=steps, bits=4)
    H.prefill(fused, inst, lens=lens0)
    H.prefill(split, inst, lens=lens0)
    B, hkv = len(lens0), wl.num_kv_heads
    q = H.bf16_tensor(inst.q)
    max_len = int(lens1.max())
    ws = t.zeros(L.oscar_decode_workspace_size(fused, B, max_len) // 4 + 64, dtype=t.float32,
                 device=H.DEV)
    for st in range(steps):
        cur = lens0 + st + 1
        kn = H.bf16_tensor(np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)] for b in range(B)]))
        vn = H.bf16_tensor(np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)] for b in range(B)]))
        lt = t.from_numpy(cur.astype(np.int32)).to(H.DEV)
        o_fused = t.zeros(inst.q.shape, dtype=t.bfloat16, device=H.DEV)
        L.oscar_decode_step(fused, q, kn, vn, lt, max_len, o_fused, ws)
        L.oscar_quantize_append(split, kn, vn, lt)
        o_split = t.zeros_like(o_fused)
        L.oscar_decode_attention(split, q, lt, max_len, o_split, ws)
        t.cuda.synchronize()
        got = H.from_bf16(o_fused)
        H.check_close(got, H.from_bf16(o_split), f"INT4 fused vs separate, step {st}")
        ref = H.attention_from_pools(fused, pp, inst.q, cur, rot, sink=4, window=W, gqa=wl.gqa)
        H.check_close(got, ref, f"INT4 fused vs oracle over the stored pools, step {st}")
    f2, fb = H.pools(fused)
    s2, sb = H.pools(split)
    np.testing.assert_array_equal(f2, s2)
    np.testing.assert_array_equal(fb, sb)
    exp = H.expected(inst, rot, pp, window=W, lens=lens1, kappa=H.kappa(wl.head_dim), bits=4)
    H.compare_pools(fused, exp)   # bytes outside flagged near-boundary entries are exact
    assert H.status(fused) == 0 and H.status(split) == 0
