"""GPU parity of the fused decode step (append + attention in one call): against
the same two steps issued separately, its attention against the oracle's over
the stored pools, and the pools against the oracle's placement (flags allowed)."""
import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl,lens0,steps,W", [
    (synth.TINY, [200, 140, 66], 5, 64),             # d=64, G=4, one KV head; one sequence
                                                      # crosses S+W during the steps
    (synth.QWEN3_8B_32K, [2000, 1503, 133], 3, 128),  # several splits per head
    # 40 sequences x 8 KV heads: more split CTAs than fit at once, so the step
    # runs with the append kernel in front instead of as one launch
    (synth.QWEN3_8B_32K, [300 + 7 * i for i in range(40)], 2, 128),
])
def test_fused_step_equals_append_then_decode(wl, lens0, steps, W):
    t = H.torch()
    L = H.lib()
    lens0 = np.array(lens0)
    lens1 = lens0 + steps
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens1)
    rot = H.oracle_rotations(inst)
    fused, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=steps)
    split, _ = H.make_cache(inst, rot, window=W, lens=lens0, growth=steps)
    H.prefill(fused, inst, lens=lens0)
    H.prefill(split, inst, lens=lens0)
    B, hkv, G = len(lens0), wl.num_kv_heads, wl.gqa
    q = H.bf16_tensor(inst.q)
    max_len = int(lens1.max())
    ws = t.zeros(L.oscar_decode_workspace_size(fused, B, max_len) // 4 + 64, dtype=t.float32,
                 device=H.DEV)
    for st in range(steps):
        cur = lens0 + st + 1
        kn = H.bf16_tensor(np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)]
                                     for b in range(B)]))
        vn = H.bf16_tensor(np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)]
                                     for b in range(B)]))
        lt = t.from_numpy(cur.astype(np.int32)).to(H.DEV)
        o_fused = t.zeros(inst.q.shape, dtype=t.bfloat16, device=H.DEV)
        L.oscar_decode_step(fused, q, kn, vn, lt, max_len, o_fused, ws)
        L.oscar_quantize_append(split, kn, vn, lt)
        o_split = t.zeros_like(o_fused)
        L.oscar_decode_attention(split, q, lt, max_len, o_split, ws)
        t.cuda.synchronize()
        got = H.from_bf16(o_fused)
        H.check_close(got, H.from_bf16(o_split), f"fused vs separate, step {st}")
        ref = H.attention_from_pools(fused, pp, inst.q, cur, rot, sink=4, window=W, gqa=G)
        H.check_close(got, ref, f"fused vs oracle over the stored pools, step {st}")
    # the append part of both paths writes the same bytes, which are the oracle's
    # placement up to flagged near-boundary codes
    f2, fb = H.pools(fused)
    s2, sb = H.pools(split)
    np.testing.assert_array_equal(f2, s2)
    np.testing.assert_array_equal(fb, sb)
    exp = H.expected(inst, rot, pp, window=W, lens=lens1, kappa=H.kappa(wl.head_dim))
    H.compare_pools(fused, exp)   # bytes outside flagged near-boundary entries are exact
    assert H.status(fused) == 0 and H.status(split) == 0
