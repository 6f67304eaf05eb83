"""GPU parity of the decode step with host buffers (oscar_decode_step_host):
the step's q, k_new, v_new in one host buffer and the output written back to
host memory inside the call, read and written in place when the buffers are
mapped page-locked memory, through the staging copies when they are ordinary
(pageable) memory.  Its output and pools are the bytes of the device-buffer
step on an identical cache, and its output matches the oracle's attention over
the stored pools."""
import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl,lens0,steps,W,rope,pinned", [
    (synth.TINY, [200, 140, 66], 3, 64, 0.0, True),  # d=64, G=4; the window boundary is crossed
    (synth.TINY, [200, 140, 66], 3, 64, 0.0, False),
    (synth.QWEN3_8B_32K, [2000, 1503, 133], 2, 128, 0.0, True),
    (synth.QWEN3_8B_32K, [2000, 1503, 133], 2, 128, 0.0, False),
    (synth.QWEN3_8B_32K, [1200, 700], 2, 128, 1e6, True),  # with the rotary step
])
def test_host_step_equals_device_step(wl, lens0, steps, W, rope, pinned):
    t = H.torch()
    L = H.lib()
    lens0 = np.array(lens0)
    lens1 = lens0 + steps
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens1)
    rot = H.oracle_rotations(inst)
    host_c, pp = H.make_cache(inst, rot, window=W, lens=lens0, growth=steps)
    dev_c, _ = H.make_cache(inst, rot, window=W, lens=lens0, growth=steps)
    H.prefill(host_c, inst, lens=lens0)
    H.prefill(dev_c, inst, lens=lens0)
    B, hkv, G = len(lens0), wl.num_kv_heads, wl.gqa
    max_len = int(lens1.max())
    ws = t.zeros(L.oscar_decode_workspace_size(dev_c, B, max_len) // 4 + 64, dtype=t.float32,
                 device=H.DEV)
    need = L.oscar_decode_step_host_staging_size(host_c, B)
    staging = t.empty(need // 4 + 4, dtype=t.float32, device=H.DEV)
    q = H.bf16_tensor(inst.q)
    out_host = t.empty(tuple(inst.q.shape), dtype=t.bfloat16)
    if pinned:
        out_host = out_host.pin_memory()
    for st in range(steps):
        cur = lens0 + st + 1
        kn = H.bf16_tensor(np.stack([[inst.k[b][h][cur[b] - 1] for h in range(hkv)]
                                     for b in range(B)]))
        vn = H.bf16_tensor(np.stack([[inst.v[b][h][cur[b] - 1] for h in range(hkv)]
                                     for b in range(B)]))
        lt = t.from_numpy(cur.astype(np.int32)).to(H.DEV)
        in_host = t.cat([q.reshape(-1), kn.reshape(-1), vn.reshape(-1)]).cpu()
        if pinned:
            in_host = in_host.pin_memory()
        out_host.fill_(0)
        L.oscar_decode_step_host(host_c, in_host, lt, max_len, out_host, staging, ws, rope_base=rope)
        o_dev = t.zeros(inst.q.shape, dtype=t.bfloat16, device=H.DEV)
        if rope > 0:
            L.oscar_decode_step_rope(dev_c, q, kn, vn, lt, max_len, rope, o_dev, ws)
        else:
            L.oscar_decode_step(dev_c, q, kn, vn, lt, max_len, o_dev, ws)
        t.cuda.synchronize()
        np.testing.assert_array_equal(out_host.view(t.int16).numpy(),
                                      o_dev.cpu().view(t.int16).numpy(), err_msg=f"step {st}")
        if rope == 0:
            ref = H.attention_from_pools(host_c, pp, inst.q, cur, rot, sink=4, window=W, gqa=G)
            H.check_close(H.from_bf16(o_dev.cpu()), ref, f"host step vs oracle, step {st}")
    h2, hb = H.pools(host_c)
    d2, db = H.pools(dev_c)
    np.testing.assert_array_equal(h2, d2)
    np.testing.assert_array_equal(hb, db)
    assert H.status(host_c) == 0 and H.status(dev_c) == 0


def test_host_step_rejects_small_staging():
    t = H.torch()
    L = H.lib()
    wl = synth.TINY
    lens = np.array([100])
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens + 1)
    rot = H.oracle_rotations(inst)
    c, _ = H.make_cache(inst, rot, window=64, lens=lens, growth=1)
    need = L.oscar_decode_step_host_staging_size(c, 1)
    staging = t.empty(need - 16, dtype=t.uint8, device=H.DEV)
    ws = t.zeros(L.oscar_decode_workspace_size(c, 1, 101) // 4 + 64, dtype=t.float32, device=H.DEV)
    in_host = t.zeros(need, dtype=t.uint8).pin_memory()
    out_host = t.zeros(tuple(inst.q.shape), dtype=t.bfloat16).pin_memory()
    lt = t.tensor([101], dtype=t.int32, device=H.DEV)
    with pytest.raises(L.OscarError) as e:
        L.oscar_decode_step_host(c, in_host, lt, 101, out_host, staging, ws)
    assert e.value.status == -3
    t.cuda.synchronize()
    assert int(out_host.view(t.int16).abs().sum()) == 0   # nothing was queued
