"""oscar_decode_attention_static: decode attention for callers that cannot
allocate device memory.

A plug-in running inside a runtime that owns every device allocation, or a
latency-bound loop that must never enter the allocator, has no workspace to
pass.  The static entry point uses a fixed scratch buffer compiled into the
library instead.  It runs the same plan and kernels as the regular call that
takes a workspace, so its output must be the same bytes, and both must agree
with the oracle's attention over the stored pools.  This file is collected last
on purpose: it exercises process-wide state (the one shared buffer), so a run
that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 16 << 20


def _static(L, cache, q, lt, batch, max_len, out):
    d = cache.desc()
    t = H.torch()
    return L.lib().oscar_decode_attention_static(ctypes.byref(d), q.data_ptr(), lt.data_ptr(),
                                                 batch, max_len, out.data_ptr(),
                                                 t.cuda.current_stream().cuda_stream)


def test_static_scratch_matches_workspace_call():
    t = H.torch()
    L = H.lib()
    wl = synth.QWEN3_8B_32K
    lens = [3000, 1250]
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, pp = H.make_cache(inst, rot, window=128)
    H.prefill(cache, inst)
    ref = H.decode(cache, inst.q, inst.seq_lens)          # the workspace entry point
    oracle = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=128, gqa=wl.gqa)
    H.check_close(ref, oracle, "workspace call vs oracle")
    q = H.bf16_tensor(inst.q)
    lt = t.from_numpy(np.asarray(lens, np.int32)).to(H.DEV)
    for _ in range(2):                                     # the buffer keeps the last call's data
        out = t.full(inst.q.shape, float("nan"), dtype=t.bfloat16, device=H.DEV)
        L.oscar_decode_attention_static(cache, q, lt, max(lens), out)
        t.cuda.synchronize()
        got = H.from_bf16(out)
        np.testing.assert_array_equal(got, ref)            # same plan, same kernels: same bytes
        H.check_close(got, oracle, "static scratch vs oracle")
    assert H.status(cache) == 0


def _largest_batch(L, cache, max_len):
    """The largest batch whose workspace fits the static buffer (the plan, and
    so the size, depends on the device's SM count)."""
    lo, hi = 1, 1
    while L.oscar_decode_workspace_size(cache, hi, max_len) <= STATIC_SCRATCH_BYTES:
        lo, hi = hi, hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if L.oscar_decode_workspace_size(cache, mid, max_len) <= STATIC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_static_scratch_at_its_size_limit():
    """At the largest batch whose workspace fits the buffer the call runs and
    gives the workspace call's bytes; one sequence more is refused before any
    launch with OSCAR_ERR_WORKSPACE."""
    t = H.torch()
    L = H.lib()
    wl = synth.QWEN3_8B_32K
    L0 = 230                         # 4 sink + 98 INT2 + 128 recent tokens
    probe = synth.draw_instance(wl, n_calib=64, seq_lens=[L0])
    rot = H.oracle_rotations(probe)
    cache0, _ = H.make_cache(probe, rot, window=128)
    B = _largest_batch(L, cache0, L0)
    assert 8 < B < 4096
    lens = [L0 - (b % 7) for b in range(B)]
    inst = synth.draw_instance(wl, n_calib=64, seq_lens=lens)
    cache, pp = H.make_cache(inst, rot, window=128)
    H.prefill(cache, inst)
    assert L.oscar_decode_workspace_size(cache, B, L0) <= STATIC_SCRATCH_BYTES
    assert L.oscar_decode_workspace_size(cache, B + 1, L0) > STATIC_SCRATCH_BYTES
    ref = H.decode(cache, inst.q, lens, max_len=L0)
    q = H.bf16_tensor(inst.q)
    lt = t.from_numpy(np.asarray(lens, np.int32)).to(H.DEV)
    out = t.full(inst.q.shape, float("nan"), dtype=t.bfloat16, device=H.DEV)
    assert _static(L, cache, q, lt, B, L0, out) == 0
    t.cuda.synchronize()
    got = H.from_bf16(out)
    np.testing.assert_array_equal(got, ref)
    sample = [0, 1, B // 2, B - 1]
    oracle = H.attention_from_pools(cache, pp, inst.q, lens, rot, sink=4, window=128, gqa=wl.gqa,
                                    seqs=sample)
    H.check_close(got[sample], oracle[sample], "static scratch at its limit vs oracle")
    # one more sequence: refused, nothing launched (the output keeps its fill)
    q1 = t.zeros((B + 1, wl.num_q_heads, wl.head_dim), dtype=t.bfloat16, device=H.DEV)
    lt1 = t.ones(B + 1, dtype=t.int32, device=H.DEV)
    out1 = t.zeros_like(q1)
    assert _static(L, cache, q1, lt1, B + 1, L0, out1) == -3   # OSCAR_ERR_WORKSPACE
    t.cuda.synchronize()
    assert float(out1.float().abs().max()) == 0.0
    assert H.status(cache) == 0
