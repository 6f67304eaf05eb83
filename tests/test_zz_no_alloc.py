"""oscar_decode_attention_static: decode attention for callers that cannot
allocate device memory.

A plug-in running inside a runtime that owns every device allocation, or a
latency-bound loop that must never enter the allocator, has no workspace to
pass.  The static entry point uses a fixed scratch buffer compiled into the
library instead, and must give the same output as the regular call that takes a
workspace.  This file is collected last on purpose: it exercises process-wide
state (the one shared buffer), so a run that stops at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import synth

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 16 << 20


def test_static_scratch_matches_workspace_call():
    t = H.torch()
    L = H.lib()
    wl = synth.QWEN3_8B_32K
    lens = [3000, 1250]
    inst = synth.draw_instance(wl, n_calib=256, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, _ = H.make_cache(inst, rot, window=128)
    H.prefill(cache, inst)
    ref = H.decode(cache, inst.q, inst.seq_lens)          # the workspace entry point
    q = H.bf16_tensor(inst.q)
    lt = t.from_numpy(np.asarray(lens, np.int32)).to(H.DEV)
    outs = []
    for _ in range(2):                                     # the buffer keeps the last call's data
        out = t.full(inst.q.shape, float("nan"), dtype=t.bfloat16, device=H.DEV)
        L.oscar_decode_attention_static(cache, q, lt, max(lens), out)
        t.cuda.synchronize()
        got = H.from_bf16(out)
        H.check_close(got, ref, "static scratch vs workspace call")
        outs.append(got)
    np.testing.assert_array_equal(outs[0], outs[1])
    assert H.status(cache) == 0


def test_static_scratch_rejects_oversized_shapes():
    t = H.torch()
    L = H.lib()
    wl = synth.QWEN3_8B_32K
    lens = [3000, 1250]
    inst = synth.draw_instance(wl, n_calib=64, seq_lens=lens)
    rot = H.oracle_rotations(inst)
    cache, _ = H.make_cache(inst, rot, window=128)
    batch, max_len = 512, max(lens)
    # host-side query with the same plan: this shape needs more than the buffer
    need = L.oscar_decode_workspace_size(cache, batch, max_len)
    assert need > STATIC_SCRATCH_BYTES
    q = t.zeros((batch, wl.num_q_heads, wl.head_dim), dtype=t.bfloat16, device=H.DEV)
    lt = t.ones(batch, dtype=t.int32, device=H.DEV)
    out = t.zeros_like(q)
    d = cache.desc()
    st = L.lib().oscar_decode_attention_static(ctypes.byref(d), q.data_ptr(), lt.data_ptr(), batch,
                                               max_len, out.data_ptr(),
                                               t.cuda.current_stream().cuda_stream)
    assert st == -3                                        # OSCAR_ERR_WORKSPACE, nothing launched
    t.cuda.synchronize()
    assert float(out.float().abs().max()) == 0.0
