"""C-ABI library on the host: it builds, loads, exports every symbol the header
declares, its host calls (calibration covariances, rotation builder) agree with
the oracle, and bad arguments are rejected before any kernel launch."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from int2_rotated_kv_gb300 import build as build_mod
from int2_rotated_kv_gb300 import synth
from oracle import rotation

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(build_mod.LIB):
        build_mod.build()
    from int2_rotated_kv_gb300 import _lib
    return _lib


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "oscar.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(oscar_[a-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", build_mod.LIB], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\b(oscar_\w+)\b", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert set(L.EXPORTED) == set(names)
    for n in names:
        getattr(L.lib(), n)
    assert L.oscar_version() >= 100
    assert L.lib().oscar_status_string(-3).decode() == "workspace too small"


def test_query_covariance_matches_oracle(L):
    rng = np.random.default_rng(0)
    q = rng.standard_normal((300, 4, 64)).astype(np.float32)
    np.testing.assert_allclose(L.oscar_query_covariance(q), rotation.query_covariance(q),
                               rtol=1e-12, atol=1e-14)


def test_score_covariance_matches_oracle(L):
    rng = np.random.default_rng(1)
    n, g, d = 160, 2, 64
    q = rng.standard_normal((n, g, d)).astype(np.float32)
    k = rng.standard_normal((n, d)).astype(np.float32)
    v = rng.standard_normal((n, d)).astype(np.float32)
    ref = rotation.score_covariance(q, k, v)
    for nt in (1, 3):
        np.testing.assert_allclose(L.oscar_score_covariance(q, k, v, nt), ref, rtol=1e-10,
                                   atol=1e-13)


@pytest.mark.parametrize("d", [64, 128])
def test_build_rotation_matches_oracle(L, d):
    inst = synth.draw_instance(synth.TINY if d == 64 else synth.QWEN3_8B_32K, n_calib=512,
                               seq_lens=[64])
    q, k = inst.calib_q[0], inst.calib_k[0]
    c = rotation.query_covariance(q)
    r64, r32, clip, ev = L.oscar_build_rotation(c, k, 99.9, L.VARIANT_OSCAR)
    ref_ev, _ = rotation.sorted_eigh(c)
    np.testing.assert_allclose(ev, ref_ev, rtol=1e-9, atol=1e-12 * abs(ref_ev).max())
    assert np.abs(r64.T @ r64 - np.eye(d)).max() <= 1e-9
    ref_r = rotation.composite_rotation(c, d)
    np.testing.assert_allclose(r64, ref_r, atol=1e-8)
    np.testing.assert_array_equal(r32, r64.astype(np.float32))
    # eigen residual of the recovered basis
    u = r64 @ rotation.bit_reversal_matrix(d).T @ rotation.hadamard(d).T
    assert np.linalg.norm(c @ u - u * ev) <= 1e-10 * np.linalg.norm(c)
    ref_clip = np.float32(rotation.clip_threshold(k, r32, 99.9))
    assert clip == pytest.approx(float(ref_clip), rel=2e-7)


def test_build_rotation_variants_and_errors(L):
    x = np.random.default_rng(2).standard_normal((50, 8)).astype(np.float32)
    _, r, _, _ = L.oscar_build_rotation(None, x, 99.9, L.VARIANT_IDENTITY)
    np.testing.assert_array_equal(r, np.eye(8, dtype=np.float32))
    _, r, _, _ = L.oscar_build_rotation(None, x, 99.9, L.VARIANT_HADAMARD)
    np.testing.assert_allclose(r, rotation.hadamard(8), atol=1e-7)
    with pytest.raises(L.OscarError) as e:
        L.oscar_build_rotation(np.eye(8), x, 99.9, L.VARIANT_OSCAR)   # degenerate spectrum
    assert e.value.status == -5
    with pytest.raises(L.OscarError):
        L.oscar_build_rotation(None, x, 99.9, L.VARIANT_OSCAR)        # C missing
    with pytest.raises(L.OscarError):
        L.oscar_build_rotation(None, np.zeros((4, 12), np.float32), 99.9, L.VARIANT_IDENTITY)


def _desc(L, **kw):
    base = dict(num_kv_heads=1, num_q_heads=4, head_dim=64, sink=4, window=64, max_pages_per_seq=8,
                num_int2_pages=8, num_bf16_pages=8, int2_pool=256, bf16_pool=512,
                int2_page_table=1024, bf16_page_table=2048, r_k=4096, r_v=8192, clip_k=16384,
                clip_v=32768, status=None)
    base.update(kw)
    return L.CacheDesc(**base)


def test_argument_errors_before_any_launch(L):
    lib = L.lib()
    ok = _desc(L)
    # shapes outside the supported set
    for bad, want in ((dict(head_dim=96), -2), (dict(num_q_heads=12, num_kv_heads=1), -2),
                      (dict(num_q_heads=6, num_kv_heads=4), -1), (dict(window=0), -1),
                      (dict(int2_pool=None), -1), (dict(int2_pool=257), -1),
                      (dict(code_bits=3), -2), (dict(code_bits=8), -2)):
        d = _desc(L, **bad)
        st = lib.oscar_decode_attention(ctypes.byref(d), 4096, 4096, 1, 16, 4096, 4096, 1 << 20, None)
        assert st == want, (bad, st)
    assert lib.oscar_decode_attention(None, 1, 1, 1, 1, 1, 1, 1, None) == -1
    # the INT4 variant (code_bits 4) passes the same checks as INT2 (2, or 0)
    for bits in (0, 2, 4):
        d4 = _desc(L, code_bits=bits)
        assert lib.oscar_decode_attention(ctypes.byref(d4), 4096, 4096, 1, 16, 4096, 4096, 8,
                                          None) == -3
    # null buffers, bad sizes
    assert lib.oscar_decode_attention(ctypes.byref(ok), None, 4096, 1, 16, 4096, 4096, 1 << 20, None) == -1
    assert lib.oscar_decode_attention(ctypes.byref(ok), 4096, 4096, 1, 0, 4096, 4096, 1 << 20, None) == -1
    assert lib.oscar_decode_attention(ctypes.byref(ok), 4096, 4096, 1, 10 ** 6, 4096, 4096, 1 << 20,
                                      None) == -1                        # beyond the page table
    assert lib.oscar_decode_attention(ctypes.byref(ok), 4096, 4096, 1, 16, 4096, 4100, 1 << 20,
                                      None) == -1                        # misaligned workspace
    assert lib.oscar_decode_attention(ctypes.byref(ok), 4096, 4096, 1, 16, 4096, 4096, 8, None) == -3
    assert lib.oscar_decode_attention(ctypes.byref(ok), 4096, 4096, 0, 16, 4096, 4096, 8, None) == 0
    assert lib.oscar_decode_workspace_size(ctypes.byref(ok), 1, 16) > 0
    assert lib.oscar_decode_workspace_size(ctypes.byref(ok), 0, 16) == 0
    assert lib.oscar_prefill_quantize(ctypes.byref(ok), None, 1, 1, 1, 1, 1, 5, None) == -1
    assert lib.oscar_prefill_quantize(ctypes.byref(ok), 1, 1, 1, 1, 1, 0, 5, None) == -1
    assert lib.oscar_prefill_quantize(ctypes.byref(ok), 1, 1, 1, 1, 1, 1, 0, None) == 0
    assert lib.oscar_quantize_append(ctypes.byref(ok), None, 1, 1, 2, None) == -1
    for base in (1.0, -3.0, float("inf"), float("nan")):     # rotary base checked first
        assert lib.oscar_decode_step_rope(ctypes.byref(ok), 4096, 4096, 4096, 4096, 1, 16, base,
                                          4096, 4096, 1 << 20, None) == -1
    assert lib.oscar_decode_step_rope(ctypes.byref(ok), 4096, None, 4096, 4096, 1, 16, 1e6,
                                      4096, 4096, 1 << 20, None) == -1
    assert lib.oscar_quantize_append(ctypes.byref(ok), 1, 1, 1, -1, None) == -1
    bf_only = _desc(L, int2_pool=None, int2_page_table=None, r_k=None, r_v=None, clip_k=None,
                    clip_v=None)
    assert lib.oscar_quantize_append(ctypes.byref(bf_only), 1, 1, 1, 2, None) == -1
    assert lib.oscar_decode_attention_bf16(ctypes.byref(bf_only), 4096, 4096, 1, 16, 4096, 4096, 8,
                                           None) == -3   # reaches the workspace check
    # the no-allocation entry point checks its arguments as the workspace call
    # does, before it sizes the plan against its fixed scratch buffer
    st = lib.oscar_decode_attention_static
    assert st(ctypes.byref(ok), 4096, 4096, 1, 10 ** 6, 4096, None) == -1   # beyond the page table
    assert st(ctypes.byref(ok), None, 4096, 1, 16, 4096, None) == -1
    assert st(ctypes.byref(ok), 4096, None, 1, 16, 4096, None) == -1
    assert st(ctypes.byref(ok), 4096, 4096, 1, 16, 4098, None) == -1       # misaligned output
    assert st(ctypes.byref(ok), 4096, 4096, -1, 16, 4096, None) == -1
    assert st(ctypes.byref(ok), 4096, 4096, 0, 16, 4096, None) == 0
    assert st(ctypes.byref(_desc(L, head_dim=96)), 4096, 4096, 1, 16, 4096, None) == -2


def test_host_step_staging_and_argument_errors_before_any_copy(L):
    """oscar_decode_step_host: staging = inputs (q, k_new, v_new back to back),
    then the output from the next multiple of 256 bytes; every argument is
    checked before the first copy is queued."""
    lib = L.lib()
    ok = _desc(L)                                    # Hkv 1, Hq 4, d 64
    # batch 3: q 3*4*64*2 = 1536 B, k and v 384 B each: inputs 2304 B (a multiple
    # of 256), output 1536 B from there
    assert lib.oscar_decode_step_host_staging_size(ctypes.byref(ok), 3) == 2304 + 1536
    g1 = _desc(L, num_q_heads=1)                     # inputs 384 B -> output from 512
    assert lib.oscar_decode_step_host_staging_size(ctypes.byref(g1), 1) == 512 + 128
    assert lib.oscar_decode_step_host_staging_size(ctypes.byref(ok), 0) == 0
    assert lib.oscar_decode_step_host_staging_size(None, 1) == 0
    need = lib.oscar_decode_step_host_staging_size(ctypes.byref(ok), 1)

    def call(in_host=4096, batch=1, max_len=16, rope=0.0, out_host=8192, staging=1 << 16,
             staging_bytes=need, ws_bytes=1 << 20, desc=ok):
        return lib.oscar_decode_step_host(ctypes.byref(desc) if desc is not None else None,
                                          in_host, 4096, batch, max_len, rope, out_host, staging,
                                          staging_bytes, 1 << 20, ws_bytes, None)

    assert call(desc=None) == -1
    assert call(in_host=None) == -1
    assert call(out_host=None) == -1
    assert call(staging=None) == -1
    assert call(staging=(1 << 16) + 8) == -1          # staging not 16-byte aligned
    assert call(staging_bytes=need - 1) == -3
    for rope in (0.5, 1.0, -1.0, float("inf"), float("nan")):
        assert call(rope=rope) == -1, rope
    assert call(max_len=0) == -1
    assert call(batch=-1) == -1
    assert call(ws_bytes=8) == -3                     # the decode step's own workspace check
    assert call(batch=0) == 0
    assert call(desc=_desc(L, head_dim=96)) == -2


def test_calibration_argument_errors_before_any_launch(L):
    lib = L.lib()
    ws = lambda *a: lib.oscar_calibration_workspace_size(*a)
    assert ws(8, 32, 128, 8192) > 2 * 8192 * 32 * 128 * 2      # holds the O pair at least
    assert ws(1, 4, 64, 1) > 0
    for bad in ((8, 32, 96, 100), (8, 24, 128, 100), (8, 36, 128, 100), (0, 4, 64, 10),
                (1, 4, 64, 0), (1, 4, 64, (1 << 24) + 1)):
        assert ws(*bad) == 0, bad
    big = 1 << 30
    # shape errors come first, then null / misaligned pointers, then the workspace size
    assert lib.oscar_query_covariance_device(1, 4, 96, 10, 4096, 4096, 4096, big, None) == -2
    assert lib.oscar_query_covariance_device(2, 3, 64, 10, 4096, 4096, 4096, big, None) == -1
    assert lib.oscar_query_covariance_device(1, 4, 64, 10, None, 4096, 4096, big, None) == -1
    assert lib.oscar_query_covariance_device(1, 4, 64, 10, 4100, 4096, 4096, big, None) == -1
    assert lib.oscar_query_covariance_device(1, 4, 64, 10, 4096, 4096, 4096, 64, None) == -3
    assert lib.oscar_score_covariance_device(1, 32, 64, 10, 4096, 4096, 4096, 4096, 4096, big,
                                             None) == -2                 # G = 32
    assert lib.oscar_score_covariance_device(1, 4, 64, 10, 4096, None, 4096, 4096, 4096, big,
                                             None) == -1
    assert lib.oscar_score_covariance_device(1, 4, 64, 10, 4096, 4096, 4096, 4096, 4096, 64,
                                             None) == -3
    assert lib.oscar_clip_threshold_device(1, 64, 10, 4096, 4096, 100.5, 4096, 4096, big,
                                           None) == -1
    assert lib.oscar_clip_threshold_device(1, 64, 10, 4096, 4096, float("nan"), 4096, 4096, big,
                                           None) == -1
    assert lib.oscar_clip_threshold_device(1, 64, 10, 4096, None, 99.9, 4096, 4096, big,
                                           None) == -1
    assert lib.oscar_clip_threshold_device(1, 64, 10, 4096, 4096, 99.9, 4096, 4096, 64,
                                           None) == -3
