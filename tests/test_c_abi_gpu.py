"""The device calls of the C ABI from plain C: tests/c_abi/decode_from_c.c
(C11, the CUDA runtime API, no Python in between) places one prompt with
oscar_prefill_quantize and attends one decode query with
oscar_decode_attention.  Its output matches the oracle's attention and is, byte
for byte, the output of the same calls made through the Python binding (whose
page plan uses other physical page ids)."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import build as build_mod
from int2_rotated_kv_gb300 import synth
from oracle import attention

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is not available")
    H.lib()   # builds the library if needed
    out = str(tmp_path_factory.mktemp("c_abi") / "decode_from_c")
    libdir = os.path.dirname(build_mod.LIB)
    cmd = ["gcc", "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c_abi", "decode_from_c.c"),
           "-L", libdir, "-loscar", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + libdir, "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_decode_from_c(program, tmp_path):
    wl, L, W = synth.TINY, 700, 64
    inst = synth.draw_instance(wl, n_calib=512, seq_lens=[L])
    rot = H.oracle_rotations(inst)
    d, hkv, hq = wl.head_dim, wl.num_kv_heads, wl.num_q_heads
    k = np.stack([inst.k[0][h] for h in range(hkv)], axis=1)     # [L][hkv][d]
    v = np.stack([inst.v[0][h] for h in range(hkv)], axis=1)
    blob = struct.pack("<6i", d, hkv, hq, 4, W, L)
    for a in (k, v, inst.q[0]):
        blob += synth.bf16_bits(np.asarray(a, np.float32)).astype(np.uint16).tobytes()
    for a in (np.stack(rot.rk), np.stack(rot.rv), np.asarray(rot.ck), np.asarray(rot.cv)):
        blob += np.ascontiguousarray(a, np.float32).tobytes()
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    src.write_bytes(blob)
    r = subprocess.run([program, str(src), str(dst)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stderr)
    buf = dst.read_bytes()
    st = np.frombuffer(buf, np.int32, 4, 0)
    assert (st == 0).all(), st
    bits = np.frombuffer(buf, np.uint16, hq * d, 16).reshape(hq, d)
    got = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = attention.mixed_decode(inst.q[:1], [inst.k[0]], [inst.v[0]], [L], rot, sink=4,
                                 window=W, gqa=wl.gqa)[0]
    H.check_close(got, ref, "decode from C vs oracle")
    cache, _ = H.make_cache(inst, rot, window=W)
    H.prefill(cache, inst)
    via_binding = H.decode(cache, inst.q, inst.seq_lens)[0]
    np.testing.assert_array_equal(got, via_binding)
