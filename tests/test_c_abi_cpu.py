"""The C ABI from plain C: tests/c_abi/host_calls.c is compiled as C99 against
include/oscar.h (warnings are errors), linked to liboscar.so, and run on seeded
calibration data; its query covariance, rotation, eigenvalues and clip are
checked against the oracle (oracle/rotation.py)."""
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

from int2_rotated_kv_gb300 import build as build_mod
from int2_rotated_kv_gb300 import synth
from oracle import rotation

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is not available")
    if not os.path.exists(build_mod.LIB):
        build_mod.build()
    out = str(tmp_path_factory.mktemp("c_abi") / "host_calls")
    libdir = os.path.dirname(build_mod.LIB)
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi", "host_calls.c"),
           "-L", libdir, "-loscar", "-Wl,-rpath," + libdir, "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_host_calls_from_c_match_oracle(program, tmp_path):
    d = 64
    inst = synth.draw_instance(synth.TINY, n_calib=512, seq_lens=[64])
    q = np.ascontiguousarray(inst.calib_q[0], np.float32)          # [n][g][d]
    x = np.ascontiguousarray(inst.calib_k[0], np.float32)          # [n][d]
    n, g = q.shape[0], q.shape[1]
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    src.write_bytes(struct.pack("<iiq", d, g, n) + q.tobytes() + x.tobytes())
    r = subprocess.run([program, str(src), str(dst)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stderr)
    buf = dst.read_bytes()
    st = np.frombuffer(buf, np.int32, 3, 0)
    assert (st == 0).all(), st
    version = np.frombuffer(buf, np.int32, 1, 12)[0]
    off = 16
    c = np.frombuffer(buf, np.float64, d * d, off).reshape(d, d); off += 8 * d * d
    r32 = np.frombuffer(buf, np.float32, d * d, off).reshape(d, d); off += 4 * d * d
    ev = np.frombuffer(buf, np.float64, d, off); off += 8 * d
    clip = np.frombuffer(buf, np.float32, 1, off)[0]; off += 4
    text = buf[off:].split(b"\0")[0].decode()
    assert version >= 100
    assert text == "workspace too small"
    ref_c = rotation.query_covariance(q)
    np.testing.assert_allclose(c, ref_c, rtol=1e-12, atol=1e-14)
    ref_ev, _ = rotation.sorted_eigh(ref_c)
    np.testing.assert_allclose(ev, ref_ev, rtol=1e-9, atol=1e-12 * abs(ref_ev).max())
    np.testing.assert_allclose(r32, rotation.composite_rotation(ref_c, d).astype(np.float32),
                               atol=1e-7)
    ref_clip = np.float32(rotation.clip_threshold(x, r32, 99.9))
    assert float(clip) == pytest.approx(float(ref_clip), rel=2e-7)
