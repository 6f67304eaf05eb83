"""The fidelity report through the product path: for OSCAR, Hadamard-only and
unrotated INT2 ([Summary 1], [Summary 4], [Abstract]: the comparison the pages
draw), the library's own calibration (oscar_query_covariance,
oscar_score_covariance, oscar_build_rotation with each variant), the GPU
prefill and the GPU decode, each against the same-design BF16 kernel's output
on the same context.  The three rel-L2 numbers must match the oracle's
fidelity report (fp64, its own calibration) within a stated slack:

  |fid_gpu - fid_oracle| <= 0.01 * (1 + fid_oracle) + 0.002

By the triangle inequality the difference is at most the two kernels' own
errors against the oracle, each within the parity tolerance's rel-L2 of 5e-3
of its output (1e-2 * (1 + fid) covers the INT2 output's norm, which is up to
(1 + fid) times the reference's), plus the effect of the groups whose codes
straddle a decision between the kernel's fp32 rotation and exact x R (0.2% of
groups, one code step each: the 0.002).  The numbers are a report, not a
target: the pages print none for synthetic inputs.
"""
import numpy as np
import pytest

import gpu_harness as H
from int2_rotated_kv_gb300 import pages, synth
from oracle import attention, cache as ocache

pytestmark = pytest.mark.gpu

VARIANTS = (("oscar", 0), ("hadamard_only", 1), ("unrotated", 2))


def _library_rotations(L, inst, variant):
    rk, rv, ck, cv = [], [], [], []
    for h in range(inst.workload.num_kv_heads):
        cq = L.oscar_query_covariance(inst.calib_q[h]) if variant == 0 else None
        cs = L.oscar_score_covariance(inst.calib_q[h], inst.calib_k[h], inst.calib_v[h], 0) \
            if variant == 0 else None
        _, r_k, c_k, _ = L.oscar_build_rotation(cq, inst.calib_k[h], 99.9, variant)
        _, r_v, c_v, _ = L.oscar_build_rotation(cs, inst.calib_v[h], 99.9, variant)
        rk.append(r_k); rv.append(r_v); ck.append(c_k); cv.append(c_v)
    return ocache.Rotations(rk, rv, ck, cv)


def _bf16_output(inst):
    """Decode through the same-design BF16 kernel over an all-BF16 cache."""
    t = H.torch()
    L = H.lib()
    w = inst.workload
    lens = np.asarray(inst.seq_lens)
    Lmax = int(lens.max())
    pp = pages.plan(lens, 0, Lmax + 1)      # every token in the recent window: BF16
    eye = np.stack([np.eye(w.head_dim, dtype=np.float32)] * w.num_kv_heads)
    one = np.ones(w.num_kv_heads, np.float32)
    c = pages.allocate(pp, hkv=w.num_kv_heads, hq=w.num_q_heads, d=w.head_dim, sink=0,
                       window=Lmax + 1, device=H.DEV, r_k=eye, r_v=eye, clip_k=one, clip_v=one)
    k, v, sid, pos = synth.dense_tokens(inst)
    L.oscar_prefill_quantize(c, H.bf16_tensor(k), H.bf16_tensor(v), t.from_numpy(sid).to(H.DEV),
                             t.from_numpy(pos).to(H.DEV),
                             t.from_numpy(lens.astype(np.int32)).to(H.DEV))
    return H.decode(c, inst.q, lens, bf16_only=True)


def test_fidelity_report_through_the_product_path():
    L = H.lib()
    w = synth.QWEN3_8B_32K
    inst = synth.draw_instance(w, n_calib=2048, seq_lens=[4096, 3001])
    ref_bf16 = _bf16_output(inst)
    oracle_rot = {name: H.oracle_rotations(inst, variant=v) for name, v in VARIANTS}
    rep = attention.fidelity_report(inst, sink=4, window=128, rotations=oracle_rot)
    got = {}
    for name, var in VARIANTS:
        rot = _library_rotations(L, inst, var)
        cache, pp = H.make_cache(inst, rot, window=128)
        H.prefill(cache, inst)
        out = H.decode(cache, inst.q, inst.seq_lens)
        got[name] = attention.rel_l2(out, ref_bf16)
        assert H.status(cache) == 0
    H.report("fidelity[qwen3_8b, 4096 + 3001 tokens, 2048 calibration]",
             gpu=got, oracle={k: v["out_rel_l2"] for k, v in rep.items()},
             oracle_kv={k: (v["k_rel_l2"], v["v_rel_l2"]) for k, v in rep.items()})
    for name, _ in VARIANTS:
        f = rep[name]["out_rel_l2"]
        assert abs(got[name] - f) <= 0.01 * (1 + f) + 0.002, (name, got[name], f)
