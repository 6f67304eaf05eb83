#!/usr/bin/env python
"""Benchmark of the OSCAR INT2 mixed-cache decode path on one GB300 (or N
independent replicas, one per GPU).

Headline (default workload ``qwen3_8b_32k_b1``): Qwen3-8B-shaped attention layer,
batch 1, context 32768 = 4 BF16 sink + 32636 INT2 + 128 BF16 recent, 32 query /
8 KV heads, head_dim 128.  One step = one decode step of one layer through the
C ABI: oscar_quantize_append (the new token enters the BF16 window, the token
leaving it is rotated/clipped/quantised into its INT2 page) followed by
oscar_decode_attention (q R_K, split-K attention over INT2 + BF16 pages, LSE
combine, o R_V^T).  Steps rotate over enough layer caches to exceed 3x the L2
size, so every step reads its cache from HBM.  Inputs are synthetic (seeded
generator); rotations come from the library's own calibration calls.

metric = algorithmic bytes per step (INT2 codes + fp16 scale/zero + BF16 sink
and window + q/out + append traffic) / step time, in GB/s.  Extra keys report
the same-design BF16 kernel at the same batch, the roofline of the decode call,
the fp64 oracle on the host (cpu_baseline) and an end-to-end number through the
C ABI with host buffers.  ``--impl reference`` times the oracle alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from int2_rotated_kv_gb300 import pages, synth  # noqa: E402

METRIC = "INT2 paged decode attn: HBM GB/s (% of ~8 TB/s), tokens/s vs own BF16 kernel"
UNIT = "GB/s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_split_qwen3_8b_32k.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="oscar", choices=["oscar", "reference"])
    ap.add_argument("--workload", default=synth.QWEN3_8B_32K.name, choices=list(synth.WORKLOADS))
    ap.add_argument("--extras", action="store_true",
                    help="also time the F1-F4 legs (several query rows, rotary step, calibration, INT4)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other target workloads (128k, batch-64 prefix, 40 GB budget)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-calib", type=int, default=None)
    ap.add_argument("--profile", action="store_true",
                    help="minimal run for ncu: one layer cache, eager steps, no extra legs")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --profile: this many sequences of the workload's context, drawn on the device")
    ap.add_argument("--code-bits", type=int, default=2, choices=[2, 4],
                    help="with --profile: the INT4 variant's caches (the headline is INT2)")
    ap.add_argument("--leg", default=None, choices=sorted(EXTRA_LEGS),
                    help="run one extra leg alone and print its JSON (for profiling)")
    return ap.parse_args()


# --------------------------------------------------------------------------- util

def max_over_ranks(ms, world, device):
    """The slowest rank's time: the job is done when every replica is."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbps(step_bytes_per_rank, ms_all, world):
    """Whole-job throughput: every rank's bytes over the slowest rank's time."""
    return world * step_bytes_per_rank / (ms_all * 1e-3) / 1e9


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def gpu_id(index):
    """The nvidia-smi identifier of torch device `index`: its UUID, so that a
    remapped CUDA_VISIBLE_DEVICES still names the GPU this process runs on (the
    torch index and the nvidia-smi index differ under remapping)."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(index).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    return str(index)


class Clocks:
    """nvidia-smi sampler running while the timed region runs; `gpu` is an
    nvidia-smi device identifier (UUID preferred, see gpu_id)."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        self.proc.wait()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[6:10]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max((num(r[4]) or 0.0) for r in rows),
                "gpu": self.gpu}


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("decode.cu", "layout.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "int2_rotated_kv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------- byte accounting

def token_bytes(d, bits=2):
    """(code token-head bytes: K+V codes + fp16 s/z; BF16 token-head bytes).
    INT2: 3d/4; the INT4 variant: 5d/4."""
    return (bits + 1) * d // 4, 4 * d


def attention_bytes(lens, hkv, hq, d, sink, window, bf16_only=False, bits=2):
    i2, bf = token_bytes(d, bits)
    tot = 0
    for L in lens:
        L = int(L)
        if bf16_only:
            tot += hkv * L * bf
        else:
            n_int2 = max(0, L - window - sink)
            tot += hkv * (n_int2 * i2 + (L - n_int2) * bf)
    tot += 2 * len(lens) * hq * d * 2          # q read, out written (bf16)
    return tot


def append_bytes(lens, hkv, d, sink, window, bf16_only=False, bits=2):
    i2, bf = token_bytes(d, bits)
    tot = 0
    for L in lens:
        tot += hkv * (bf + bf)                  # read new token, write it to its BF16 slot
        if not bf16_only and int(L) - 1 - window >= sink:
            tot += hkv * (bf + i2)              # read the leaving token, write its INT2 form
    return tot


# ----------------------------------------------------------------- setup

def calibrate_with_library(inst, n_calib):
    """R_K, R_V and clips per KV head through the library's host calls."""
    from int2_rotated_kv_gb300 import _lib as L
    rk, rv, ck, cv = [], [], [], []
    for h in range(inst.workload.num_kv_heads):
        q = inst.calib_q[h][:n_calib]
        k = inst.calib_k[h][:n_calib]
        v = inst.calib_v[h][:n_calib]
        cq = L.oscar_query_covariance(q)
        cs = L.oscar_score_covariance(q, k, v, 0)
        _, r_k, c_k, _ = L.oscar_build_rotation(cq, k, 99.9, L.VARIANT_OSCAR)
        _, r_v, c_v, _ = L.oscar_build_rotation(cs, v, 99.9, L.VARIANT_OSCAR)
        rk.append(r_k); rv.append(r_v); ck.append(c_k); cv.append(c_v)
    return np.stack(rk), np.stack(rv), np.array(ck, np.float32), np.array(cv, np.float32)


def bf16_dev(a, dev):
    import torch
    return torch.from_numpy(synth.bf16_bits(np.asarray(a, np.float32)).view(np.int16).copy()).view(
        torch.bfloat16).to(dev)


def device_inputs(inst, dev):
    """A host-drawn Instance in the DeviceInstance layout: prefill lists of
    tokens [0, L_b - 1), the new token L_b - 1 and the decode query."""
    import torch
    H = inst.workload.num_kv_heads
    lens = np.asarray(inst.seq_lens, np.int64)
    ks, vs, sid, pos = [], [], [], []
    for b, L in enumerate(lens):
        n = int(L) - 1
        ks.append(np.stack([inst.k[b][h][:n] for h in range(H)], 1))
        vs.append(np.stack([inst.v[b][h][:n] for h in range(H)], 1))
        sid.append(np.full(n, b, np.int32))
        pos.append(np.arange(n, dtype=np.int32))
    kn = np.stack([[inst.k[b][h][int(lens[b]) - 1] for h in range(H)] for b in range(len(lens))])
    vn = np.stack([[inst.v[b][h][int(lens[b]) - 1] for h in range(H)] for b in range(len(lens))])
    return synth.DeviceInstance(
        inst.workload, inst.params, inst.calib_q, inst.calib_k, inst.calib_v, lens,
        bf16_dev(np.concatenate(ks), dev), bf16_dev(np.concatenate(vs), dev),
        torch.from_numpy(np.concatenate(sid)).to(dev), torch.from_numpy(np.concatenate(pos)).to(dev),
        bf16_dev(kn, dev), bf16_dev(vn, dev), bf16_dev(inst.q, dev))


def clone_cache(c):
    import dataclasses
    return dataclasses.replace(c, int2_pool=c.int2_pool.clone(), bf16_pool=c.bf16_pool.clone())


class Decoder:
    """One set of layer caches plus the per-step calls (INT2 mixed or BF16-only)."""

    def __init__(self, di, rot, dev, *, bf16_only=False, l2_bytes=0, code_bits=2, rope_base=0.0):
        import torch
        from int2_rotated_kv_gb300 import _lib as L
        w = di.workload
        lens_final = di.seq_lens
        self.L, self.torch, self.dev = L, torch, dev
        self.w, self.bf16_only = w, bf16_only
        self.S = w.sink
        self.W = max(int(lens_final.max()) + 1, 1) if bf16_only else w.window
        if bf16_only:
            self.S = 0
        self.lens = np.asarray(lens_final, np.int64)
        B, hkv, hq, d = len(self.lens), w.num_kv_heads, w.num_q_heads, w.head_dim
        # the cache is filled up to L-1; every step re-plays the decode step to L
        pp = pages.plan(self.lens - 1, self.S, self.W, growth=1,
                        shared_prefix_tokens=w.shared_prefix)
        rk, rv, ck, cv = rot
        base = pages.allocate(pp, hkv=hkv, hq=hq, d=d, sink=self.S, window=self.W, device=dev,
                              r_k=rk, r_v=rv, clip_k=ck, clip_v=cv, code_bits=code_bits)
        L.oscar_prefill_quantize(base, di.k_tok, di.v_tok, di.seq_ids, di.positions,
                                 torch.tensor((self.lens - 1).astype(np.int32), device=dev))
        torch.cuda.synchronize()
        self.layer_bytes = (base.int2_pool.numel() + base.bf16_pool.numel() * 2)
        self.step_bytes = attention_bytes(self.lens, hkv, hq, d, self.S, self.W, bf16_only, code_bits)
        self.attn_bytes = self.step_bytes
        self.step_bytes += append_bytes(self.lens, hkv, d, self.S, self.W, bf16_only, code_bits)
        touched = self.attn_bytes
        n_layers = max(2, math.ceil(3 * l2_bytes / max(touched, 1)) + 1) if l2_bytes else 1
        self.caches = [base] + [clone_cache(base) for _ in range(n_layers - 1)]
        self.k_new, self.v_new, self.q = di.k_new, di.v_new, di.q
        self.lens_dev = torch.tensor(self.lens.astype(np.int32), device=dev)
        self.max_len = int(self.lens.max())
        self.out = torch.zeros((B, hq, d), dtype=torch.bfloat16, device=dev)
        ws = L.oscar_decode_workspace_size(base, B, self.max_len)
        self.ws = torch.zeros(ws // 4 + 64, dtype=torch.float32, device=dev)
        self.n_layers = n_layers
        self.rope_base = rope_base     # > 0: the fused step with rotary embedding
        self.launches_per_step = 3     # INT2: append+q', split, combine; BF16: append, split, combine

    def append(self, i, k=None, v=None, lens=None):
        c = self.caches[i % self.n_layers]
        self.L.oscar_quantize_append(c, self.k_new if k is None else k, self.v_new if v is None else v,
                                     self.lens_dev if lens is None else lens)

    def attend(self, i, q=None, lens=None, out=None):
        c = self.caches[i % self.n_layers]
        fn = self.L.oscar_decode_attention_bf16 if self.bf16_only else self.L.oscar_decode_attention
        fn(c, self.q if q is None else q, self.lens_dev if lens is None else lens, self.max_len,
           self.out if out is None else out, self.ws)

    def step(self, i, q=None, k=None, v=None, out=None):
        if self.bf16_only:
            self.append(i, k, v)
            self.attend(i, q, out=out)
        elif self.rope_base > 0:   # the fused step with rotary embedding of q and the new key
            c = self.caches[i % self.n_layers]
            self.L.oscar_decode_step_rope(c, self.q if q is None else q, self.k_new if k is None else k,
                                          self.v_new if v is None else v, self.lens_dev, self.max_len,
                                          self.rope_base, self.out if out is None else out, self.ws)
        else:   # the library's fused step: append + attention in one call
            c = self.caches[i % self.n_layers]
            self.L.oscar_decode_step(c, self.q if q is None else q, self.k_new if k is None else k,
                                     self.v_new if v is None else v, self.lens_dev, self.max_len,
                                     self.out if out is None else out, self.ws)

    def graph(self, first, count):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for i in range(first, first + count):     # populate allocator / attributes
                self.step(i)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for i in range(first, first + count):
                self.step(i)
        return g


def time_steps(dec, steps, warmup, chunk=64, clocks=None, barrier=None):
    """Time exactly `steps` decode steps (graph replays), after `warmup` steps."""
    torch = dec.torch
    chunk = max(dec.n_layers, (chunk // dec.n_layers) * dec.n_layers)
    g_full = dec.graph(0, chunk)
    rem = steps % chunk
    g_rem = dec.graph(0, rem) if rem else None
    for i in range(warmup):
        dec.step(i)
    # the first replay of a graph uploads it to the device: done here, untimed
    g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    if clocks:
        clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    # a spin kernel ahead of the start event keeps the stream busy while the
    # host submits the graphs, so their launch latency is not device time
    torch.cuda._sleep(2_000_000)
    e0.record()
    for _ in range(steps // chunk):
        g_full.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    if barrier:
        barrier()
    return e0.elapsed_time(e1) / steps, clk


def time_graph(dec, fn, steps, warmup, chunk=64):
    """Device time of fn(i) (one call per layer index), replayed from CUDA graphs."""
    torch = dec.torch
    chunk = max(dec.n_layers, (chunk // dec.n_layers) * dec.n_layers)
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(0)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for i in range(chunk):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // chunk)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(2_000_000)   # the stream stays busy while the replays are submitted
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (reps * chunk)


def time_decode_calls(dec, iters=200, batch=40):
    """Average duration of one oscar_decode_attention call (its three kernels),
    bracketed by CUDA events on the launching stream, cold L2 (rotating layers).
    A spin kernel keeps the stream busy while a batch of calls is queued, so the
    host's launch cost never shows up between the events."""
    torch = dec.torch
    for i in range(10):
        dec.attend(i)
    torch.cuda.synchronize()
    ts = []
    done = 0
    while done < iters:
        n = min(batch, iters - done)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        torch.cuda._sleep(20_000_000)
        for k, (a, b) in enumerate(evs):
            a.record()
            dec.attend(done + k)
            b.record()
        torch.cuda.synchronize()
        ts += [a.elapsed_time(b) for a, b in evs]
        done += n
    return statistics.median(ts), statistics.mean(ts)


def time_e2e(dec, steps, warmup):
    """Through the C ABI with host buffers (oscar_decode_step_host): every step
    the library copies q and the new K/V in from one pinned host buffer, runs
    the fused step, and copies the output back to pinned host memory."""
    torch, L = dec.torch, dec.L
    assert not dec.bf16_only
    hin = torch.cat([dec.q.reshape(-1), dec.k_new.reshape(-1),
                     dec.v_new.reshape(-1)]).cpu().pin_memory()
    ho = torch.empty(dec.out.shape, dtype=torch.bfloat16).pin_memory()
    B = int(dec.lens_dev.numel())
    staging = torch.empty(L.oscar_decode_step_host_staging_size(dec.caches[0], B) // 4 + 4,
                          dtype=torch.float32, device=dec.dev)

    def one(i):
        L.oscar_decode_step_host(dec.caches[i % dec.n_layers], hin, dec.lens_dev, dec.max_len, ho,
                                 staging, dec.ws, rope_base=dec.rope_base)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        one(i)
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, hin.numel() * 2, ho.numel() * 2


def fidelity_leg(inst, di, rot_oscar, dev, n_calib):
    """Attention-output error of the INT2 cache against the same-design BF16
    kernel on the same context, for OSCAR, Hadamard-only and unrotated INT2
    (the comparison the pages draw): rotations from the library's calibration
    calls, one fused decode step each, rel-L2 of the outputs.  A report, not a
    target."""
    torch = __import__("torch")
    from int2_rotated_kv_gb300 import _lib as L
    rots = {"oscar": rot_oscar}
    for name, var in (("hadamard_only", L.VARIANT_HADAMARD), ("unrotated", L.VARIANT_IDENTITY)):
        rk, rv, ck, cv = [], [], [], []
        for h in range(inst.workload.num_kv_heads):
            _, r_k, c_k, _ = L.oscar_build_rotation(None, inst.calib_k[h][:n_calib], 99.9, var)
            _, r_v, c_v, _ = L.oscar_build_rotation(None, inst.calib_v[h][:n_calib], 99.9, var)
            rk.append(r_k); rv.append(r_v); ck.append(c_k); cv.append(c_v)
        rots[name] = (np.stack(rk), np.stack(rv), np.array(ck, np.float32), np.array(cv, np.float32))

    def out_of(dec):
        dec.step(0)
        torch.cuda.synchronize()
        return dec.out.float().cpu().numpy().astype(np.float64)
    ref = out_of(Decoder(di, rot_oscar, dev, bf16_only=True))
    res = {"workload": inst.workload.name, "context": int(inst.seq_lens.max()),
           "metric": "rel-L2 of the decode output against the same-design BF16 kernel's",
           "n_calib": n_calib}
    for name, rot in rots.items():
        o = out_of(Decoder(di, rot, dev))
        res[name] = round(float(np.linalg.norm(o - ref) / max(np.linalg.norm(ref), 1e-300)), 5)
    torch.cuda.empty_cache()
    return res


# -------------------------------------------------------------- CPU / oracle

def oracle_sample(inst, rot, n_heads=1, max_tokens=None):
    """The oracle's decode for the first `n_heads` KV heads of sequence 0 (its
    INT2 tokens rebuilt and attended in fp64).  Returns (bytes, seconds)."""
    from oracle import attention, cache as ocache
    w = inst.workload
    rk, rv, ck, cv = rot
    L = int(inst.seq_lens[0]) if max_tokens is None else min(int(inst.seq_lens[0]), max_tokens)
    G = w.gqa
    t0 = time.perf_counter()
    for h in range(n_heads):
        r = ocache.Rotations([rk[h]], [rv[h]], [ck[h]], [cv[h]])
        attention.mixed_decode(inst.q[:1, h * G:(h + 1) * G], [[inst.k[0][h][:L]]],
                               [[inst.v[0][h][:L]]], [L], r, sink=w.sink, window=w.window, gqa=G)
    dt = time.perf_counter() - t0
    nb = attention_bytes([L], n_heads, n_heads * G, w.head_dim, w.sink, w.window)
    return nb, dt


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = max((i.get("num_threads", 1) for i in info), default=os.cpu_count())
        return int(n)
    except Exception:
        return os.cpu_count()


def cpu_baseline(inst, rot, budget_s=12.0, max_passes=400):
    """The oracle on the host cores: whole passes over every KV head of the
    step (sequence 0, full context), repeated until ~budget_s of CPU work."""
    hkv = inst.workload.num_kv_heads
    tot_b = tot_t = 0.0
    passes = 0
    while tot_t < budget_s and passes < max_passes:
        b2, t2 = oracle_sample(inst, rot, hkv)
        tot_b += b2
        tot_t += t2
        passes += 1
    return {"value": round(tot_b / tot_t / 1e9, 4), "unit": UNIT, "cores": blas_threads(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle decode, {passes} pass(es) over all {hkv} KV heads "
                      f"(G={inst.workload.gqa} query heads, full {int(inst.seq_lens[0])}-token "
                      f"context of sequence 0); {tot_t:.1f} s of CPU work"}


def cpu_one_thread_sample(workload_name, budget_s=6.0):
    """The oracle's decode pass timed in a child process whose BLAS / OpenMP pools
    are limited to one thread (they are fixed when numpy loads, so a fresh
    process is needed).  No GPU is touched there."""
    code = (
        "import json, sys, time, numpy as np\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import bench\n"
        "from int2_rotated_kv_gb300 import synth\n"
        "from oracle import attention\n"
        f"w = synth.WORKLOADS[{workload_name!r}]\n"
        "inst = synth.draw_instance(w, n_calib=512)\n"
        "r = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)\n"
        "rot = (np.stack(r.rk), np.stack(r.rv), np.array(r.ck), np.array(r.cv))\n"
        "tb = tt = 0.0\n"
        "heads = 0\n"
        f"while tt < {budget_s} and heads < 64:\n"
        "    b, t = bench.oracle_sample(inst, rot, 1)\n"
        "    tb += b; tt += t; heads += 1\n"
        "print(json.dumps({'value': tb / tt / 1e9, 'heads': heads, 'seconds': tt}))\n")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                           timeout=600)
        res = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": round(res["value"], 4), "unit": UNIT, "cores": 1,
                "sample": f"{res['heads']} single-KV-head pass(es), {res['seconds']:.1f} s"}
    except Exception as e:
        return {"error": str(e)[:200]}


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    inst = synth.draw_instance(w, n_calib=min(w.n_calib, 1024))
    from oracle import attention
    rot_o = attention.calibrate(inst.calib_q, inst.calib_k, inst.calib_v, 0)
    rot = (np.stack(rot_o.rk), np.stack(rot_o.rv), np.array(rot_o.ck), np.array(rot_o.cv))
    # size the per-step sample so the whole run stays within ~2 minutes
    nb, dt = oracle_sample(inst, rot, 1, max_tokens=2048)
    per_tok = dt / 2048
    budget = 100.0 / max(1, args.steps + args.warmup)
    ntok = int(min(int(inst.seq_lens[0]), max(w.window + w.sink + 16, budget / per_tok)))
    for _ in range(args.warmup):
        oracle_sample(inst, rot, 1, max_tokens=ntok)
    tb = tt = 0.0
    for _ in range(args.steps):
        b, t = oracle_sample(inst, rot, 1, max_tokens=ntok)
        tb += b
        tt += t
    v = tb / tt / 1e9
    sample = (f"fp64 numpy oracle, 1 KV head (G={w.gqa}) of sequence 0, first {ntok} tokens "
              f"of the context per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "sample_tokens": ntok},
        "cpu_baseline": {"value": round(v, 5), "unit": UNIT, "kind": "oracle",
                         "cores": blas_threads(), "sample": sample},
        "e2e": {"value": round(v, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------- extras

def decode_leg(di, rot, dev, l2, steps=200, warmup=10, bf16_only=False, code_bits=2, rope_base=0.0):
    """One layer's decode step (append + attention) at di's shape: µs, GB/s,
    and the decode call alone."""
    torch = __import__("torch")
    dec = Decoder(di, rot, dev, bf16_only=bf16_only, l2_bytes=l2, code_bits=code_bits,
                  rope_base=rope_base)
    t, clk = time_steps(dec, steps, warmup, clocks=Clocks(gpu_id(torch.cuda.current_device())))
    med, mean = time_decode_calls(dec, 100)
    peak, peak_kind = peaks()
    call_gbps = dec.attn_bytes / med / 1e6
    step_gbps = dec.step_bytes / t / 1e6
    res = {"batch": len(di.seq_lens), "us_per_layer_step": round(t * 1e3, 3),
           "GBps": round(step_gbps, 1), "decode_call_us": round(med * 1e3, 3),
           "decode_call_GBps": round(call_gbps, 1),
           "roofline": {"bound": "hbm", "achieved": round(call_gbps, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(call_gbps / peak, 4), "step_frac": round(step_gbps / peak, 4),
                        "kernel": "decode call (algorithmic bytes / median CUDA-event time)",
                        "peak_kind": f"{peak_kind} hbm_gbs", "traffic": None},
           "algorithmic_bytes_per_step": int(dec.step_bytes), "layers_rotated": dec.n_layers,
           "cache_bytes_per_layer": int(dec.layer_bytes), "clocks": clk}
    del dec
    torch.cuda.empty_cache()
    return res


def extra_long(dev, l2, n_calib):
    """Qwen3-32B shape, one 131072-token sequence: INT2 and BF16 at batch 1."""
    w = synth.QWEN3_32B_128K
    di = synth.draw_device(w, w.seq_lens(), dev, n_calib=n_calib)
    rot = calibrate_with_library(di, n_calib)
    res = decode_leg(di, rot, dev, l2)
    bf = decode_leg(di, rot, dev, l2, bf16_only=True)
    res["bf16"] = bf
    res["speedup_vs_bf16"] = round(bf["us_per_layer_step"] / res["us_per_layer_step"], 3)
    return res


def extra_prefix(dev, l2, n_calib):
    """Qwen3-4B shape, 64 sequences of U{4096..8192} tokens sharing a 2048-token
    prefix (128 pages per sequence with equal page ids).  GB/s on unique bytes:
    the shared pages count once."""
    w = synth.QWEN3_4B_PREFIX
    lens = w.seq_lens()
    di = synth.draw_device(w, lens, dev, n_calib=n_calib)
    rot = calibrate_with_library(di, n_calib)
    res = decode_leg(di, rot, dev, l2)
    i2, bfb = token_bytes(w.head_dim)
    P, B, H = w.shared_prefix, len(lens), w.num_kv_heads
    shared_int2 = H * (w.sink * bfb + (P - w.sink) * i2)
    shared_bf16 = H * P * bfb
    res["unique_GBps"] = round((res["algorithmic_bytes_per_step"] - (B - 1) * shared_int2) /
                               res["us_per_layer_step"] / 1e3, 1)
    bf = decode_leg(di, rot, dev, l2, bf16_only=True)
    bf["unique_GBps"] = round((bf["algorithmic_bytes_per_step"] - (B - 1) * shared_bf16) /
                              bf["us_per_layer_step"] / 1e3, 1)
    res["bf16"] = bf
    res["speedup_vs_bf16"] = round(bf["us_per_layer_step"] / res["us_per_layer_step"], 3)
    res["seq_lens"] = {"min": int(lens.min()), "max": int(lens.max()), "sum": int(lens.sum())}
    return res


def extra_multiquery(dev, l2, n_calib, rows=16):
    """Several query rows per sequence (a chunk of new tokens at the end of a
    32768-token Qwen3-8B cache) through oscar_multiquery_attention."""
    torch = __import__("torch")
    from int2_rotated_kv_gb300 import _lib as L
    w = synth.QWEN3_8B_32K
    di = synth.draw_device(w, w.seq_lens(), dev, n_calib=n_calib)
    rot = calibrate_with_library(di, n_calib)
    dec = Decoder(di, rot, dev, l2_bytes=l2)
    Lc = int(dec.lens[0])
    pos = torch.arange(Lc - rows, Lc, dtype=torch.int32, device=dev)[None]
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    q = torch.randn((1, rows, w.num_q_heads, w.head_dim), generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty_like(q)
    ws = torch.zeros(L.oscar_multiquery_workspace_size(dec.caches[0], 1, rows, Lc) // 4 + 64,
                     dtype=torch.float32, device=dev)
    # the caches hold L-1 tokens until a step runs; one step fills the last slot
    for i in range(dec.n_layers):
        dec.step(i)
    torch.cuda.synchronize()

    def call(i):
        L.oscar_multiquery_attention(dec.caches[i % dec.n_layers], q, dec.lens_dev, pos, Lc, out, ws)
    t = time_graph(dec, call, 200, 10)
    unique = attention_bytes(dec.lens, w.num_kv_heads, w.num_q_heads, w.head_dim, w.sink, w.window)
    res = {"rows": rows, "us_per_call": round(t * 1e3, 3), "rows_per_s": round(rows / (t * 1e-3), 1),
           "unique_GBps": round(unique / t / 1e6, 1),
           "page_reads_GBps": round(rows / (8 // w.gqa) * unique / t / 1e6, 1),
           "note": f"{8 // w.gqa} rows of the sequence share each CTA's page reads"}
    del dec
    torch.cuda.empty_cache()
    return res


def calib_attention_flops(n, hq, d):
    """Useful FLOPs of causal calibration attention: query t meets t + 1 keys,
    2d FLOPs for its logit and 2d for its share of P V."""
    return 4.0 * d * hq * n * (n + 1) / 2


def extra_calibration(dev, l2, n_calib=8192):
    """Device calibration of one Qwen3-8B layer (32/8 heads, d = 128, 8192
    calibration tokens): C_Q, C_S, then the clips of K and V under the R the
    host builds from them."""
    torch = __import__("torch")
    from int2_rotated_kv_gb300 import _lib as L
    w = synth.QWEN3_8B_32K
    inst = synth.draw_instance(w, n_calib=n_calib, seq_lens=[1])
    hkv, hq, d, G = w.num_kv_heads, w.num_q_heads, w.head_dim, w.gqa
    q = np.zeros((n_calib, hq, d), np.float32)
    for h in range(hkv):
        q[:, h * G:(h + 1) * G] = inst.calib_q[h]
    qd = bf16_dev(q, dev)
    kd = bf16_dev(np.stack(inst.calib_k, axis=1), dev)
    vd = bf16_dev(np.stack(inst.calib_v, axis=1), dev)
    ws = torch.empty(L.oscar_calibration_workspace_size(hkv, hq, d, n_calib) // 4 + 64,
                     dtype=torch.float32, device=dev)
    cq = torch.empty((hkv, d, d), dtype=torch.float64, device=dev)
    cs = torch.empty_like(cq)
    ck = torch.empty(hkv, dtype=torch.float32, device=dev)
    cv = torch.empty_like(ck)

    def timed(fn, reps=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    t_q = timed(lambda: L.oscar_query_covariance_device(qd, hkv, cq, ws))
    t_s = timed(lambda: L.oscar_score_covariance_device(qd, kd, vd, cs, ws))
    t0 = time.perf_counter()
    cq_h, cs_h = cq.cpu().numpy(), cs.cpu().numpy()
    rk = np.stack([L.oscar_build_rotation(cq_h[h], inst.calib_k[h][:1], 99.9)[1] for h in range(hkv)])
    rv = np.stack([L.oscar_build_rotation(cs_h[h], inst.calib_v[h][:1], 99.9)[1] for h in range(hkv)])
    t_eig = time.perf_counter() - t0
    rkd = torch.from_numpy(rk).to(dev)
    rvd = torch.from_numpy(rv).to(dev)
    t_c = timed(lambda: (L.oscar_clip_threshold_device(kd, rkd, 99.9, ck, ws),
                         L.oscar_clip_threshold_device(vd, rvd, 99.9, cv, ws)))
    fl = calib_attention_flops(n_calib, hq, d)
    q_bytes = n_calib * hq * d * 2
    res = {"n_calib": n_calib, "shape": f"{hq}/{hkv} heads, d={d}",
           "query_covariance_ms": round(t_q, 4),
           "query_covariance_GBps": round(q_bytes / t_q / 1e6, 1),
           "score_covariance_ms": round(t_s, 4),
           "score_attention_useful_TFLOPs": round(fl / t_s / 1e9, 1),
           "clip_k_and_v_ms": round(t_c, 4),
           "host_eigendecomposition_s": round(t_eig, 3),
           "device_total_ms": round(t_q + t_s + t_c, 3)}
    del ws, qd, kd, vd
    torch.cuda.empty_cache()
    return res


def pool_bytes_per_seq(w, L, bf16_only, code_bits=2):
    """Allocated page-slot bytes of one sequence of L tokens in one layer (the
    same page plan the decoder allocates: cache filled to L - 1 plus one page of growth)."""
    S, W = (0, L + 1) if bf16_only else (w.sink, w.window)
    pp = pages.plan(np.array([L - 1]), S, W, growth=1)
    d, H = w.head_dim, w.num_kv_heads
    return (pp.num_int2_pages * pages.int2_bytes_per_page(H, d, code_bits)
            + pp.num_bf16_pages * pages.bf16_bytes_per_page(H, d))


def extra_rope(dev, l2, n_calib):
    """The fused step with rotary position embedding (base 1e6, Qwen3) against
    the same step without it, Qwen3-8B shape at 32768 tokens, batch 1."""
    w = synth.QWEN3_8B_32K
    di = synth.draw_device(w, w.seq_lens(), dev, n_calib=n_calib)
    rot = calibrate_with_library(di, n_calib)
    r = decode_leg(di, rot, dev, l2, rope_base=1.0e6)
    r0 = decode_leg(di, rot, dev, l2)
    r.pop("clocks", None)
    r["without_rope_us_per_layer_step"] = r0["us_per_layer_step"]
    return r


def extra_int4(dev, l2, n_calib, budget=40e9):
    """The INT4 variant (16 levels, two 2-bit planes) beside INT2: the Qwen3-8B
    32k and Qwen3-32B 128k steps at batch 1, and the batch and tokens/s that fit
    the 40e9-byte budget at L = 4096 (36 layers, one timed)."""
    torch = __import__("torch")
    res = {}
    for w in (synth.QWEN3_8B_32K, synth.QWEN3_32B_128K):
        di = synth.draw_device(w, w.seq_lens(), dev, n_calib=n_calib)
        rot = calibrate_with_library(di, n_calib)
        r4 = decode_leg(di, rot, dev, l2, code_bits=4)
        r2 = decode_leg(di, rot, dev, l2)
        r4.pop("clocks", None)
        r4["int2_us_per_layer_step"] = r2["us_per_layer_step"]
        r4["int4_over_int2_time"] = round(r4["us_per_layer_step"] / r2["us_per_layer_step"], 3)
        res[w.name] = r4
        del di
        torch.cuda.empty_cache()
    w = synth.QWEN3_8B_BUDGET
    Lc, layers = int(w.context), w.layers
    per_i4 = pool_bytes_per_seq(w, Lc, False, 4) * layers
    b_i4 = int(budget // per_i4)
    di = synth.draw_device(w, np.full(b_i4, Lc), dev, n_calib=n_calib)
    rot = calibrate_with_library(di, n_calib)
    r = decode_leg(di, rot, dev, l2, steps=100, warmup=5, code_bits=4)
    r.pop("clocks", None)
    r["tokens_per_s"] = round(b_i4 / (layers * r["us_per_layer_step"] * 1e-6), 1)
    res["budget40GB_L4096"] = {"int4_bytes_per_seq": per_i4, "int4_batch": b_i4, "int4": r}
    del di
    torch.cuda.empty_cache()
    return res


def extra_budget(dev, l2, n_calib, budget=40e9):
    """Qwen3-8B shape at L = 4096 under a 40e9-byte cache budget over 36 layers:
    the INT2 and BF16 batches that fit, one layer timed (tokens/s = batch /
    (36 t_layer), attention only); INT2 also at the BF16 batch; the append at
    batch 256 alone; the bulk prefill of 256 x 4096 tokens."""
    torch = __import__("torch")
    from int2_rotated_kv_gb300 import _lib as L
    w = synth.QWEN3_8B_BUDGET
    Lc, layers = int(w.context), w.layers
    per_i2 = pool_bytes_per_seq(w, Lc, False) * layers
    per_bf = pool_bytes_per_seq(w, Lc, True) * layers
    b_i2, b_bf = int(budget // per_i2), int(budget // per_bf)
    res = {"budget_bytes": budget, "layers": layers, "int2_bytes_per_seq": per_i2,
           "bf16_bytes_per_seq": per_bf, "int2_batch": b_i2, "bf16_batch": b_bf}
    di = synth.draw_device(w, np.full(b_i2, Lc), dev, n_calib=n_calib)
    rot = calibrate_with_library(di, n_calib)
    r = decode_leg(di, rot, dev, l2, steps=100, warmup=5)
    r["tokens_per_s"] = round(b_i2 / (layers * r["us_per_layer_step"] * 1e-6), 1)
    res["int2_at_budget"] = r
    del di
    di = synth.draw_device(w, np.full(b_bf, Lc), dev, n_calib=n_calib)
    r = decode_leg(di, rot, dev, l2, steps=100, warmup=5, bf16_only=True)
    r["tokens_per_s"] = round(b_bf / (layers * r["us_per_layer_step"] * 1e-6), 1)
    res["bf16_at_budget"] = r
    r = decode_leg(di, rot, dev, l2, steps=100, warmup=5)
    r["tokens_per_s"] = round(b_bf / (layers * r["us_per_layer_step"] * 1e-6), 1)
    res["int2_at_bf16_batch"] = r
    res["tokens_per_s_ratio_at_equal_memory"] = round(
        res["int2_at_budget"]["tokens_per_s"] / res["bf16_at_budget"]["tokens_per_s"], 3)
    del di
    torch.cuda.empty_cache()
    # append alone at batch 256 (graph-replayed, rotating layer caches)
    di = synth.draw_device(w, np.full(256, Lc), dev, n_calib=n_calib)
    dec = Decoder(di, rot, dev, l2_bytes=l2)
    t = time_graph(dec, dec.append, 400, 10)
    nb = append_bytes(dec.lens, w.num_kv_heads, w.head_dim, w.sink, w.window)
    peak, peak_kind = peaks()
    res["append_b256"] = {"us": round(t * 1e3, 3), "GBps": round(nb / t / 1e6, 1),
                          "algorithmic_bytes": int(nb),
                          "roofline": {"bound": "latency", "achieved": round(nb / t / 1e6, 1),
                                       "peak": peak, "unit": "GB/s",
                                       "frac": round(nb / t / 1e6 / peak, 4),
                                       "peak_kind": f"{peak_kind} hbm_gbs", "traffic": None,
                                       "note": "3.3 MB per call: a chain of dependent loads, not bandwidth"}}
    del dec, di
    torch.cuda.empty_cache()
    # bulk prefill: 256 sequences x 4096 tokens placed in one call
    di = synth.draw_device(w, np.full(256, Lc + 1), dev, n_calib=n_calib)
    lens_f = np.full(256, Lc)
    pp = pages.plan(lens_f, w.sink, w.window, growth=0)
    c = pages.allocate(pp, hkv=w.num_kv_heads, hq=w.num_q_heads, d=w.head_dim, sink=w.sink,
                       window=w.window, device=dev, r_k=rot[0], r_v=rot[1], clip_k=rot[2],
                       clip_v=rot[3])
    lt = torch.tensor(lens_f.astype(np.int32), device=dev)

    def pf():
        L.oscar_prefill_quantize(c, di.k_tok, di.v_tok, di.seq_ids, di.positions, lt)
    for _ in range(2):
        pf()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    e0.record()
    for _ in range(reps):
        pf()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / reps
    T = int(di.k_tok.shape[0])
    i2b, bfb = token_bytes(w.head_dim)
    n_i2 = 256 * max(0, Lc - w.window - w.sink)
    rd = 2 * T * w.num_kv_heads * w.head_dim * 2
    wr = w.num_kv_heads * (n_i2 * i2b + (T - n_i2) * bfb)
    flops = 2 * 2 * n_i2 * w.num_kv_heads * w.head_dim * w.head_dim
    res["prefill_256x4096"] = {"ms": round(t, 3), "tokens": T, "read_bytes": rd, "write_bytes": wr,
                               "GBps": round((rd + wr) / t / 1e6, 1),
                               "rotation_TFLOPs": round(flops / t / 1e9, 2),
                               "roofline": {"bound": "hbm", "achieved": round((rd + wr) / t / 1e6, 1),
                                            "peak": peak, "unit": "GB/s",
                                            "frac": round((rd + wr) / t / 1e6 / peak, 4),
                                            "peak_kind": f"{peak_kind} hbm_gbs", "traffic": None}}
    del c, di
    torch.cuda.empty_cache()
    return res


# Extra legs: name -> fn(device, l2_bytes, calibration tokens for the rotations).
# The calibration leg times calibration itself, on the 8192 tokens of the 8B workload.
# The other target workloads, measured in every default run beside the headline.
CONFIG_LEGS = (synth.QWEN3_32B_128K.name, synth.QWEN3_4B_PREFIX.name, synth.QWEN3_8B_BUDGET.name)

EXTRA_LEGS = {
    synth.QWEN3_32B_128K.name: extra_long,
    synth.QWEN3_4B_PREFIX.name: extra_prefix,
    synth.QWEN3_8B_BUDGET.name: extra_budget,
    "qwen3_8b_32k_chunk16": extra_multiquery,
    "qwen3_8b_calibration_8192": lambda dev, l2, _n: extra_calibration(dev, l2, 8192),
    "int4_variant": extra_int4,
    "qwen3_8b_32k_rope": extra_rope,
}


# --------------------------------------------------------------------- main

def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))

        def barrier():
            dist.barrier()
    from int2_rotated_kv_gb300 import _lib as L
    L.lib()
    if args.leg:
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        print(json.dumps({"leg": args.leg, **EXTRA_LEGS[args.leg](dev, l2, 2048)}), flush=True)
        return
    w = synth.WORKLOADS[args.workload]
    n_calib = args.n_calib or w.n_calib
    t0 = time.time()
    inst = synth.draw_instance(w, n_calib=n_calib)
    t_gen = time.time() - t0
    t0 = time.time()
    rot = calibrate_with_library(inst, n_calib)
    t_cal = time.time() - t0
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    if args.profile:
        # launches in order: 1 prefill, then per step the fused append (+ q'), split, combine
        if args.batch:   # a large batch: inputs drawn on the device, the same recipe
            di = synth.draw_device(w, np.full(args.batch, int(w.seq_lens().max())), dev, n_calib=n_calib)
        else:
            di = device_inputs(inst, dev)
        dec = Decoder(di, rot, dev, l2_bytes=0, code_bits=args.code_bits)
        for i in range(args.warmup + args.steps):
            dec.step(i)
        torch.cuda.synchronize()
        print(json.dumps({"profile": w.name, "code_bits": args.code_bits, "steps": args.steps,
                          "warmup": args.warmup,
                          "launches_per_step": dec.launches_per_step,
                          "attention_bytes": int(dec.attn_bytes)}), flush=True)
        return
    di = device_inputs(inst, dev)
    dec = Decoder(di, rot, dev, l2_bytes=l2)
    clocks = Clocks(gpu_id(local))
    ms, clk = time_steps(dec, args.steps, args.warmup, clocks=clocks, barrier=barrier)
    ms_all = max_over_ranks(ms, world, dev)
    value = job_gbps(dec.step_bytes, ms_all, world)
    # roofline of the decode call (qrot + split + combine), cold L2
    med, mean = time_decode_calls(dec, 200)
    peak, peak_kind = peaks()
    achieved = dec.attn_bytes / (mean * 1e-3) / 1e9
    traffic = None
    try:
        with open(PROFILE_TRAFFIC) as f:
            prof = json.load(f)
        if prof.get("source_hash") == kernel_source_hash() and prof.get("workload") == w.name:
            traffic = prof.get("traffic_bytes_per_launch")
    except Exception:
        pass
    # end to end through the C ABI with host buffers
    e2e_ms, h2d, d2h = time_e2e(dec, min(args.steps, 500), max(3, args.warmup))
    e2e_val = job_gbps(dec.step_bytes, max_over_ranks(e2e_ms, world, dev), world)
    # same-design BF16 kernel, same batch
    bf = {}
    try:
        decb = Decoder(di, rot, dev, bf16_only=True, l2_bytes=l2)
        msb, _ = time_steps(decb, min(args.steps, 1000), args.warmup)
        medb, meanb = time_decode_calls(decb, 100)
        bf = {"bf16_ms_per_step": round(msb, 5), "bf16_GBps": round(decb.step_bytes / msb / 1e6, 1),
              "bf16_decode_call_us": round(meanb * 1e3, 3),
              "bf16_decode_call_GBps": round(decb.attn_bytes / meanb / 1e6, 1),
              "speedup_vs_bf16": round(msb / ms, 3),
              "bf16_cache_bytes_per_layer": int(decb.attn_bytes)}
        del decb
        torch.cuda.empty_cache()
    except Exception as e:
        bf = {"bf16_error": str(e)[:200]}
    B = len(inst.seq_lens)
    layers_model = w.layers if w.layers > 1 else 1
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_all, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int2+bf16/f32acc",
        "data": "synthetic (seeded generator; rotations from the library's calibration calls)",
        "config": {"workload": w.name, "batch": B, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "context": int(inst.seq_lens.max()), "sink": w.sink, "window": w.window,
                   "n_calib": n_calib, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: steps rotate over {dec.n_layers} layer caches "
                         f"({dec.n_layers * dec.attn_bytes / 1e6:.0f} MB touched vs L2 {l2 / 1e6:.0f} MB)",
                   "step": "oscar_decode_step (append + attention fused), one layer, CUDA graph"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "oscar_decode_attention call (qrot + split + combine kernels)",
                     "peak_kind": f"{peak_kind} hbm_gbs", "call_us_median": round(med * 1e3, 3),
                     "call_us_mean": round(mean * 1e3, 3),
                     "algorithmic_bytes_per_call": int(dec.attn_bytes)},
        "e2e": {"value": round(e2e_val, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": dec.launches_per_step * args.steps,
        "clocks": clk,
        "us_per_layer_step": round(ms_all * 1e3, 3),
        "decode_tokens_per_s_attention_only": round(world * B / (layers_model * ms_all * 1e-3), 1),
        "tokens_per_s_layers": layers_model,
        "algorithmic_bytes_per_step": int(dec.step_bytes),
        "setup_s": {"generate": round(t_gen, 1), "calibrate": round(t_cal, 1)},
    }
    out.update(bf)
    if rank == 0:
        try:
            out["fidelity"] = fidelity_leg(inst, di, rot, dev, n_calib)
        except Exception as e:
            out["fidelity"] = {"error": f"{type(e).__name__}: {str(e)[:200]}"}
    if rank == 0 and not args.no_configs:
        # every other target workload, each with its roofline and clock record
        del dec
        torch.cuda.empty_cache()
        cf = {}
        for name in CONFIG_LEGS:
            try:
                cf[name] = EXTRA_LEGS[name](dev, l2, 2048)
            except Exception as e:
                cf[name] = {"error": f"{type(e).__name__}: {str(e)[:300]}"}
            torch.cuda.empty_cache()
        out["configs"] = cf
    if args.extras and rank == 0:
        ex = {}
        torch.cuda.empty_cache()
        for name, fn in EXTRA_LEGS.items():
            if name in CONFIG_LEGS:
                continue
            try:
                ex[name] = fn(dev, l2, 2048)
            except Exception as e:
                ex[name] = {"error": f"{type(e).__name__}: {str(e)[:300]}"}
            torch.cuda.empty_cache()
        out["extras"] = ex
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(inst, rot)
        out["cpu_baseline"]["one_thread"] = cpu_one_thread_sample(w.name)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
