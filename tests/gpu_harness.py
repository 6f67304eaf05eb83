"""Helpers for the GPU parity tests: upload synthetic inputs, run the library
through its C ABI, read pools back.  Expected values come from ``oracle`` only."""
import numpy as np

from int2_rotated_kv_gb300 import pages, synth
from oracle import attention, cache as ocache, layout, quant

DEV = "cuda:0"
TOL_MAX_ABS = 1e-2       # attention output vs oracle (fp32 accumulate, bf16 store)
TOL_REL_L2 = 5e-3


def torch():
    import torch as t
    return t


def lib():
    from int2_rotated_kv_gb300 import _lib
    _lib.lib()
    return _lib


def bf16_tensor(a):
    t = torch()
    bits = synth.bf16_bits(np.asarray(a, np.float32))
    return t.from_numpy(bits.view(np.int16).copy()).view(t.bfloat16).to(DEV)


def from_bf16(x):
    t = torch()
    return x.detach().float().cpu().numpy().astype(np.float64)


def oracle_rotations(inst, variant=0, n_calib=None):
    cq = inst.calib_q if n_calib is None else [x[:n_calib] for x in inst.calib_q]
    ck = inst.calib_k if n_calib is None else [x[:n_calib] for x in inst.calib_k]
    cv = inst.calib_v if n_calib is None else [x[:n_calib] for x in inst.calib_v]
    return attention.calibrate(cq, ck, cv, variant)


def make_cache(inst, rot, *, window, sink=4, growth=0, shared=0, permute=None, lens=None,
               max_len=None, bits=2):
    w = inst.workload
    lens = inst.seq_lens if lens is None else lens
    pp = pages.plan(lens, sink, window, shared_prefix_tokens=shared, growth=growth,
                    permute_seed=permute, max_len=max_len)
    c = pages.allocate(pp, hkv=w.num_kv_heads, hq=w.num_q_heads, d=w.head_dim, sink=sink,
                       window=window, device=DEV, r_k=np.stack(rot.rk), r_v=np.stack(rot.rv),
                       clip_k=np.array(rot.ck, np.float32), clip_v=np.array(rot.cv, np.float32),
                       code_bits=bits)
    return c, pp


def misaligned_copy(x):
    """A device copy of x whose data starts 8 bytes past a 16-byte boundary:
    inputs the tensor-memory-access prefill cannot take, so the library runs its
    CUDA-core quantiser instead."""
    t = torch()
    buf = t.empty(x.numel() + 8, dtype=x.dtype, device=x.device)
    view = buf[4:4 + x.numel()].view(x.shape)
    view.copy_(x)
    assert view.data_ptr() % 16 == 8
    return view


def prefill(cache, inst, lens=None, upto=None, misalign=False):
    """Place tokens [0, upto_b) of every sequence (default: all), final length lens.
    misalign: hand the key/value rows over at an address the tensor-core path
    rejects (the CUDA-core quantiser then places them)."""
    t = torch()
    lens = inst.seq_lens if lens is None else np.asarray(lens)
    ks, vs, sid, pos = [], [], [], []
    for b, L in enumerate(lens):
        n = int(L) if upto is None else int(upto[b])
        H = inst.workload.num_kv_heads
        ks.append(np.stack([inst.k[b][h][:n] for h in range(H)], 1))
        vs.append(np.stack([inst.v[b][h][:n] for h in range(H)], 1))
        sid.append(np.full(n, b, np.int32))
        pos.append(np.arange(n, dtype=np.int32))
    k = bf16_tensor(np.concatenate(ks))
    v = bf16_tensor(np.concatenate(vs))
    if misalign:
        k, v = misaligned_copy(k), misaligned_copy(v)
    L = lib()
    L.oscar_prefill_quantize(cache, k, v, t.from_numpy(np.concatenate(sid)).to(DEV),
                             t.from_numpy(np.concatenate(pos)).to(DEV),
                             t.from_numpy(np.asarray(lens, np.int32)).to(DEV))
    t.cuda.synchronize()


def pools(cache):
    t = torch()
    if t.cuda.is_available():
        t.cuda.synchronize()
    return cache.int2_pool.cpu().numpy(), cache.bf16_pool.view(t.int16).cpu().numpy().view(np.uint16)


def expected(inst, rot, pp, *, window, sink=4, lens=None, kappa=None, bits=2):
    w = inst.workload
    lens = inst.seq_lens if lens is None else lens
    return ocache.expected_pools(inst.k, inst.v, lens, rot, sink=sink, window=window,
                                 d=w.head_dim, hkv=w.num_kv_heads, int2_table=pp.int2_table,
                                 bf16_table=pp.bf16_table, num_int2_pages=pp.num_int2_pages,
                                 num_bf16_pages=pp.num_bf16_pages, kappa=kappa, bits=bits)


def compare_pools(cache, exp):
    """Bit-exact on every byte the oracle defines, except bytes of flagged
    near-boundary entries; returns (#mismatched flagged bytes, #flagged bytes)."""
    got2, gotb = pools(cache)
    bad = exp.int2_defined & ~exp.int2_maydiffer & (got2 != exp.int2)
    assert not bad.any(), f"{int(bad.sum())} INT2 bytes differ outside flagged entries; first at {np.flatnonzero(bad)[:8]}"
    badb = exp.bf16_defined & (gotb != exp.bf16)
    assert not badb.any(), f"{int(badb.sum())} BF16 elements differ"
    flagged = exp.int2_defined & exp.int2_maydiffer
    return int((flagged & (got2 != exp.int2)).sum()), int(flagged.sum())


def decode(cache, q, lens, max_len=None, bf16_only=False, out=None):
    t = torch()
    L = lib()
    lens = np.asarray(lens, np.int32)
    max_len = int(lens.max()) if max_len is None else max_len
    B, Hq, d = q.shape
    qt = bf16_tensor(q)
    o = t.zeros((B, Hq, d), dtype=t.bfloat16, device=DEV) if out is None else out
    ws_bytes = L.oscar_decode_workspace_size(cache, B, max_len)
    ws = t.zeros(ws_bytes // 4 + 64, dtype=t.float32, device=DEV)
    lt = t.from_numpy(lens).to(DEV)
    fn = L.oscar_decode_attention_bf16 if bf16_only else L.oscar_decode_attention
    fn(cache, qt, lt, max_len, o, ws)
    t.cuda.synchronize()
    return from_bf16(o)


def attention_from_pools(cache, pp, q, lens, rot, *, sink, window, gqa, drop=None, upto=None,
                         heads=None, seqs=None):
    """The oracle's attention over what the GPU actually stored: every token of
    every sequence read back from the pools (INT2 codes, s16, z16 dequantised and
    rotated back with R^T; BF16 tokens as stored), then fp64 softmax attention.
    Separates the decode kernels' parity from the quantiser's (whose flagged
    near-boundary codes may differ from the oracle's by one step).  ``drop``:
    optional {sequence: logical pages} whose tokens are left out.  ``upto``:
    optional last visible position per sequence (a query row of a chunk).  The
    code width (INT2 or the INT4 variant) is the cache's ``code_bits``.
    ``heads``: optional KV heads to compute (the others' outputs stay zero).
    ``seqs``: optional sequences to compute (likewise)."""
    got2, gotb = pools(cache)
    B, Hq, d = q.shape
    hkv = Hq // gqa
    bits = getattr(cache, "code_bits", 2)
    blk2 = layout.int2_block_bytes(d, bits)
    blkb = layout.bf16_block_bytes(d) // 2
    out = np.zeros((B, Hq, d))
    for b in (range(B) if seqs is None else seqs):
        L = int(lens[b])
        t = np.arange(L)
        m = ocache.is_int2(t, L, sink, window)
        for h in (range(hkv) if heads is None else heads):
            k = np.zeros((L, d))
            v = np.zeros((L, d))
            for pg in range((L + 15) // 16):
                ts = t[16 * pg:16 * pg + 16]
                slots = ts - 16 * pg
                mi = m[ts]
                if mi.any():
                    pid = int(pp.int2_table[b, pg])
                    kc, ks, kz, vc, vs, vz = layout.unpack_int2_block(
                        got2[(pid * hkv + h) * blk2:(pid * hkv + h + 1) * blk2], d, bits)
                    sl = slots[mi]
                    yk = quant.dequantize(kc[sl], ks[sl], kz[sl])
                    yv = quant.dequantize(vc[sl], vs[sl], vz[sl])
                    k[ts[mi]] = yk @ np.asarray(rot.rk[h], np.float64).T
                    v[ts[mi]] = yv @ np.asarray(rot.rv[h], np.float64).T
                if (~mi).any():
                    pid = int(pp.bf16_table[b, pg])
                    kb, vb = layout.unpack_bf16_block(gotb[(pid * hkv + h) * blkb:(pid * hkv + h + 1) * blkb], d)
                    sl = slots[~mi]
                    k[ts[~mi]] = synth.bf16_from_bits(kb[sl])
                    v[ts[~mi]] = synth.bf16_from_bits(vb[sl])
            keep = np.ones(L, bool)
            for pg in (drop or {}).get(b, ()):
                keep[16 * pg:16 * pg + 16] = False
            if upto is not None:
                keep[int(upto[b]) + 1:] = False
            out[b, h * gqa:(h + 1) * gqa] = attention.softmax_attention(q[b, h * gqa:(h + 1) * gqa],
                                                                      k[keep], v[keep])
    return out


def status(cache):
    return int(cache.status.cpu().item())


def bf16_half_ulp(x):
    """Half a bf16 ulp at |x| (8 significant bits): the store's own rounding."""
    x = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(x)) - 8)


# the last check_close's largest deviation beyond the bf16 rounding of ref
LAST_CHECK = {}


def check_close(got, ref, what=""):
    """Output parity: rel-L2 <= 5e-3 and, per element, |got - ref| <= 1e-2 plus
    half a bf16 ulp of ref (the output is stored in bf16; for |out| >= 4 the
    rounding of an exact result alone can exceed 1e-2)."""
    dev = np.abs(got - ref)
    excess = dev - bf16_half_ulp(ref)
    err = float(dev.max())
    worst = float(excess.max())
    rel = attention.rel_l2(got, ref)
    LAST_CHECK["excess"] = worst
    assert worst <= TOL_MAX_ABS and rel <= TOL_REL_L2, \
        f"{what}: max-abs {err:.3e} (beyond bf16 rounding {worst:.3e}), rel-L2 {rel:.3e}"
    return err, rel


def kappa(d):
    # sequential fp32 FMA chain of d terms: |error| <= d * 2^-24 * sum |x_i R_ij|
    return 1.01 * d * 2.0 ** -24


# ---------------------------------------------------------------- traced placement
#
# The quantising kernels' diagnostic forms return the fp32 rotated values y they
# computed.  That splits the check of a placement in two:
#   rotation:  |y_kernel - x R| <= kappa * sum_i |x_i| |R_ij|, with x R exact (fp64)
#              and kappa the a-priori error bound of the kernel's fp32 arithmetic;
#   decisions: clip, group range, s16, z16 and every code are a function of y
#              alone, so the stored entries must equal the oracle's quantiser
#              applied to y_kernel, bit for bit, in every group (no exemptions).

# tensor-core prefill: x (bf16) times R split into three bf16 pieces, products
# exact, 3d of them summed in fp32 by the tensor core (truncating adds allowed)
def kappa_tc(d):
    return 3 * d * 2.0 ** -23


def prefill_trace(cache, inst, lens=None, upto=None, misalign=False):
    """As ``prefill`` through oscar_prefill_quantize_trace.  Returns
    (y float32 [T, Hkv, 2, d], {b: (first item, count)})."""
    t = torch()
    lens = inst.seq_lens if lens is None else np.asarray(lens)
    H = inst.workload.num_kv_heads
    ks, vs, sid, pos, where = [], [], [], [], {}
    at = 0
    for b, L in enumerate(lens):
        n = int(L) if upto is None else int(upto[b])
        ks.append(np.stack([inst.k[b][h][:n] for h in range(H)], 1))
        vs.append(np.stack([inst.v[b][h][:n] for h in range(H)], 1))
        sid.append(np.full(n, b, np.int32))
        pos.append(np.arange(n, dtype=np.int32))
        where[b] = (at, n)
        at += n
    k = bf16_tensor(np.concatenate(ks))
    v = bf16_tensor(np.concatenate(vs))
    if misalign:
        k, v = misaligned_copy(k), misaligned_copy(v)
    y = t.full((at, H, 2, inst.workload.head_dim), float("nan"), dtype=t.float32, device=DEV)
    L = lib()
    L.oscar_prefill_quantize_trace(cache, k, v, t.from_numpy(np.concatenate(sid)).to(DEV),
                                   t.from_numpy(np.concatenate(pos)).to(DEV),
                                   t.from_numpy(np.asarray(lens, np.int32)).to(DEV), y)
    t.cuda.synchronize()
    return y.cpu().numpy(), where


def stored_int2(cache, pp, b, h, positions, d, bits=2, pools_=None):
    """The INT2 entries the pools hold for positions of sequence b, KV head h:
    (kc, ks, kz, vc, vs, vz), codes [n, d], scales and zeros [n, d/32]."""
    got2 = pools(cache)[0] if pools_ is None else pools_
    hkv = cache.num_kv_heads
    blk = layout.int2_block_bytes(d, bits)
    positions = np.asarray(positions, np.int64)
    n, ng = positions.size, d // 32
    out = [np.zeros((n, d), np.uint8), np.zeros((n, ng), np.float16), np.zeros((n, ng), np.float16),
           np.zeros((n, d), np.uint8), np.zeros((n, ng), np.float16), np.zeros((n, ng), np.float16)]
    for pg in np.unique(positions // 16):
        sel = np.flatnonzero(positions // 16 == pg)
        pid = int(pp.int2_table[b, pg])
        parts = layout.unpack_int2_block(got2[(pid * hkv + h) * blk:(pid * hkv + h + 1) * blk], d, bits)
        slots = positions[sel] - 16 * pg
        for o, part in zip(out, parts):
            o[sel] = part[slots]
    return tuple(out)


def check_traced(cache, pp, inst, rot, rows, kappa, *, lens, sink, window, bits=2, pools_=None):
    """Rotation and decision checks of traced placements.

    rows: {b: (positions, y float32 [n, Hkv, 2, d])}; only positions in the
    INT2 region of sequence b (length lens[b]) are checked.  Returns counts:
    groups checked, the largest |y_kernel - x R| / sum |x| |R| seen, and the
    groups whose stored entries differ from the oracle's placement from the
    exact x R (allowed only where y_kernel and x R straddle a decision)."""
    levels = quant.INT2_MAX_CODE if bits == 2 else quant.INT4_MAX_CODE
    w = inst.workload
    d, hkv = w.head_dim, w.num_kv_heads
    got2 = pools(cache)[0] if pools_ is None else pools_
    groups = straddle = 0
    worst = 0.0
    for b, (positions, yb) in rows.items():
        positions = np.asarray(positions, np.int64)
        m = ocache.is_int2(positions, int(lens[b]), sink, window)
        ti, yb = positions[m], yb[m]
        if ti.size == 0:
            continue
        for h in range(hkv):
            st = stored_int2(cache, pp, b, h, ti, d, bits, got2)
            for kv, (xs, r, c, (sc, ss, sz)) in enumerate((
                    (inst.k, rot.rk[h], rot.ck[h], st[:3]), (inst.v, rot.rv[h], rot.cv[h], st[3:]))):
                x = np.asarray(xs[b][h], np.float64)[ti]
                yk = yb[:, h, kv, :].astype(np.float64)
                assert np.isfinite(yk).all(), "a traced INT2 placement wrote no rotated values"
                ye = quant.rotate(x, r)
                bnd = np.abs(x) @ np.abs(np.asarray(r, np.float64))
                err = np.abs(yk - ye)
                assert (err <= kappa * bnd).all(), \
                    f"rotation error {float((err / np.maximum(bnd, 1e-300)).max()):.3e} beyond {kappa:.3e}"
                worst = max(worst, float((err / np.maximum(bnd, 1e-300)).max()))
                qc, qs, qz = quant.quantize(yk, c, levels=levels)
                np.testing.assert_array_equal(sc, qc, err_msg=f"codes, seq {b} head {h} kv {kv}")
                np.testing.assert_array_equal(ss.view(np.uint16), qs.view(np.uint16))
                np.testing.assert_array_equal(sz.view(np.uint16), qz.view(np.uint16))
                ec, es, ez = quant.quantize(ye, c, levels=levels)
                differs = ((ec != qc).reshape(len(ti), -1, 32).any(-1) | (es.view(np.uint16) != qs.view(np.uint16))
                           | (ez.view(np.uint16) != qz.view(np.uint16)))
                groups += differs.size
                straddle += int(differs.sum())
    return {"groups": groups, "max_rotation_error_ratio": worst, "straddling_groups": straddle}


def report(name, **stats):
    """Append one JSON line of parity statistics to the file named by the
    environment variable OSCAR_PARITY_REPORT (nothing when it is unset)."""
    import json
    import os
    path = os.environ.get("OSCAR_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"test": name, **stats}) + "\n")
