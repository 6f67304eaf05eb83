"""Expected page-pool contents of the mixed-precision cache.

[Summary 2.2B] Mixed-Precision Layout: sink tokens (the first ones) and recent
tokens stay in BF16; the middle history is stored in INT2 after rotation and
clipping.  Readings taken where the pages are silent: S = 4 sink tokens, a
recent window of W tokens, and for a sequence of length L (current token
included) token t is BF16 when t < S or t >= L - W and INT2 otherwise.  BF16
tokens are stored unrotated.  On a decode step that brings the length to L,
the token L - 1 - W leaves the window and moves to INT2 (once L > S + W).

Physical placement: logical page p = t // 16, slot t % 16; the page tables map
(sequence, logical page) to a physical page id (two tables: INT2 pages and BF16
pages).  Prefix sharing is equal ids in several sequences' rows.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import layout, quant

PAGE = 16


def is_int2(t, L: int, sink: int, window: int):
    t = np.asarray(t)
    return (t >= sink) & (t < L - window)


@dataclasses.dataclass
class Rotations:
    rk: list      # per KV head fp32 [d, d]
    rv: list
    ck: list      # per KV head fp32 clip
    cv: list


@dataclasses.dataclass
class ExpectedPools:
    int2: np.ndarray          # uint8 [num_int2_pages * Hkv * 12d]
    int2_defined: np.ndarray  # bool, bytes owned by a token stored in INT2
    int2_maydiffer: np.ndarray  # bool, bytes of near-boundary entries (see quant)
    bf16: np.ndarray          # uint16 [num_bf16_pages * Hkv * 32d]
    bf16_defined: np.ndarray
    n_flag_elems: int = 0
    n_flag_groups: int = 0


def expected_pools(k, v, lens, rot: Rotations, *, sink: int, window: int, d: int, hkv: int,
                   int2_table: np.ndarray, bf16_table: np.ndarray,
                   num_int2_pages: int, num_bf16_pages: int, kappa: float | None = None,
                   tokens=None, bits: int = 2) -> ExpectedPools:
    """Pools after every token of every sequence has been placed.

    k[b][h], v[b][h]: float arrays [L_b, d] of bf16 values.  ``tokens`` (optional)
    restricts to a dict {b: iterable of positions}; by default all positions.
    ``kappa`` enables near-boundary flags for kernels with fp32 rotation error.
    ``bits``: 2 (INT2 pages) or 4 (the INT4 variant: codes 0..15 in two planes).
    """
    levels = quant.INT2_MAX_CODE if bits == 2 else quant.INT4_MAX_CODE
    blk = layout.int2_block_bytes(d, bits)
    bblk = layout.bf16_block_bytes(d) // 2
    int2 = np.zeros(num_int2_pages * hkv * blk, np.uint8)
    idef = np.zeros_like(int2, dtype=bool)
    imay = np.zeros_like(int2, dtype=bool)
    bf = np.zeros(num_bf16_pages * hkv * bblk, np.uint16)
    bdef = np.zeros_like(bf, dtype=bool)
    tb = layout.tables(d, bits)
    owner, bowner = tb["owner"], tb["bowner"]
    o = layout.offsets(d, bits)
    plane_offs = [o["plane"] * q for q in range(layout.planes(bits))]
    ng = d // quant.GROUP
    nfe = nfg = 0
    for b, L in enumerate(lens):
        L = int(L)
        pos = np.arange(L) if tokens is None else np.asarray(sorted(tokens[b]), np.int64)
        if pos.size == 0:
            continue
        m_int2 = is_int2(pos, L, sink, window)
        for h in range(hkv):
            kk = np.asarray(k[b][h], np.float64)
            vv = np.asarray(v[b][h], np.float64)
            ti = pos[m_int2]
            if ti.size:
                kc, ks, kz = quant.quantize(quant.rotate(kk[ti], rot.rk[h]), rot.ck[h], levels=levels)
                vc, vs, vz = quant.quantize(quant.rotate(vv[ti], rot.rv[h]), rot.cv[h], levels=levels)
                if kappa is not None:
                    ekf, gkf = quant.near_boundary_flags(kk[ti], rot.rk[h], rot.ck[h], kappa,
                                                         levels=levels)
                    evf, gvf = quant.near_boundary_flags(vv[ti], rot.rv[h], rot.cv[h], kappa,
                                                         levels=levels)
                    nfe += int(ekf.sum() + evf.sum())
                    nfg += int(gkf.sum() + gvf.sum())
                for n, t in enumerate(ti):
                    page = int(int2_table[b, t // PAGE])
                    base = (page * hkv + h) * blk
                    block = int2[base:base + blk]
                    slot = int(t % PAGE)
                    layout.pack_int2_block(block, d, slot, kc[n], ks[n], kz[n], vc[n], vs[n], vz[n],
                                           bits=bits)
                    idef[base:base + blk] |= owner == slot
                    if kappa is not None:
                        may = imay[base:base + blk]
                        for po in plane_offs:
                            kbytes = o["Kc"] + po + tb["kbyte"][slot]
                            vbytes = o["Vc"] + po + tb["vbyte"][slot]
                            for g in range(ng):
                                cols = slice(32 * g, 32 * g + 32)
                                if gkf[n, g]:
                                    may[kbytes[cols]] = True
                                if gvf[n, g]:
                                    may[vbytes[cols]] = True
                            may[kbytes[ekf[n]]] = True
                            may[vbytes[evf[n]]] = True
                        for g in range(ng):
                            if gkf[n, g]:
                                e0 = o["Ksz"] + 4 * (slot * ng + g)
                                may[e0:e0 + 4] = True
                            if gvf[n, g]:
                                for part in ("Vs", "Vz"):
                                    e0 = o[part] + 2 * tb["vsz"][slot, g]
                                    may[e0:e0 + 2] = True
            tb16 = pos[~m_int2]
            for t in tb16:
                page = int(bf16_table[b, t // PAGE])
                base = (page * hkv + h) * bblk
                block = bf[base:base + bblk]
                slot = int(t % PAGE)
                kb = (np.asarray(kk[t], np.float32).view(np.uint32) >> 16).astype(np.uint16)
                vb = (np.asarray(vv[t], np.float32).view(np.uint32) >> 16).astype(np.uint16)
                layout.pack_bf16_block(block, d, slot, kb, vb)
                bdef[base:base + bblk] |= bowner == slot
    return ExpectedPools(int2, idef, imay, bf, bdef, nfe, nfg)
