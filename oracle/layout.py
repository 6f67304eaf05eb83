"""The library's page formats, written out as index formulas.

The pages require a paged KV cache with BF16 sink/recent tokens and INT2
history [Summary 2.2B] but fix no byte layout; the layout is the library's own.
It is restated here independently of the kernels so that pool contents written
by the GPU can be compared byte for byte.

Constants: P = 16 tokens per page, groups of 32 channels, head dim d in {64, 128},
ng = d/32 groups, token t in [0, 16), channel j in [0, d).

INT2 page-head block (12*d bytes), byte offsets:
  Kc  [0,    4d)   key codes      Ksz [4d,  6d)  key (s16, z16) pairs
  Vc  [6d,  10d)   value codes    Vs  [10d, 11d) value s16     Vz [11d, 12d) value z16
Codes are 2-bit fields of little-endian 32-bit words, addressed by a lane
L in [0,32) and a word m in [0, d/32) (``k_code_pos`` / ``v_code_pos``):
  key   (t, j):  kk=j>>4, h=(j>>3)&1, tig=(j>>1)&3, e=j&1, gid=t&7, th=t>>3
                 L=4*gid+tig, m=kk>>1, i=kk&1, s=2*th+h
  value (t, j):  mt=j>>4, ch=(j>>3)&1, gid=j&7, tig=(t>>1)&3, e=t&1, th=t>>3
                 L=4*gid+tig, m=mt>>1, i=mt&1, s=ch+2*th
  word = L*(d/32) + m,  bit = 16*e + 4*s + 2*i.
Every byte of Kc / Vc holds codes of a single token.
Ksz: 32-bit entries (s16 low half, z16 high half) at index t*ng + grp.
Vs, Vz: fp16 at index ((tig*2 + th)*ng + grp)*2 + e with t = 8*th + 2*tig + e.

BF16 page-head block (64*d bytes): key part then value part, 16*d bf16 each,
as 32-bit words of two bf16 (first element in the low half):
  key   (t, j): word (kk*32 + L)*4 + r, r = th + 2*h   (kk,h,tig,e,gid,th as above)
  value (t, j): word (mt*32 + L)*4 + r, r = ch + 2*th  (mt,ch,gid,tig,e,th as above)
  element index = 2*word + e.

Pools: block (physical page p, KV head h) sits at (p*Hkv + h) * block_bytes.

INT4 variant (bits = 4): a 4-bit code c is stored as two 2-bit planes, the high
bits c >> 2 in plane 0 and the low bits c & 3 in plane 1, each plane laid out
exactly as the INT2 code area above.  Block (20*d bytes):
  Kc plane 0 [0, 4d) | Kc plane 1 [4d, 8d) | Ksz [8d, 10d) | Vc plane 0 [10d, 14d)
  | Vc plane 1 [14d, 18d) | Vs [18d, 19d) | Vz [19d, 20d).
In general with P = bits/2 planes: Kc plane q at 4d*q, Ksz at 4dP, Vc plane q
at 4dP + 2d + 4d*q, Vs at 8dP + 2d, Vz at 8dP + 3d; block (8P + 4)*d bytes.
"""
from __future__ import annotations

import numpy as np

PAGE = 16
GROUP = 32


def planes(bits: int) -> int:
    if bits not in (2, 4):
        raise ValueError("code bits must be 2 or 4")
    return bits // 2


def int2_block_bytes(d: int, bits: int = 2) -> int:
    """Bytes of one code page-head block (INT2: 12d, INT4: 20d)."""
    return (8 * planes(bits) + 4) * d


def bf16_block_bytes(d: int) -> int:
    return 64 * d


def offsets(d: int, bits: int = 2) -> dict:
    """Byte offsets of the block's parts; Kc / Vc are plane 0, plane q adds 4d*q."""
    P = planes(bits)
    return {"Kc": 0, "Ksz": 4 * d * P, "Vc": 4 * d * P + 2 * d, "Vs": 8 * d * P + 2 * d,
            "Vz": 8 * d * P + 3 * d, "plane": 4 * d}


def k_code_pos(t: int, j: int, d: int):
    """(byte offset inside Kc, bit offset inside that byte) of key code (t, j)."""
    kk, h, tig, e = j >> 4, (j >> 3) & 1, (j >> 1) & 3, j & 1
    gid, th = t & 7, t >> 3
    lane, m, i, s = 4 * gid + tig, kk >> 1, kk & 1, 2 * th + h
    word = lane * (d // 32) + m
    bit = 16 * e + 4 * s + 2 * i
    return 4 * word + bit // 8, bit % 8


def v_code_pos(t: int, j: int, d: int):
    """(byte offset inside Vc, bit offset inside that byte) of value code (t, j)."""
    mt, ch, gid = j >> 4, (j >> 3) & 1, j & 7
    tig, e, th = (t >> 1) & 3, t & 1, t >> 3
    lane, m, i, s = 4 * gid + tig, mt >> 1, mt & 1, ch + 2 * th
    word = lane * (d // 32) + m
    bit = 16 * e + 4 * s + 2 * i
    return 4 * word + bit // 8, bit % 8


def vsz_index(t: int, grp: int, d: int) -> int:
    ng = d // GROUP
    th, tig, e = t >> 3, (t >> 1) & 3, t & 1
    return ((tig * 2 + th) * ng + grp) * 2 + e


def bf16_k_elem(t: int, j: int) -> int:
    kk, h, tig, e = j >> 4, (j >> 3) & 1, (j >> 1) & 3, j & 1
    gid, th = t & 7, t >> 3
    lane, r = 4 * gid + tig, th + 2 * h
    return 2 * ((kk * 32 + lane) * 4 + r) + e


def bf16_v_elem(t: int, j: int) -> int:
    mt, ch, gid = j >> 4, (j >> 3) & 1, j & 7
    tig, e, th = (t >> 1) & 3, t & 1, t >> 3
    lane, r = 4 * gid + tig, ch + 2 * th
    return 2 * ((mt * 32 + lane) * 4 + r) + e


# ----------------------------------------------------------------------------
# Tables (cached per d) so packing whole pools stays vectorised
# ----------------------------------------------------------------------------

_TABLES: dict = {}


def tables(d: int, bits: int = 2) -> dict:
    if (d, bits) in _TABLES:
        return _TABLES[(d, bits)]
    ng = d // GROUP
    kbyte = np.zeros((PAGE, d), np.int64)
    kbit = np.zeros((PAGE, d), np.int64)
    vbyte = np.zeros((PAGE, d), np.int64)
    vbit = np.zeros((PAGE, d), np.int64)
    bk = np.zeros((PAGE, d), np.int64)
    bv = np.zeros((PAGE, d), np.int64)
    for t in range(PAGE):
        for j in range(d):
            kbyte[t, j], kbit[t, j] = k_code_pos(t, j, d)
            vbyte[t, j], vbit[t, j] = v_code_pos(t, j, d)
            bk[t, j] = bf16_k_elem(t, j)
            bv[t, j] = bf16_v_elem(t, j)
    vsz = np.zeros((PAGE, ng), np.int64)
    for t in range(PAGE):
        for g in range(ng):
            vsz[t, g] = vsz_index(t, g, d)
    o = offsets(d, bits)
    # owner token of every byte of a code block (each byte belongs to one token)
    owner = np.full(int2_block_bytes(d, bits), -1, np.int64)
    for q in range(planes(bits)):
        owner[o["Kc"] + o["plane"] * q + kbyte] = np.repeat(np.arange(PAGE), d).reshape(PAGE, d)
        owner[o["Vc"] + o["plane"] * q + vbyte] = np.repeat(np.arange(PAGE), d).reshape(PAGE, d)
    for t in range(PAGE):
        for g in range(ng):
            base = o["Ksz"] + 4 * (t * ng + g)
            owner[base:base + 4] = t
            for part in ("Vs", "Vz"):
                b = o[part] + 2 * vsz[t, g]
                owner[b:b + 2] = t
    bowner = np.full(bf16_block_bytes(d) // 2, -1, np.int64)
    bowner[bk] = np.repeat(np.arange(PAGE), d).reshape(PAGE, d)
    bowner[16 * d + bv] = np.repeat(np.arange(PAGE), d).reshape(PAGE, d)
    tb = dict(kbyte=kbyte, kbit=kbit, vbyte=vbyte, vbit=vbit, bk=bk, bv=bv, vsz=vsz,
              owner=owner, bowner=bowner)
    _TABLES[(d, bits)] = tb
    return tb


def pack_int2_block(block: np.ndarray, d: int, t: int, kc, ks, kz, vc, vs, vz,
                    bits: int = 2) -> None:
    """Write token t's codes/scales/zeros into a code block (uint8, in place;
    12d bytes for INT2, 20d for INT4).

    kc, vc: uint8 [d] codes (0..3 or 0..15); ks, kz, vs, vz: float16 [ng]."""
    tb = tables(d, bits)
    o = offsets(d, bits)
    ng = d // GROUP
    P = planes(bits)
    kc = np.asarray(kc, np.uint8)
    vc = np.asarray(vc, np.uint8)
    for q in range(P):
        shift = 2 * (P - 1 - q)          # plane 0 holds the highest two bits
        kb = o["Kc"] + o["plane"] * q + tb["kbyte"][t]
        vb = o["Vc"] + o["plane"] * q + tb["vbyte"][t]
        # clear this token's code bytes, then OR the fields in
        block[kb] = 0
        block[vb] = 0
        np.bitwise_or.at(block, kb, (((kc >> shift) & 3) << tb["kbit"][t]).astype(np.uint8))
        np.bitwise_or.at(block, vb, (((vc >> shift) & 3) << tb["vbit"][t]).astype(np.uint8))
    ksz = np.zeros(ng * 2, np.float16)
    ksz[0::2] = ks
    ksz[1::2] = kz
    block[o["Ksz"] + 4 * t * ng: o["Ksz"] + 4 * (t + 1) * ng] = ksz.view(np.uint8)
    vs_view = block[o["Vs"]:o["Vz"]].view(np.float16)
    vz_view = block[o["Vz"]:o["Vz"] + d].view(np.float16)
    vs_view[tb["vsz"][t]] = vs
    vz_view[tb["vsz"][t]] = vz


def unpack_int2_block(block: np.ndarray, d: int, bits: int = 2):
    """Inverse of ``pack_int2_block`` for all 16 slots: (kc, ks, kz, vc, vs, vz)."""
    tb = tables(d, bits)
    o = offsets(d, bits)
    ng = d // GROUP
    P = planes(bits)
    kc = np.zeros((PAGE, d), np.int64)
    vc = np.zeros((PAGE, d), np.int64)
    for q in range(P):
        shift = 2 * (P - 1 - q)
        kc |= ((block[o["Kc"] + o["plane"] * q + tb["kbyte"]] >> tb["kbit"]) & 3).astype(np.int64) << shift
        vc |= ((block[o["Vc"] + o["plane"] * q + tb["vbyte"]] >> tb["vbit"]) & 3).astype(np.int64) << shift
    ksz = block[o["Ksz"]:o["Vc"]].view(np.float16).reshape(PAGE, ng, 2)
    vs_view = block[o["Vs"]:o["Vz"]].view(np.float16)
    vz_view = block[o["Vz"]:o["Vz"] + d].view(np.float16)
    return (kc.astype(np.uint8), ksz[..., 0].copy(), ksz[..., 1].copy(), vc.astype(np.uint8),
            vs_view[tb["vsz"]].copy(), vz_view[tb["vsz"]].copy())


def pack_bf16_block(block16: np.ndarray, d: int, t: int, k_bits, v_bits) -> None:
    """Write token t's bf16 key/value bit patterns (uint16 [d]) into a BF16 block
    viewed as uint16 [32d]."""
    tb = tables(d)
    block16[tb["bk"][t]] = k_bits
    block16[16 * d + tb["bv"][t]] = v_bits


def unpack_bf16_block(block16: np.ndarray, d: int):
    tb = tables(d)
    return block16[tb["bk"]].copy(), block16[16 * d + tb["bv"]].copy()
