"""Pins for the page formats (oracle/layout.py).

The formats are the library's own choice (the pages fix none), so they are
pinned structurally: every code / scale / value has exactly one home, every
code byte belongs to one token, pack and unpack are inverse, and a lane's words
yield exactly the m16n8k16 operand fragments the PTX ISA defines for the
layout's intended use (A = keys [token x channel] for q.K, A = values^T
[channel x token] for p.V).
"""
import numpy as np
import pytest

from oracle import layout


def frag_a(lane, reg):
    """PTX ISA, mma.m16n8k16 .f16/.bf16, A fragment: (row, col) of the two
    elements held in register ``reg`` (low half first)."""
    gid, tig = lane >> 2, lane & 3
    row = gid + 8 * (reg & 1)
    col = 2 * tig + 8 * (reg >> 1)
    return [(row, col), (row, col + 1)]


@pytest.mark.parametrize("d", [64, 128])
def test_code_positions_are_a_bijection(d):
    for pos in (layout.k_code_pos, layout.v_code_pos):
        seen = set()
        for t in range(16):
            for j in range(d):
                byte, bit = pos(t, j, d)
                assert 0 <= byte < 4 * d and bit in (0, 2, 4, 6)
                seen.add((byte, bit))
        assert len(seen) == 16 * d


@pytest.mark.parametrize("d", [64, 128])
def test_each_byte_belongs_to_one_token(d):
    tb = layout.tables(d)
    assert np.all(tb["owner"] >= 0)            # every byte of the block is owned
    for key in ("kbyte", "vbyte"):
        by = tb[key]
        for t in range(16):
            others = np.delete(by, t, axis=0)
            assert not np.intersect1d(by[t], others).size
    assert np.all(tb["bowner"] >= 0)
    assert sorted(tb["bk"].ravel()) == list(range(16 * d))
    assert sorted(tb["bv"].ravel()) == list(range(16 * d))


@pytest.mark.parametrize("d", [64, 128])
def test_pack_unpack_roundtrip(d):
    rng = np.random.default_rng(0)
    ng = d // 32
    blk = np.zeros(layout.int2_block_bytes(d), np.uint8)
    kc = rng.integers(0, 4, (16, d)).astype(np.uint8)
    vc = rng.integers(0, 4, (16, d)).astype(np.uint8)
    ks, kz, vs, vz = (rng.standard_normal((16, ng)).astype(np.float16) for _ in range(4))
    for t in rng.permutation(16):
        layout.pack_int2_block(blk, d, t, kc[t], ks[t], kz[t], vc[t], vs[t], vz[t])
    out = layout.unpack_int2_block(blk, d)
    for a, b in zip(out, (kc, ks, kz, vc, vs, vz)):
        np.testing.assert_array_equal(a, b)
    # overwrite one slot: others unchanged
    layout.pack_int2_block(blk, d, 3, 3 - kc[3], ks[3], kz[3], 3 - vc[3], vs[3], vz[3])
    out2 = layout.unpack_int2_block(blk, d)
    np.testing.assert_array_equal(out2[0][3], 3 - kc[3])
    np.testing.assert_array_equal(np.delete(out2[0], 3, 0), np.delete(kc, 3, 0))
    b16 = np.zeros(layout.bf16_block_bytes(d) // 2, np.uint16)
    kb = rng.integers(0, 65535, (16, d)).astype(np.uint16)
    vb = rng.integers(0, 65535, (16, d)).astype(np.uint16)
    for t in range(16):
        layout.pack_bf16_block(b16, d, t, kb[t], vb[t])
    k2, v2 = layout.unpack_bf16_block(b16, d)
    np.testing.assert_array_equal(k2, kb)
    np.testing.assert_array_equal(v2, vb)


def _words(block, off, n):
    return block[off:off + 4 * n].view("<u4")


@pytest.mark.parametrize("d", [64, 128])
def test_int2_words_give_mma_fragments(d):
    """Lane L's words, split with (w >> 4s) & (3 << 2i) per 16-bit half, are the
    A fragments: keys for k-step kk (rows = tokens, cols = channels 16kk..),
    values for channel tile mt (rows = channels 16mt.., cols = tokens)."""
    rng = np.random.default_rng(1)
    ng = d // 32
    kc = rng.integers(0, 4, (16, d)).astype(np.uint8)
    vc = rng.integers(0, 4, (16, d)).astype(np.uint8)
    z = np.zeros((16, ng), np.float16)
    blk = np.zeros(layout.int2_block_bytes(d), np.uint8)
    for t in range(16):
        layout.pack_int2_block(blk, d, t, kc[t], z[t], z[t], vc[t], z[t], z[t])
    o = layout.offsets(d)
    kw = _words(blk, o["Kc"], d).reshape(32, d // 32)
    vw = _words(blk, o["Vc"], d).reshape(32, d // 32)
    s_of_reg_k = [0, 2, 1, 3]          # key words: s = 2*th + h, reg = th + 2*h
    for lane in range(32):
        for step in range(d // 16):
            m, i = step >> 1, step & 1
            for reg in range(4):
                sk = s_of_reg_k[reg]
                wk = int(kw[lane, m]) >> (4 * sk)
                wv = int(vw[lane, m]) >> (4 * reg)    # value words: s = reg
                (r0, c0), (r1, c1) = frag_a(lane, reg)
                for half, (r, c) in enumerate(((r0, c0), (r1, c1))):
                    ck = (wk >> (16 * half + 2 * i)) & 3
                    cv = (wv >> (16 * half + 2 * i)) & 3
                    assert ck == kc[r, 16 * step + c]
                    assert cv == vc[c, 16 * step + r]


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_words_give_mma_fragments(d):
    rng = np.random.default_rng(2)
    kb = rng.integers(0, 65535, (16, d)).astype(np.uint16)
    vb = rng.integers(0, 65535, (16, d)).astype(np.uint16)
    b16 = np.zeros(layout.bf16_block_bytes(d) // 2, np.uint16)
    for t in range(16):
        layout.pack_bf16_block(b16, d, t, kb[t], vb[t])
    words = b16.view("<u4")
    for lane in range(32):
        for step in range(d // 16):
            for reg in range(4):
                wk = int(words[(step * 32 + lane) * 4 + reg])
                wv = int(words[8 * d + (step * 32 + lane) * 4 + reg])
                (r0, c0), (r1, c1) = frag_a(lane, reg)
                assert wk & 0xFFFF == kb[r0, 16 * step + c0] and wk >> 16 == kb[r1, 16 * step + c1]
                assert wv & 0xFFFF == vb[c0, 16 * step + r0] and wv >> 16 == vb[c1, 16 * step + r1]


# ------------------------------------------------------------ INT4 variant (two planes)

@pytest.mark.parametrize("d", [64, 128])
def test_int4_block_sizes_and_ownership(d):
    assert layout.int2_block_bytes(d, 4) == 20 * d and layout.int2_block_bytes(d) == 12 * d
    o = layout.offsets(d, 4)
    assert (o["Kc"], o["Ksz"], o["Vc"], o["Vs"], o["Vz"]) == (0, 8 * d, 10 * d, 18 * d, 19 * d)
    tb = layout.tables(d, 4)
    assert tb["owner"].size == 20 * d and np.all(tb["owner"] >= 0)
    with pytest.raises(ValueError):
        layout.planes(3)


@pytest.mark.parametrize("d", [64, 128])
def test_int4_pack_unpack_roundtrip(d):
    rng = np.random.default_rng(5)
    ng = d // 32
    blk = np.zeros(layout.int2_block_bytes(d, 4), np.uint8)
    kc = rng.integers(0, 16, (16, d)).astype(np.uint8)
    vc = rng.integers(0, 16, (16, d)).astype(np.uint8)
    ks, kz, vs, vz = (rng.standard_normal((16, ng)).astype(np.float16) for _ in range(4))
    for t in rng.permutation(16):
        layout.pack_int2_block(blk, d, t, kc[t], ks[t], kz[t], vc[t], vs[t], vz[t], bits=4)
    out = layout.unpack_int2_block(blk, d, bits=4)
    for a, b in zip(out, (kc, ks, kz, vc, vs, vz)):
        np.testing.assert_array_equal(a, b)
    layout.pack_int2_block(blk, d, 9, 15 - kc[9], ks[9], kz[9], 15 - vc[9], vs[9], vz[9], bits=4)
    out2 = layout.unpack_int2_block(blk, d, bits=4)
    np.testing.assert_array_equal(out2[3][9], 15 - vc[9])
    np.testing.assert_array_equal(np.delete(out2[3], 9, 0), np.delete(vc, 9, 0))


@pytest.mark.parametrize("d", [64, 128])
def test_int4_planes_are_int2_code_areas(d):
    """Plane 0 of an INT4 block is the INT2 code area of the high bits c >> 2,
    plane 1 that of the low bits c & 3 (so each plane keeps the INT2 fragment
    order pinned above); scales and zeros are the INT2 ones, moved by 8d."""
    rng = np.random.default_rng(6)
    ng = d // 32
    kc = rng.integers(0, 16, (16, d)).astype(np.uint8)
    vc = rng.integers(0, 16, (16, d)).astype(np.uint8)
    ks, kz, vs, vz = (rng.standard_normal((16, ng)).astype(np.float16) for _ in range(4))
    b4 = np.zeros(layout.int2_block_bytes(d, 4), np.uint8)
    hi = np.zeros(layout.int2_block_bytes(d), np.uint8)
    lo = np.zeros(layout.int2_block_bytes(d), np.uint8)
    for t in range(16):
        layout.pack_int2_block(b4, d, t, kc[t], ks[t], kz[t], vc[t], vs[t], vz[t], bits=4)
        layout.pack_int2_block(hi, d, t, kc[t] >> 2, ks[t], kz[t], vc[t] >> 2, vs[t], vz[t])
        layout.pack_int2_block(lo, d, t, kc[t] & 3, ks[t], kz[t], vc[t] & 3, vs[t], vz[t])
    o2, o4 = layout.offsets(d), layout.offsets(d, 4)
    np.testing.assert_array_equal(b4[0:4 * d], hi[0:4 * d])
    np.testing.assert_array_equal(b4[4 * d:8 * d], lo[0:4 * d])
    np.testing.assert_array_equal(b4[o4["Vc"]:o4["Vc"] + 4 * d], hi[o2["Vc"]:o2["Vc"] + 4 * d])
    np.testing.assert_array_equal(b4[o4["Vc"] + 4 * d:o4["Vc"] + 8 * d], lo[o2["Vc"]:o2["Vc"] + 4 * d])
    np.testing.assert_array_equal(b4[o4["Ksz"]:o4["Ksz"] + 2 * d], hi[o2["Ksz"]:o2["Ksz"] + 2 * d])
    np.testing.assert_array_equal(b4[o4["Vs"]:], hi[o2["Vs"]:])
