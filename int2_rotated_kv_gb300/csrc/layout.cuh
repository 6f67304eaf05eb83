// Page formats of the mixed-precision cache (device side).
//
// The pages ask for a paged KV cache that keeps sink and recent tokens in BF16
// and the rotated, clipped middle history in INT2 ("Technical Summary: OSCAR
// ...", section 2.2B), and fix no byte layout.  The layout below is chosen so
// that one 16-byte shared-memory load per lane yields, for a page of 16 tokens,
// exactly the mma.m16n8k16 A-operand fragments the decode kernel feeds to the
// tensor cores (PTX ISA fragment layout: lane = 4*gid + tig, register r holds
// rows gid + 8*(r&1), columns 2*tig + 8*(r>>1) + {0,1}).
//
// d = head dim (64/128), ng = d/32 groups, t = slot in page, j = channel.
// INT2 block (12*d bytes): Kc [0,4d) | Ksz [4d,6d) | Vc [6d,10d) | Vs [10d,11d)
//   | Vz [11d,12d).  Codes are 2-bit fields of 32-bit words word = L*(d/32)+m
//   at bit 16*e + 4*s + 2*i:
//   key   (t, j): kk=j/16, h=(j/8)&1, tig=(j/2)&3, e=j&1, gid=t&7, th=t/8,
//                 L=4*gid+tig, m=kk/2, i=kk&1, s=2*th+h
//   value (t, j): mt=j/16, ch=(j/8)&1, gid=j&7, tig=(t/2)&3, e=t&1, th=t/8,
//                 L=4*gid+tig, m=mt/2, i=mt&1, s=ch+2*th
//   Ksz: 32-bit (s16 | z16 << 16) at index t*ng + grp.
//   Vs / Vz: fp16 at index ((tig*2 + th)*ng + grp)*2 + e, t = 8*th + 2*tig + e.
// BF16 block (64*d bytes): keys then values, 32-bit words of two bf16:
//   key   (t, j): word (kk*32 + L)*4 + r, r = th + 2*h
//   value (t, j): word (mt*32 + L)*4 + r, r = ch + 2*th;   element 2*word + e.
// Word m of a lane's key codes covers k-steps 2m, 2m+1 (channels of group m);
// word m of its value codes covers channel tiles 2m, 2m+1 (group m).  Pair
// (s, i) sits at bits (4s+2i, 16+4s+2i), so (w >> 4s) & (0x00030003 << 2i) is
// a half2 whose halves are the two codes times 4^i, read as fp16 subnormals
// (code * 4^i * 2^-24): exact tensor-core operands without any conversion.
//
// INT4 variant (P = 2 planes): a 4-bit code c is kept as two 2-bit planes, the
// high bits c >> 2 in plane 0 and the low bits c & 3 in plane 1, each plane a
// code area in exactly the order above.  Block (20*d bytes): Kc plane 0 [0,4d)
// | Kc plane 1 [4d,8d) | Ksz [8d,10d) | Vc planes [10d,18d) | Vs [18d,19d) |
// Vz [19d,20d).  The decode kernel runs the INT2 fragment arithmetic on both
// planes and weighs the high plane by 4.
#pragma once

#include <stdint.h>

namespace oscar {

template <int D, int P = 1>
struct Fmt {
  static constexpr int kNG = D / 32;          // groups per token
  static constexpr int kNK = D / 16;          // 16-channel k-steps / tiles
  static constexpr int kWords = D / 32;       // code words per lane
  static constexpr int kPlane = 4 * D;        // bytes of one 2-bit code plane
  static constexpr int kInt2Block = (8 * P + 4) * D;   // code block (12d INT2, 20d INT4)
  static constexpr int kKc = 0;               // key plane q at kKc + q * kPlane
  static constexpr int kKsz = 4 * D * P;
  static constexpr int kVc = 4 * D * P + 2 * D;   // value plane q at kVc + q * kPlane
  static constexpr int kVs = 8 * D * P + 2 * D;
  static constexpr int kVz = 8 * D * P + 3 * D;
  static constexpr int kBf16Block = 64 * D;   // bytes
  static constexpr int kBf16V = 32 * D;       // byte offset of the value half
};

// Byte of a key code block that holds channels {16(2m+i) + 8h + 2tig + e}
// (h, i in {0,1}) of token t, and the bit of (h, i) inside it is 4h + 2i.
template <int D>
__device__ __forceinline__ int key_byte(int t, int tig, int m, int e) {
  const int lane = 4 * (t & 7) + tig;
  return 4 * (lane * Fmt<D>::kWords + m) + 2 * e + (t >> 3);
}

// Byte of a value code block holding channels {16(2m+i) + 8ch + gid} (ch, i in
// {0,1}) of token t; bit of (ch, i) is 4ch + 2i.
template <int D>
__device__ __forceinline__ int value_byte(int t, int gid, int m) {
  const int lane = 4 * gid + ((t >> 1) & 3);
  return 4 * (lane * Fmt<D>::kWords + m) + 2 * (t & 1) + (t >> 3);
}

template <int D>
__device__ __forceinline__ int vsz_index(int t, int grp) {
  return ((((t >> 1) & 3) * 2 + (t >> 3)) * Fmt<D>::kNG + grp) * 2 + (t & 1);
}

// bf16 element index (inside the key or value half of a BF16 block)
__device__ __forceinline__ int bf16_key_elem(int t, int j) {
  const int kk = j >> 4, h = (j >> 3) & 1, tig = (j >> 1) & 3, e = j & 1;
  const int lane = 4 * (t & 7) + tig, r = (t >> 3) + 2 * h;
  return 2 * ((kk * 32 + lane) * 4 + r) + e;
}

__device__ __forceinline__ int bf16_value_elem(int t, int j) {
  const int mt = j >> 4, ch = (j >> 3) & 1, gid = j & 7;
  const int tig = (t >> 1) & 3, e = t & 1, th = t >> 3;
  const int lane = 4 * gid + tig, r = ch + 2 * th;
  return 2 * ((mt * 32 + lane) * 4 + r) + e;
}

}  // namespace oscar
