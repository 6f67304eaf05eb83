// Pieces of the decode step's append shared by the append kernel and the
// single-launch decode step: the rotary embedding of the step's new query and
// key, and the clip / quantise / pack of one 32-channel group of the token that
// leaves the recent window ("Technical Summary: OSCAR ...", section 2.2B: the
// history is stored in INT2 after the fixed rotation and clipping).  Both
// callers run exactly this arithmetic, so their pool bytes are identical.
#pragma once

#include "common.cuh"
#include "layout.cuh"

namespace oscar {

// cos and sin of the rotary angle m * f: the product and its reduction to
// [-pi, pi] in fp64, then sincosf.
__device__ __forceinline__ void rope_cs(int m, double f, float& c, float& s) {
  double a = static_cast<double>(m) * f;
  a -= 6.283185307179586 * rint(a * 0.15915494309189535);
  sincosf(static_cast<float>(a), &s, &c);
}

// Rotary embedding of channel j of a head vector x (pairs j, j +- D/2), fp32,
// rounded to bf16 (the activation precision).
template <int D>
__device__ __forceinline__ float rope_bf16(float xj, float xpartner, int j, int m,
                                           const double* inv_freq) {
  float c, s;
  rope_cs(m, inv_freq[j % (D / 2)], c, s);
  const float y = j < D / 2 ? __fsub_rn(__fmul_rn(xj, c), __fmul_rn(xpartner, s))
                            : __fadd_rn(__fmul_rn(xj, c), __fmul_rn(xpartner, s));
  return __bfloat162float(__float2bfloat16_rn(y));
}

// One warp, lane j holding the rotated value y of channel 32*grp + j of the
// token that leaves the window: a group with a non-finite value becomes a zero
// group (s = z = 0, codes 0; OSCAR_DEVERR_NONFINITE), else clip, group range,
// s16 = fp16((max - min)/levels), z16 = fp16(min), code = rint((y_c - z16)/s16)
// clamped, each step rounded in fp32 as written; the codes and (s, z) are
// written into slot `slot` of the code block `blk` (kv 0: keys, 1: values).
// cs: 32 bytes of shared memory owned by the warp.
template <int D, int P>
__device__ __forceinline__ void append_group(float y, float clip, int lane, int grp, int kv,
                                             int slot, uint8_t* blk, uint8_t* cs,
                                             int32_t* status) {
  using F = Fmt<D, P>;
  constexpr int NG = D / 32;
  constexpr float kLevels = P == 2 ? 15.f : 3.f;   // largest code: INT4 variant / INT2
  constexpr int kMaxCode = P == 2 ? 15 : 3;
  if (__any_sync(0xffffffffu, !isfinite(y))) {   // stored as a zero group
    if (lane == 0 && status) atomicOr(status, OSCAR_DEVERR_NONFINITE);
    y = 0.f;
  }
  const float yc = fminf(fmaxf(y, -clip), clip);
  const float mn = warp_min(yc);
  const float mx = warp_max(yc);
  const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), kLevels));
  const __half z16 = __float2half_rn(mn);
  const float sf = __half2float(s16);
  const float zf = __half2float(z16);
  int code = 0;
  if (sf != 0.f) code = min(max(__float2int_rn(__fdiv_rn(__fsub_rn(yc, zf), sf)), 0), kMaxCode);
  cs[lane] = static_cast<uint8_t>(code);
  __syncwarp();
  if (lane < 8 * P) {   // 8 code bytes of this group per plane; plane 0 = highest bits
    const int pl = lane >> 3, lb = lane & 7, shift = 2 * (P - 1 - pl);
    uint32_t byte = 0;
    if (kv == 0) {
      const int tig = lb >> 1, e = lb & 1;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int i = 0; i < 2; ++i)
          byte |= ((static_cast<uint32_t>(cs[16 * i + 8 * hh + 2 * tig + e]) >> shift) & 3u)
                  << (4 * hh + 2 * i);
      blk[F::kKc + pl * F::kPlane + key_byte<D>(slot, tig, grp, e)] = static_cast<uint8_t>(byte);
    } else {
      const int gid = lb;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int i = 0; i < 2; ++i)
          byte |= ((static_cast<uint32_t>(cs[16 * i + 8 * ch + gid]) >> shift) & 3u)
                  << (4 * ch + 2 * i);
      blk[F::kVc + pl * F::kPlane + value_byte<D>(slot, gid, grp)] = static_cast<uint8_t>(byte);
    }
  } else if (lane == 8 * P) {
    const uint32_t sz = static_cast<uint32_t>(__half_as_ushort(s16)) |
                        (static_cast<uint32_t>(__half_as_ushort(z16)) << 16);
    if (kv == 0) {
      reinterpret_cast<uint32_t*>(blk + F::kKsz)[slot * NG + grp] = sz;
    } else {
      const int e = vsz_index<D>(slot, grp);
      reinterpret_cast<uint16_t*>(blk + F::kVs)[e] = static_cast<uint16_t>(sz & 0xffffu);
      reinterpret_cast<uint16_t*>(blk + F::kVz)[e] = static_cast<uint16_t>(sz >> 16);
    }
  }
  __syncwarp();
}

}  // namespace oscar
