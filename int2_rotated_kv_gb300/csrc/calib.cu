// Calibration on the device for one layer: the covariance targets C_Q and C_S
// and the clipping thresholds, for long calibration sets and many layers.
//   [Summary 2.1]   query-aware key target C_Q, score-aware value target C_S;
//   [Summary 2.2A]  step 1 (accumulate the covariances over calibration data),
//                   step 4 (clip = a high percentile of |x R| per layer).
// The eigendecomposition and R = U H P_br stay on the host (oscar_build_rotation),
// which takes the fp64 C these kernels produce.
//
// Kernels
//   gram_kernel            partial X^T X of one 64x64 block of C over a token chunk
//                          (mma.sync bf16, fp32 accumulators flushed every 128 rows
//                          into compensated (hi, lo) fp32 pairs)
//   gram_reduce_kernel     fixed-order sum of the chunk partials, then fp64 and 1/(nG)
//   calib_attention_kernel causal softmax(q k^T / sqrt(d)) v per query head, the
//                          probabilities split into a bf16 (hi, lo) pair for P V; the
//                          output O is stored as a bf16 (hi, lo) pair for the Gram
//   rotate_abs_kernel      |x R| in fp32 (sequential FMA over the input channel)
//   radix_hist_kernel,     exact selection of the order statistics the linear
//   radix_digit_kernel,    percentile interpolates, three 11/11/10-bit radix passes
//   next_above_kernel,     on the fp32 bit patterns (monotone for values >= 0)
//   clip_finish_kernel
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "common.cuh"
#include "oscar.h"

namespace oscar {
namespace calib {

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  // src-size 0 writes 16 zero bytes and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// Row-major tile of rows of `row_bytes` bytes, 16-byte chunks XOR-swizzled by
// the row's low three bits: the eight rows an ldmatrix reads at one logical
// chunk land in eight different bank groups.
__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
  return static_cast<uint32_t>(row * row_bytes + ((chunk ^ (row & 7)) << 4));
}

// Knuth's TwoSum: hi + lo accumulates a exactly up to the final rounding of lo.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float a) {
  const float s = __fadd_rn(hi, a);
  const float bp = __fsub_rn(s, hi);
  const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(a, bp));
  hi = s;
  lo = __fadd_rn(lo, e);
}

// ------------------------------------------------------------------ Gram X^T X

constexpr int kGramRows = 64;     // rows per pipeline stage
constexpr int kGramStages = 3;
constexpr int kGramFlush = 2;     // stages between compensated flushes (128 rows)
constexpr int kGramThreads = 128; // 4 warps, each a 32x32 piece of a 64x64 block
constexpr int kSlab = 64;         // channels per block side
constexpr int kSlabBytes = kGramRows * kSlab * 2;   // 8 KB: 64 rows x 64 bf16

struct GramParams {
  const __nv_bfloat16* x[2];   // pieces summed into one value: [n][heads][d] bf16
  int heads;                   // heads of x per token
  int G;                       // heads [h*G, h*G+G) pool into KV head h
  int d;
  int64_t n;
  int64_t tokens_per_chunk;
  int chunks;
  int blocks;                  // upper-triangular 64x64 blocks of C: nb(nb+1)/2
  float2* part;                // [hkv][chunks][blocks][64][64] (hi, lo)
};

__host__ __device__ inline void block_coords(int blk, int nb, int& bi, int& bj) {
  // enumerate bi <= bj row by row
  int r = 0, base = 0;
  while (blk >= base + (nb - r)) {
    base += nb - r;
    ++r;
  }
  bi = r;
  bj = r + (blk - base);
}

__device__ __forceinline__ int block_index(int bi, int bj, int nb) {
  return bi * nb - bi * (bi - 1) / 2 + (bj - bi);
}

template <int kPieces>
__global__ void __launch_bounds__(kGramThreads) gram_kernel(GramParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int chunk = blockIdx.x, h = blockIdx.y, blk = blockIdx.z;
  const int nb = p.d / kSlab;
  int bi, bj;
  block_coords(blk, nb, bi, bj);
  const bool diag = bi == bj;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wi = warp >> 1, wj = warp & 1;

  const int64_t n0 = static_cast<int64_t>(chunk) * p.tokens_per_chunk;
  const int64_t n1 = n0 + p.tokens_per_chunk < p.n ? n0 + p.tokens_per_chunk : p.n;
  const int64_t rows = n1 > n0 ? (n1 - n0) * p.G : 0;
  const int stages = static_cast<int>((rows + kGramRows - 1) / kGramRows);

  // stage buffer layout: [stage][piece][slab I, slab J]
  auto slab = [&](int buf, int piece, int side) -> unsigned char* {
    return smem + ((buf * kPieces + piece) * 2 + side) * kSlabBytes;
  };

  auto load = [&](int st) {
    const int buf = st % kGramStages;
    constexpr int kChunks = kGramRows * (kSlab / 8);   // 16-byte chunks per slab
    for (int c = threadIdx.x; c < kChunks; c += kGramThreads) {
      const int r = c >> 3, ch = c & 7;
      const int64_t R = static_cast<int64_t>(st) * kGramRows + r;
      const bool ok = R < rows;
      const int64_t tok = ok ? n0 + R / p.G : 0;
      const int g = ok ? static_cast<int>(R % p.G) : 0;
      const size_t row_off = (static_cast<size_t>(tok) * p.heads + static_cast<size_t>(h) * p.G + g) *
                             static_cast<size_t>(p.d);
#pragma unroll
      for (int piece = 0; piece < kPieces; ++piece) {
        const __nv_bfloat16* src = p.x[piece];
        cp_async16(slab(buf, piece, 0) + swz(r, ch, kSlab * 2),
                   ok ? src + row_off + bi * kSlab + ch * 8 : src, ok);
        if (!diag)
          cp_async16(slab(buf, piece, 1) + swz(r, ch, kSlab * 2),
                     ok ? src + row_off + bj * kSlab + ch * 8 : src, ok);
      }
    }
  };

  float acc[2][4][4], hi[2][4][4], lo[2][4][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][b][e] = hi[a][b][e] = lo[a][b][e] = 0.f;

#pragma unroll
  for (int s = 0; s < kGramStages - 1; ++s) {
    if (s < stages) load(s);
    cp_async_commit();
  }

  const int mi = lane >> 3, rr = lane & 7;
  for (int st = 0; st < stages; ++st) {
    cp_async_wait<kGramStages - 2>();
    __syncthreads();
    if (st + kGramStages - 1 < stages) load(st + kGramStages - 1);
    cp_async_commit();
    const int buf = st % kGramStages;
#pragma unroll
    for (int ks = 0; ks < kGramRows / 16; ++ks) {
      const int r0 = ks * 16;
      uint32_t A[kPieces][2][4], B[kPieces][4][2];
#pragma unroll
      for (int piece = 0; piece < kPieces; ++piece) {
        const unsigned char* sI = slab(buf, piece, 0);
        const unsigned char* sJ = slab(buf, piece, diag ? 0 : 1);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          // A = X^T: m = channel (32 wi + 16 a ..), k = row; transposed 8x8 loads
          const int row = r0 + rr + 8 * (mi >> 1);
          const int ch = ((32 * wi + 16 * a) >> 3) + (mi & 1);
          ldsm_x4_t(A[piece][a], smem_u32(sI + swz(row, ch, kSlab * 2)));
        }
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          // B = X: k = row, n = channel (32 wj + 16 bb ..), two 8-channel blocks
          const int row = r0 + rr + 8 * (mi & 1);
          const int ch = ((32 * wj + 16 * bb) >> 3) + (mi >> 1);
          uint32_t t[4];
          ldsm_x4_t(t, smem_u32(sJ + swz(row, ch, kSlab * 2)));
          B[piece][2 * bb][0] = t[0];
          B[piece][2 * bb][1] = t[1];
          B[piece][2 * bb + 1][0] = t[2];
          B[piece][2 * bb + 1][1] = t[3];
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          mma_bf16(acc[a][b], A[0][a][0], A[0][a][1], A[0][a][2], A[0][a][3], B[0][b][0], B[0][b][1]);
          if (kPieces == 2) {
            // (hi + lo)^T (hi + lo) without the lo^T lo term (2^-16 below the rest)
            mma_bf16(acc[a][b], A[0][a][0], A[0][a][1], A[0][a][2], A[0][a][3],
                     B[kPieces - 1][b][0], B[kPieces - 1][b][1]);
            mma_bf16(acc[a][b], A[kPieces - 1][a][0], A[kPieces - 1][a][1], A[kPieces - 1][a][2],
                     A[kPieces - 1][a][3], B[0][b][0], B[0][b][1]);
          }
        }
    }
    if ((st + 1) % kGramFlush == 0 || st == stages - 1) {
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            two_sum_acc(hi[a][b][e], lo[a][b][e], acc[a][b][e]);
            acc[a][b][e] = 0.f;
          }
    }
  }
  cp_async_wait<0>();

  float2* out = p.part + ((static_cast<size_t>(h) * p.chunks + chunk) * p.blocks + blk) * kSlab * kSlab;
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 32 * wi + 16 * a + (lane >> 2) + 8 * (e >> 1);
        const int j = 32 * wj + 8 * b + 2 * (lane & 3) + (e & 1);
        out[i * kSlab + j] = make_float2(hi[a][b][e], lo[a][b][e]);
      }
}

// C[h][i][j] = (sum over chunks of the partials) / (n G), fp64 at the end.
__global__ void gram_reduce_kernel(const float2* __restrict__ part, int chunks, int blocks, int d,
                                   double inv, double* __restrict__ c) {
  const int h = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= d * d) return;
  const int i = idx / d, j = idx % d;
  const int nb = d / kSlab;
  int bi = i / kSlab, bj = j / kSlab, ii = i % kSlab, jj = j % kSlab;
  if (bi > bj) {   // lower blocks are the transposes of upper ones
    const int t = bi; bi = bj; bj = t;
    const int u = ii; ii = jj; jj = u;
  }
  const int blk = block_index(bi, bj, nb);
  float s_hi = 0.f, s_lo = 0.f;
  for (int ch = 0; ch < chunks; ++ch) {
    const float2 v = part[((static_cast<size_t>(h) * chunks + ch) * blocks + blk) * kSlab * kSlab +
                          ii * kSlab + jj];
    two_sum_acc(s_hi, s_lo, v.x);
    s_lo = __fadd_rn(s_lo, v.y);
  }
  c[(static_cast<size_t>(h) * d + i) * d + j] =
      (static_cast<double>(s_hi) + static_cast<double>(s_lo)) * inv;
}

// ------------------------------------------------- causal calibration attention

constexpr int kAttnRows = 128;   // query rows per CTA: 8 warps x 16
constexpr int kAttnKeys = 64;    // keys per tile
constexpr int kAttnThreads = 256;

template <int D>
struct AttnCfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kQBytes = kAttnRows * kRowBytes;
  static constexpr int kKVBytes = kAttnKeys * kRowBytes;
  static constexpr int kBytes = kQBytes + 4 * kKVBytes;   // Q + two stages of (K, V)
};

struct AttnParams {
  const __nv_bfloat16* q;   // [n][hq][D]
  const __nv_bfloat16* k;   // [n][hkv][D]
  const __nv_bfloat16* v;   // [n][hkv][D]
  __nv_bfloat16* o_hi;      // [n][hq][D]
  __nv_bfloat16* o_lo;      // [n][hq][D]
  int hq, hkv, G;
  int64_t n;
  float scale_log2;         // log2(e) / sqrt(D)
};

// bf16 pair (hi, lo) of two floats: hi = bf16(x), lo = bf16(x - hi).
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf162(x0, x1);
  lo = pack_bf162(x0 - bf16_lo_value(hi), x1 - bf16_hi_value(hi));
}

// One CTA: 128 query rows = 128/G consecutive tokens x the G query heads of KV
// head blockIdx.y (row r <-> token t0 + r / G, head h G + r % G).  Tiles with
// the most keys are issued first.
template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) calib_attention_kernel(AttnParams p) {
  using C = AttnCfg<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* sq = smem;
  const int h = blockIdx.y;
  const int TB = kAttnRows / p.G;
  const int64_t t0 = static_cast<int64_t>(gridDim.x - 1 - blockIdx.x) * TB;
  const int64_t t_end = t0 + TB < p.n ? t0 + TB : p.n;
  const int ntiles = static_cast<int>((t_end - 1) / kAttnKeys) + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int c = threadIdx.x; c < kAttnRows * (D / 8); c += kAttnThreads) {
    const int r = c / (D / 8), ch = c % (D / 8);
    const int64_t t = t0 + r / p.G;
    const int g = r % p.G;
    const bool ok = t < p.n;
    const size_t off = (static_cast<size_t>(t) * p.hq + static_cast<size_t>(h) * p.G + g) * D + ch * 8;
    cp_async16(sq + swz(r, ch, C::kRowBytes), ok ? p.q + off : p.q, ok);
  }
  auto kbuf = [&](int b) { return smem + C::kQBytes + b * 2 * C::kKVBytes; };
  auto vbuf = [&](int b) { return smem + C::kQBytes + b * 2 * C::kKVBytes + C::kKVBytes; };
  auto load_kv = [&](int kt, int b) {
    for (int c = threadIdx.x; c < kAttnKeys * (D / 8); c += kAttnThreads) {
      const int r = c / (D / 8), ch = c % (D / 8);
      const int64_t j = static_cast<int64_t>(kt) * kAttnKeys + r;
      const bool ok = j < p.n;
      const size_t off = (static_cast<size_t>(j) * p.hkv + h) * D + ch * 8;
      cp_async16(kbuf(b) + swz(r, ch, C::kRowBytes), ok ? p.k + off : p.k, ok);
      cp_async16(vbuf(b) + swz(r, ch, C::kRowBytes), ok ? p.v + off : p.v, ok);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  const int ra = 16 * warp + (lane >> 2);   // this thread's rows ra and ra + 8
  const int64_t ta = t0 + ra / p.G;
  const int64_t tb = t0 + (ra + 8) / p.G;
  const int64_t tw_min = t0 + (16 * warp) / p.G;
  const int64_t tw_max = t0 + (16 * warp + 15) / p.G;

  uint32_t qf[D / 16][4];
  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  for (int kt = 0; kt < ntiles; ++kt) {
    if (kt + 1 < ntiles) load_kv(kt + 1, (kt + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int row = 16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1);
        ldsm_x4(qf[ks], smem_u32(sq + swz(row, 2 * ks + (lane >> 4), C::kRowBytes)));
      }
    }
    const int64_t kbase = static_cast<int64_t>(kt) * kAttnKeys;
    if (kbase <= tw_max) {
      const unsigned char* kb = kbuf(kt & 1);
      const unsigned char* vb = vbuf(kt & 1);
      float s[8][4];
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ks += 2)
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
          uint32_t b[4];
          ldsm_x4(b, smem_u32(kb + swz(8 * nb + (lane & 7), 2 * ks + (lane >> 3), C::kRowBytes)));
          mma_bf16(s[nb], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b[0], b[1]);
          mma_bf16(s[nb], qf[ks + 1][0], qf[ks + 1][1], qf[ks + 1][2], qf[ks + 1][3], b[2], b[3]);
        }
      const bool mask = kbase + kAttnKeys - 1 > tw_min;
      float mx_a = m_a, mx_b = m_b;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = s[nb][e] * p.scale_log2;
          if (mask) {
            const int64_t key = kbase + 8 * nb + 2 * (lane & 3) + (e & 1);
            if (key > (e < 2 ? ta : tb)) x = -INFINITY;
          }
          s[nb][e] = x;
          if (e < 2) mx_a = fmaxf(mx_a, x);
          else mx_b = fmaxf(mx_b, x);
        }
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
      // tile 0 holds key 0, visible to every row, so the running maxima are finite
      const float corr_a = fast_exp2(m_a - mx_a), corr_b = fast_exp2(m_b - mx_b);
      m_a = mx_a;
      m_b = mx_b;
      float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        s[nb][0] = fast_exp2(s[nb][0] - mx_a);
        s[nb][1] = fast_exp2(s[nb][1] - mx_a);
        s[nb][2] = fast_exp2(s[nb][2] - mx_b);
        s[nb][3] = fast_exp2(s[nb][3] - mx_b);
        sum_a += s[nb][0] + s[nb][1];
        sum_b += s[nb][2] + s[nb][3];
      }
      l_a = l_a * corr_a + sum_a;
      l_b = l_b * corr_b + sum_b;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        o[i][0] *= corr_a;
        o[i][1] *= corr_a;
        o[i][2] *= corr_b;
        o[i][3] *= corr_b;
      }
#pragma unroll
      for (int kk = 0; kk < kAttnKeys / 16; ++kk) {
        uint32_t ah[4], al[4];
        split_pair(s[2 * kk][0], s[2 * kk][1], ah[0], al[0]);
        split_pair(s[2 * kk][2], s[2 * kk][3], ah[1], al[1]);
        split_pair(s[2 * kk + 1][0], s[2 * kk + 1][1], ah[2], al[2]);
        split_pair(s[2 * kk + 1][2], s[2 * kk + 1][3], ah[3], al[3]);
#pragma unroll
        for (int vc = 0; vc < D / 8; vc += 2) {
          uint32_t b[4];
          const int row = 16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1);
          ldsm_x4_t(b, smem_u32(vb + swz(row, vc + (lane >> 4), C::kRowBytes)));
          mma_bf16(o[vc], ah[0], ah[1], ah[2], ah[3], b[0], b[1]);
          mma_bf16(o[vc], al[0], al[1], al[2], al[3], b[0], b[1]);
          mma_bf16(o[vc + 1], ah[0], ah[1], ah[2], ah[3], b[2], b[3]);
          mma_bf16(o[vc + 1], al[0], al[1], al[2], al[3], b[2], b[3]);
        }
      }
    }
    __syncthreads();
  }

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  const float inv_a = 1.f / l_a, inv_b = 1.f / l_b;
  const int hq_a = h * p.G + ra % p.G, hq_b = h * p.G + (ra + 8) % p.G;
#pragma unroll
  for (int vc = 0; vc < D / 8; ++vc) {
    const int ch = 8 * vc + 2 * (lane & 3);
    if (ta < p.n) {
      uint32_t hw, lw;
      split_pair(o[vc][0] * inv_a, o[vc][1] * inv_a, hw, lw);
      const size_t off = (static_cast<size_t>(ta) * p.hq + hq_a) * D + ch;
      *reinterpret_cast<uint32_t*>(p.o_hi + off) = hw;
      *reinterpret_cast<uint32_t*>(p.o_lo + off) = lw;
    }
    if (tb < p.n) {
      uint32_t hw, lw;
      split_pair(o[vc][2] * inv_b, o[vc][3] * inv_b, hw, lw);
      const size_t off = (static_cast<size_t>(tb) * p.hq + hq_b) * D + ch;
      *reinterpret_cast<uint32_t*>(p.o_hi + off) = hw;
      *reinterpret_cast<uint32_t*>(p.o_lo + off) = lw;
    }
  }
}

// ----------------------------------------------------------- clip threshold

constexpr int kRotTokens = 64;
constexpr int kRotThreads = 256;
constexpr int kRadixBins = 2048;

struct SelectState {
  uint32_t prefix;      // bits of the selected value found so far
  uint32_t mask;        // which bits of prefix are known
  uint32_t eq_count;    // values in the last selected bin
  uint32_t next_bits;   // smallest value above the selection (atomicMin)
  uint64_t rank;        // rank still to be resolved inside the matching set
  uint64_t pad;
};

template <int D>
struct RotCfg {
  static constexpr int kXs = D + 1;   // padded token row: the two token groups of a warp hit different banks
  static constexpr int kBytes = (D * D + kRotTokens * kXs) * 4;
};

// |x R| for one (64-token tile, KV head): each thread 4 tokens x D/16 channels
// (channels tx, tx + 16, ...), y_j = sum_i x_i R_ij accumulated in order
// i = 0 .. D-1 with fp32 FMA.  Block
// (0, h) also resets head h's selection state.
template <int D>
__global__ void __launch_bounds__(kRotThreads) rotate_abs_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ r, int hkv, int64_t n,
    uint32_t* __restrict__ abs_bits, uint32_t* __restrict__ hist, SelectState* __restrict__ state,
    uint64_t rank_lo) {
  extern __shared__ __align__(16) float fsm[];
  float* rs = fsm;               // [D][D]
  float* xs = fsm + D * D;       // [64][D + 1]
  constexpr int kXs = RotCfg<D>::kXs;
  const int h = blockIdx.y;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kRotTokens;
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < kRadixBins; i += kRotThreads) hist[h * kRadixBins + i] = 0u;
    if (threadIdx.x == 0) {
      SelectState s{};
      s.next_bits = 0xffffffffu;
      s.rank = rank_lo;
      state[h] = s;
    }
  }
  const float4* r4 = reinterpret_cast<const float4*>(r + static_cast<size_t>(h) * D * D);
  for (int i = threadIdx.x; i < D * D / 4; i += kRotThreads) reinterpret_cast<float4*>(rs)[i] = r4[i];
  for (int i = threadIdx.x; i < kRotTokens * D / 2; i += kRotThreads) {
    const int tk = (2 * i) / D, c = (2 * i) % D;
    const int64_t t = t0 + tk;
    float2 f = make_float2(0.f, 0.f);
    if (t < n) {
      const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(
          x + (static_cast<size_t>(t) * hkv + h) * D + c);
      f = __bfloat1622float2(b);
    }
    xs[tk * kXs + c] = f.x;
    xs[tk * kXs + c + 1] = f.y;
  }
  __syncthreads();
  constexpr int kC = D / 16;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float acc[4][kC];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < kC; ++c) acc[a][c] = 0.f;
  for (int i = 0; i < D; ++i) {
    float xv[4], rv[kC];
#pragma unroll
    for (int a = 0; a < 4; ++a) xv[a] = xs[(4 * ty + a) * kXs + i];
#pragma unroll
    for (int c = 0; c < kC; ++c) rv[c] = rs[i * D + c * 16 + tx];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < kC; ++c) acc[a][c] = fmaf(xv[a], rv[c], acc[a][c]);
  }
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int64_t t = t0 + 4 * ty + a;
    if (t >= n) continue;
    uint32_t* dst = abs_bits + static_cast<size_t>(h) * n * D + static_cast<size_t>(t) * D + tx;
#pragma unroll
    for (int c = 0; c < kC; ++c) dst[c * 16] = __float_as_uint(fabsf(acc[a][c]));
  }
}

// Histogram of the next digit over the values whose known bits match.
__global__ void radix_hist_kernel(const uint32_t* __restrict__ bits, int64_t m,
                                  const SelectState* __restrict__ state, uint32_t* __restrict__ hist,
                                  int shift, uint32_t digit_mask) {
  __shared__ uint32_t sh[kRadixBins];
  const int h = blockIdx.y;
  for (int i = threadIdx.x; i < kRadixBins; i += blockDim.x) sh[i] = 0u;
  __syncthreads();
  const uint32_t prefix = state[h].prefix, mask = state[h].mask;
  const uint32_t* v = bits + static_cast<size_t>(h) * m;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < m;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t b = v[i];
    if ((b & mask) == prefix) atomicAdd(&sh[(b >> shift) & digit_mask], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kRadixBins; i += blockDim.x)
    if (sh[i]) atomicAdd(&hist[h * kRadixBins + i], sh[i]);
}

// Picks the bin that holds the remaining rank, narrows the state, clears the
// histogram for the next pass.  One block of 256 threads per head, 8 bins each.
__global__ void __launch_bounds__(256) radix_digit_kernel(uint32_t* __restrict__ hist,
                                                          SelectState* __restrict__ state, int shift,
                                                          uint32_t digit_mask) {
  __shared__ uint64_t warp_tot[8];
  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SelectState s0 = state[h];   // read by every thread before the barrier below
  uint32_t* hh = hist + h * kRadixBins;
  uint32_t c[8];
  uint64_t local = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = hh[tid * 8 + i];
    local += c[i];
  }
  uint64_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint64_t before = incl - local;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  const uint64_t rank = s0.rank;
  if (rank >= before && rank < before + local) {
    uint64_t cum = before;
    for (int i = 0; i < 8; ++i) {
      if (rank < cum + c[i]) {
        const uint32_t digit = static_cast<uint32_t>(tid * 8 + i) & digit_mask;
        SelectState s = s0;
        s.prefix |= digit << shift;
        s.mask |= digit_mask << shift;
        s.rank = rank - cum;
        s.eq_count = c[i];
        state[h] = s;
        break;
      }
      cum += c[i];
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) hh[tid * 8 + i] = 0u;
}

// Smallest value strictly above the selected one, needed only when the selected
// value's rank is the last among its equals.
__global__ void next_above_kernel(const uint32_t* __restrict__ bits, int64_t m,
                                  SelectState* __restrict__ state) {
  __shared__ uint32_t warp_min[32];
  const int h = blockIdx.y;
  const SelectState s = state[h];
  if (s.rank + 1 < s.eq_count) return;   // the next order statistic equals this one
  const uint32_t sel = s.prefix;
  uint32_t best = 0xffffffffu;
  const uint32_t* v = bits + static_cast<size_t>(h) * m;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < m;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t b = v[i];
    if (b > sel && b < best) best = b;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) warp_min[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t b = 0xffffffffu;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = min(b, warp_min[w]);
    if (b != 0xffffffffu) atomicMin(&state[h].next_bits, b);
  }
}

// clip = x_lo + frac (x_hi - x_lo) in fp64, rounded to fp32.
__global__ void clip_finish_kernel(const SelectState* __restrict__ state, int hkv, double frac,
                                   float* __restrict__ clip) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= hkv) return;
  const SelectState s = state[h];
  const double xlo = static_cast<double>(__uint_as_float(s.prefix));
  double xhi = xlo;
  if (s.rank + 1 >= s.eq_count && s.next_bits != 0xffffffffu)
    xhi = static_cast<double>(__uint_as_float(s.next_bits));
  clip[h] = static_cast<float>(xlo + frac * (xhi - xlo));
}

// ------------------------------------------------------------ host planning

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct GramPlan {
  int chunks = 0, blocks = 0;
  int64_t tokens_per_chunk = 0;
  size_t bytes = 0;
};

inline GramPlan plan_gram(int hkv, int G, int d, int64_t n) {
  GramPlan g;
  const int nb = d / kSlab;
  g.blocks = nb * (nb + 1) / 2;
  // about two resident CTAs per SM in one wave, and at least 512 rows per chunk
  int64_t chunks = std::max<int64_t>(1, 2LL * oscar_host::sm_count() / (hkv * g.blocks));
  const int64_t max_chunks = std::max<int64_t>(1, (n * G + 511) / 512);
  chunks = std::min(chunks, max_chunks);
  g.tokens_per_chunk = (n + chunks - 1) / chunks;
  g.chunks = static_cast<int>((n + g.tokens_per_chunk - 1) / g.tokens_per_chunk);
  g.bytes = align_up(static_cast<size_t>(hkv) * g.chunks * g.blocks * kSlab * kSlab * sizeof(float2));
  return g;
}

struct ClipPlan {
  size_t abs_off = 0, hist_off = 0, state_off = 0, total = 0;
};

inline ClipPlan plan_clip(int hkv, int d, int64_t n) {
  ClipPlan c;
  c.abs_off = 0;
  c.hist_off = align_up(static_cast<size_t>(hkv) * n * d * 4);
  c.state_off = c.hist_off + align_up(static_cast<size_t>(hkv) * kRadixBins * 4);
  c.total = c.state_off + align_up(static_cast<size_t>(hkv) * sizeof(SelectState));
  return c;
}

inline bool g_ok(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

inline oscar_status check_shape(int hkv, int hq, int d, int64_t n) {
  if (hkv < 1 || hq < 1 || n < 1) return OSCAR_ERR_INVALID_ARG;
  if (hq % hkv) return OSCAR_ERR_INVALID_ARG;
  if (!oscar_host::head_dim_ok(d) || !g_ok(hq / hkv)) return OSCAR_ERR_UNSUPPORTED;
  if (n > (int64_t(1) << 24)) return OSCAR_ERR_UNSUPPORTED;   // 32-bit histogram counts
  return OSCAR_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

inline oscar_status launched() {
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

template <int kPieces>
oscar_status run_gram(const __nv_bfloat16* x0, const __nv_bfloat16* x1, int heads, int hkv, int d,
                      int64_t n, const GramPlan& g, void* part, double* c_out, cudaStream_t st) {
  GramParams p{};
  p.x[0] = x0;
  p.x[1] = x1;
  p.heads = heads;
  p.G = heads / hkv;
  p.d = d;
  p.n = n;
  p.tokens_per_chunk = g.tokens_per_chunk;
  p.chunks = g.chunks;
  p.blocks = g.blocks;
  p.part = static_cast<float2*>(part);
  const int smem = kGramStages * kPieces * 2 * kSlabBytes;
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(gram_kernel<kPieces>), smem))
    return OSCAR_ERR_CUDA;
  gram_kernel<kPieces><<<dim3(g.chunks, hkv, g.blocks), kGramThreads, smem, st>>>(p);
  if (launched() != OSCAR_OK) return OSCAR_ERR_CUDA;
  const double inv = 1.0 / (static_cast<double>(n) * p.G);
  gram_reduce_kernel<<<dim3((d * d + 255) / 256, hkv), 256, 0, st>>>(p.part, g.chunks, g.blocks, d,
                                                                     inv, c_out);
  return launched();
}

template <int D>
oscar_status run_attention(const AttnParams& p, cudaStream_t st) {
  using C = AttnCfg<D>;
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(calib_attention_kernel<D>), C::kBytes))
    return OSCAR_ERR_CUDA;
  const int TB = kAttnRows / p.G;
  const int64_t tiles = (p.n + TB - 1) / TB;
  if (tiles > 0x7fffffff) return OSCAR_ERR_UNSUPPORTED;
  calib_attention_kernel<D><<<dim3(static_cast<unsigned>(tiles), p.hkv), kAttnThreads, C::kBytes, st>>>(p);
  return launched();
}

template <int D>
oscar_status run_clip(const __nv_bfloat16* x, const float* r, int hkv, int64_t n, double percentile,
                      float* clip_out, unsigned char* ws, cudaStream_t st) {
  const ClipPlan cp = plan_clip(hkv, D, n);
  uint32_t* abs_bits = reinterpret_cast<uint32_t*>(ws + cp.abs_off);
  uint32_t* hist = reinterpret_cast<uint32_t*>(ws + cp.hist_off);
  SelectState* state = reinterpret_cast<SelectState*>(ws + cp.state_off);
  // linear interpolation between order statistics lo and lo + 1 (0-based) of
  // the m = n d values, h = (m - 1) p / 100
  const int64_t m = n * D;
  const double hpos = (static_cast<double>(m) - 1.0) * percentile / 100.0;
  int64_t lo = static_cast<int64_t>(std::floor(hpos));
  double frac = hpos - static_cast<double>(lo);
  if (lo >= m - 1) {
    lo = m - 1;
    frac = 0.0;
  }
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(rotate_abs_kernel<D>), RotCfg<D>::kBytes))
    return OSCAR_ERR_CUDA;
  const int64_t tiles = (n + kRotTokens - 1) / kRotTokens;
  rotate_abs_kernel<D><<<dim3(static_cast<unsigned>(tiles), hkv), kRotThreads, RotCfg<D>::kBytes, st>>>(
      x, r, hkv, n, abs_bits, hist, state, static_cast<uint64_t>(lo));
  if (launched() != OSCAR_OK) return OSCAR_ERR_CUDA;
  const int per_head = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>((m + 4095) / 4096, 2LL * oscar_host::sm_count() / hkv + 1)));
  const int shifts[3] = {21, 10, 0};
  const uint32_t masks[3] = {0x7ffu, 0x7ffu, 0x3ffu};
  for (int pass = 0; pass < 3; ++pass) {
    radix_hist_kernel<<<dim3(per_head, hkv), 256, 0, st>>>(abs_bits, m, state, hist, shifts[pass],
                                                          masks[pass]);
    radix_digit_kernel<<<hkv, 256, 0, st>>>(hist, state, shifts[pass], masks[pass]);
  }
  next_above_kernel<<<dim3(per_head, hkv), 256, 0, st>>>(abs_bits, m, state);
  clip_finish_kernel<<<(hkv + 127) / 128, 128, 0, st>>>(state, hkv, frac, clip_out);
  return launched();
}

}  // namespace calib
}  // namespace oscar

using namespace oscar::calib;

extern "C" {

size_t oscar_calibration_workspace_size(int32_t num_kv_heads, int32_t num_q_heads, int32_t d,
                                        int64_t n) {
  if (check_shape(num_kv_heads, num_q_heads, d, n) != OSCAR_OK) return 0;
  const int G = num_q_heads / num_kv_heads;
  const GramPlan g = plan_gram(num_kv_heads, G, d, n);
  const size_t o_bytes = align_up(static_cast<size_t>(n) * num_q_heads * d * 2);
  const size_t score = 2 * o_bytes + g.bytes;
  const size_t clip = plan_clip(num_kv_heads, d, n).total;
  return std::max(score, clip);
}

oscar_status oscar_query_covariance_device(int32_t num_kv_heads, int32_t num_q_heads, int32_t d,
                                           int64_t n, const void* q, double* c_out,
                                           void* workspace, size_t workspace_bytes, void* stream) {
  const oscar_status s = check_shape(num_kv_heads, num_q_heads, d, n);
  if (s != OSCAR_OK) return s;
  if (!q || !c_out || !workspace || !aligned16(q) || !aligned16(workspace))
    return OSCAR_ERR_INVALID_ARG;
  const GramPlan g = plan_gram(num_kv_heads, num_q_heads / num_kv_heads, d, n);
  if (workspace_bytes < g.bytes) return OSCAR_ERR_WORKSPACE;
  const auto* x = static_cast<const __nv_bfloat16*>(q);
  return run_gram<1>(x, x, num_q_heads, num_kv_heads, d, n, g, workspace, c_out,
                     static_cast<cudaStream_t>(stream));
}

oscar_status oscar_score_covariance_device(int32_t num_kv_heads, int32_t num_q_heads, int32_t d,
                                           int64_t n, const void* q, const void* k, const void* v,
                                           double* c_out, void* workspace, size_t workspace_bytes,
                                           void* stream) {
  const oscar_status s = check_shape(num_kv_heads, num_q_heads, d, n);
  if (s != OSCAR_OK) return s;
  if (!q || !k || !v || !c_out || !workspace || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(workspace))
    return OSCAR_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  const GramPlan g = plan_gram(num_kv_heads, G, d, n);
  const size_t o_bytes = align_up(static_cast<size_t>(n) * num_q_heads * d * 2);
  if (workspace_bytes < 2 * o_bytes + g.bytes) return OSCAR_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  AttnParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o_hi = reinterpret_cast<__nv_bfloat16*>(ws);
  p.o_lo = reinterpret_cast<__nv_bfloat16*>(ws + o_bytes);
  p.hq = num_q_heads;
  p.hkv = num_kv_heads;
  p.G = G;
  p.n = n;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const oscar_status a = d == 128 ? run_attention<128>(p, st) : run_attention<64>(p, st);
  if (a != OSCAR_OK) return a;
  return run_gram<2>(p.o_hi, p.o_lo, num_q_heads, num_kv_heads, d, n, g, ws + 2 * o_bytes, c_out, st);
}

oscar_status oscar_clip_threshold_device(int32_t num_kv_heads, int32_t d, int64_t n, const void* x,
                                         const float* r, double percentile, float* clip_out,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  const oscar_status s = check_shape(num_kv_heads, num_kv_heads, d, n);
  if (s != OSCAR_OK) return s;
  if (!x || !r || !clip_out || !workspace || !aligned16(x) || !aligned16(r) || !aligned16(workspace))
    return OSCAR_ERR_INVALID_ARG;
  if (!(percentile >= 0.0 && percentile <= 100.0)) return OSCAR_ERR_INVALID_ARG;
  if (workspace_bytes < plan_clip(num_kv_heads, d, n).total) return OSCAR_ERR_WORKSPACE;
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return d == 128 ? run_clip<128>(xb, r, num_kv_heads, n, percentile, clip_out, ws, st)
                  : run_clip<64>(xb, r, num_kv_heads, n, percentile, clip_out, ws, st);
}

}  // extern "C"
