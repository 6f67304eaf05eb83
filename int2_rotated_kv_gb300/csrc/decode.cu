// Split-K paged decode attention over the mixed BF16 / INT2 cache.
//
// "Technical Summary: OSCAR ...", section 2.2B ("Kernel Integration": one fused
// kernel unpacks, dequantises, inverse-rotates and attends over the INT2
// history, works with paged KV and prefix caching, and adds no memory
// traffic) and the arXiv abstract (custom INT2 attention kernel).
//
// Design for sm_103a.  Nothing is dequantised or inverse-rotated per token.
// The query is rotated once (q' = q R_K) and attention over INT2 tokens runs
// in the rotated basis; the INT2 part of the output is rotated back once
// (o R_V^T) in the combine step.  By associativity this equals attending over
// k~ = y_hat_K R_K^T and v~ = y_hat_V R_V^T.  With y_hat = code * s + z per
// group of 32 channels:
//   logit_t = scale * sum_grp ( s_t,grp * (c_t . q')_grp + z_t,grp * sum_grp q' )
//   o'     += p_t * s_t,grp * c_t   (+ p_t * z_t,grp broadcast over the group)
// so the tensor cores only ever see exact operands: 2-bit codes read as fp16
// subnormals straight out of the page bytes (no conversion), q' in fp16, and
// p or p*s in fp16; s and z are applied in fp32 around the MMAs.
//
// Kernels (one call = three launches chained with programmatic dependent
// launch, so each starts while its predecessor drains):
//   qrot_kernel     q' = q R_K per (sequence, KV head), fp32.
//   split_kernel    grid (split, KV head, sequence).  Each warp streams its
//                   pages through a private ring of shared-memory stages
//                   filled by bulk TMA copies (one copy per page-head block),
//                   runs m16n8k16 MMAs for q.K (token x query-head tiles) and
//                   p.V (channel x query-head tiles), and keeps an online
//                   softmax per query head.  The last split of a sequence
//                   handles the BF16 sink + recent tokens with raw q.
//   combine_kernel  log-sum-exp merge of the splits, out = (o_raw +
//                   o_rot R_V^T) / l, stored as bf16.
// The same split/combine pair with every page in BF16 is the baseline kernel.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <type_traits>
#include <utility>
#include <vector>

#include "common.cuh"
#include "layout.cuh"

namespace oscar {

constexpr int kDWarps = 8;
constexpr int kDThreads = 32 * kDWarps;
constexpr int kMaxCtaPages = 1024;

struct DecodeParams {
  int hkv, hq, G, sink, window, max_pages;
  // query heads per CTA: the MMA tiles hold 8, so G = 16 is served as two halves
  // of 8 query heads (each half reads the KV head's pages)
  int gq, halves;
  int64_t n_int2_pages, n_bf16_pages;
  const uint8_t* int2_pool;
  const uint8_t* bf16_pool;
  const int32_t* int2_pt;
  const int32_t* bf16_pt;
  const float* r_k;
  const float* r_v;
  const float* clip_k;
  const float* clip_v;
  int32_t* status;
  const uint16_t* q;
  uint16_t* out;
  const int32_t* seq_lens;
  int batch, max_len;
  int n_main;     // splits over the main region
  int pps;        // pages per main split
  int n_splits;   // partial slots per (sequence, query head)
  float* qrot;    // [B][Hq][D]
  float* part;    // [B][Hq][n_splits][D + 2]
  float scale_log2;
  int wait_first; // wait for the predecessor grid before reading any input
  // launched right after the step's append kernel (no rotation kernel between):
  // pages that kernel writes -- the INT2 page of the token leaving the window,
  // the BF16 page of the new token -- are copied only after griddepcontrol.wait
  int after_append;
  // several query rows per sequence: row b of the batch belongs to sequence
  // b / rows_per_seq and sees stored tokens 0 .. limits[b] only (null: decode)
  int rows_per_seq;
  const int32_t* limits;
  // rows of one sequence packed into the MMA tile's 8 query columns: a split
  // CTA serves rpu consecutive rows (rpu * gq <= 8; 1 for a decode), so those
  // rows share every page read; units = CTAs per (split, KV head slice)
  int rpu, units;
};

// ------------------------------------------------------------------ q R_K

template <int D>
__global__ void __launch_bounds__(1024) qrot_kernel(const DecodeParams p) {
  // the caller's earlier work (q, rotations, cache writes) is complete after the
  // wait; only then may the split kernel launch and prefetch pages
  pdl_wait();
  pdl_trigger();
  __shared__ float qs[8][D];
  __shared__ float partial[1024 / D][8][D];
  const int h = blockIdx.x / p.halves, b = blockIdx.y, tid = threadIdx.x;
  const int qh0 = h * p.G + (blockIdx.x % p.halves) * p.gq;   // first query head of this CTA
  const int G = p.gq;
  constexpr int CH = 1024 / D;          // chunks of the contraction index
  constexpr int PER = D / CH;
  const int j = tid % D, c = tid / D;
  // the rotation and the query are fetched in the same round trip
  const float* r = p.r_k + static_cast<size_t>(h) * D * D;
  float rv[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) rv[u] = r[(c * PER + u) * D + j];
  for (int i = tid; i < G * D; i += blockDim.x)
    qs[i / D][i % D] = bf16_to_float(p.q[(static_cast<size_t>(b) * p.hq + qh0) * D + i]);
  __syncthreads();
  for (int g = 0; g < G; ++g) {
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < PER; ++u) acc = fmaf(qs[g][c * PER + u], rv[u], acc);
    partial[c][g][j] = acc;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += blockDim.x) {
    const int g = i / D, jj = i % D;
    float acc = 0.f;
#pragma unroll
    for (int cc = 0; cc < CH; ++cc) acc += partial[cc][g][jj];
    p.qrot[(static_cast<size_t>(b) * p.hq + qh0 + g) * D + jj] = acc;
  }
}

// ---------------------------------------------------------------- split-K

// P: 2-bit code planes of the cache (1: INT2; 2: the INT4 variant, whose 20d
// blocks allow four ring stages per warp at two CTAs per SM)
template <int D, bool kBf16Only, int P = 1>
struct SplitCfg {
  // code-page ring depth per warp: 64 bulk copies in flight per SM at two CTAs
  // per SM (the streaming rate falls with more outstanding copies per SM)
  static constexpr int kStagesI = 4;
  static constexpr int kStagesB = kBf16Only ? 3 : 1;     // BF16 ring depth per warp
  static constexpr int kRingI = kDWarps * kStagesI * Fmt<D, P>::kInt2Block;
  static constexpr int kRingB = kDWarps * kStagesB * Fmt<D>::kBf16Block;
  static constexpr int kRing = kBf16Only ? kRingB : (kRingI > kRingB ? kRingI : kRingB);
  static constexpr int kScratch = kDWarps * (16 + 8 * D) * 4;
  static_assert(kScratch <= kRing, "merge scratch reuses the ring");
  static constexpr int kIds = 0;                                      // int [kMaxCtaPages]
  // the BF16 split's logical pages; in an INT2 split the same bytes hold the
  // query operands: q' as fp16 hi and lo fragments ([D/16][32] uint2 each),
  // then the zero-term operand (uint32 [32])
  static constexpr int kLps = kIds + kMaxCtaPages * 4;
  static constexpr int kQzOff = 2 * (D / 16) * 32 * 8;                 // zero-term operand, flags
  static constexpr int kQOperands = kQzOff + 32 * 4 + 16;
  static constexpr int kLpsBytes = kMaxCtaPages * 4 > kQOperands ? kMaxCtaPages * 4 : kQOperands;
  static constexpr int kBars = (kLps + kLpsBytes + 15) / 16 * 16;    // u64 [warps][stages]
  static constexpr int kRingOff = kBars + kDWarps * 8 * 8;
  static constexpr int kBytes = kRingOff + kRing;
  static constexpr int kCtasPerSm = kBf16Only ? 1 : 2;
  static_assert(kStagesI <= 8 && kStagesB <= 8, "eight mbarriers per warp");
};

struct Softmax {
  float m0, m1, l0, l1;   // running max (log2 domain) and partial sum for g = 2tig, 2tig+1
};

// Online-softmax update for one 16-token tile.  l[] are log2-domain logits in
// the m16n8 accumulator layout (rows = tokens gid / gid+8, cols = query heads
// 2tig / 2tig+1).  The running max is only raised (cross-lane reduction plus
// rescale of the accumulators) when some logit exceeds it by more than kTau,
// so most tiles skip the shuffles; probabilities stay <= 2^kTau.
constexpr float kTau = 8.f;

template <int NT>
__device__ __forceinline__ void softmax_tile(Softmax& st, float (&l)[4], float (&o)[NT][4],
                                             float (&z)[4], float (&pr)[4]) {
  float mx0 = fmaxf(l[0], l[2]), mx1 = fmaxf(l[1], l[3]);
  if (__any_sync(0xffffffffu, mx0 > st.m0 + kTau || mx1 > st.m1 + kTau)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
    const float a0 = (n0 == st.m0) ? 1.f : fast_exp2(st.m0 - n0);
    const float a1 = (n1 == st.m1) ? 1.f : fast_exp2(st.m1 - n1);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      o[t][0] *= a0; o[t][2] *= a0;
      o[t][1] *= a1; o[t][3] *= a1;
    }
    z[0] *= a0; z[1] *= a1;
    st.l0 *= a0; st.l1 *= a1;
    st.m0 = n0; st.m1 = n1;
  }
  const float b0 = st.m0 == -INFINITY ? 0.f : st.m0;
  const float b1 = st.m1 == -INFINITY ? 0.f : st.m1;
  pr[0] = fast_exp2(l[0] - b0);
  pr[1] = fast_exp2(l[1] - b1);
  pr[2] = fast_exp2(l[2] - b0);
  pr[3] = fast_exp2(l[3] - b1);
  st.l0 += pr[0] + pr[2];
  st.l1 += pr[1] + pr[3];
}

// Same update for two 16-token tiles at once (one vote, one rescale).  The
// probability sum is accumulated elsewhere (ones row of the zero-term MMA).
// The probabilities come out weighed by 2^pe (see int2_pscale_log2).
template <int NT>
__device__ __forceinline__ void softmax_pair(Softmax& st, float (&la)[4], float (&lb)[4],
                                             float (&o)[NT][4], float (&z)[4], float (&pa)[4],
                                             float (&pb)[4], float pe) {
  float mx0 = fmaxf(fmaxf(la[0], la[2]), fmaxf(lb[0], lb[2]));
  float mx1 = fmaxf(fmaxf(la[1], la[3]), fmaxf(lb[1], lb[3]));
  if (__any_sync(0xffffffffu, mx0 > st.m0 + kTau || mx1 > st.m1 + kTau)) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
    const float a0 = (n0 == st.m0) ? 1.f : fast_exp2(st.m0 - n0);
    const float a1 = (n1 == st.m1) ? 1.f : fast_exp2(st.m1 - n1);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      o[t][0] *= a0; o[t][2] *= a0;
      o[t][1] *= a1; o[t][3] *= a1;
    }
    z[0] *= a0; z[1] *= a1; z[2] *= a0; z[3] *= a1;
    st.m0 = n0; st.m1 = n1;
  }
  const float b0 = (st.m0 == -INFINITY ? 0.f : st.m0) - pe;
  const float b1 = (st.m1 == -INFINITY ? 0.f : st.m1) - pe;
  pa[0] = fast_exp2(la[0] - b0); pa[1] = fast_exp2(la[1] - b1);
  pa[2] = fast_exp2(la[2] - b0); pa[3] = fast_exp2(la[3] - b1);
  pb[0] = fast_exp2(lb[0] - b0); pb[1] = fast_exp2(lb[1] - b1);
  pb[2] = fast_exp2(lb[2] - b0); pb[3] = fast_exp2(lb[3] - b1);
}

// Exponent pe of the power-of-two weight 2^pe the INT2 probabilities carry
// into p.V.  There the tensor cores see p and p * s in fp16, with p <= 2^kTau
// (the lazily raised running max) and s <= fp16((max - min)/3) <= 2 clip / 3
// (the group range lies inside [-clip, clip]).  pe is the largest exponent
// with 2^pe * 2^kTau * s_max <= 2^15 (at most 7, so 2^pe p stays below fp16's
// largest value): p * s never overflows and small p * s stay out of fp16's
// subnormal range as far as the headroom allows.  The weight cancels out of
// the split's results (output and probability sum are divided by it).
__device__ __forceinline__ float int2_pscale_log2(float clip_v) {
  const float smax = fminf(65504.f, fmaxf(clip_v, 0.f) * (2.f / 3.f) * 1.001f);
  if (!(smax > 0.f)) return 7.f;
  return fmaxf(-24.f, fminf(7.f, floorf(log2f(32768.f / (exp2f(kTau) * smax)))));
}

// The INT2 loop's precision, chosen once per split CTA.  With q' and p * s in
// fp16 alone (2^-12 relative) the error of an output element grows with the
// size of the logits and of the values; the fast loop is kept where both stay
// at the scale of unit-variance activations with outliers (|logits| below
// 2^4 in log2 units, bounded by max |q'| * clip_K / sqrt(d) / ln 2, and a value
// clip below 32, where the measured error of the fast loop is below a quarter
// of the output tolerance), and the precise loop (fp16 pairs for both,
// ~2^-22) runs otherwise.
constexpr float kFastLogitLog2 = 16.f;
constexpr float kFastValueClip = 32.f;

__device__ __forceinline__ bool split_precise(float qmax, float clip_k, float clip_v,
                                              float scale_log2) {
  return !(qmax * fabsf(clip_k) * scale_log2 <= kFastLogitLog2 && fabsf(clip_v) <= kFastValueClip);
}

// The query columns of one split CTA.  MMA column c (0..7) holds query head
// qh0 + c % gq of batch row row0 + c / gq, for c < gq * nrows (the rest are
// unused).  lim0 / lim1: the visibility limits (positions below) of this
// thread's columns 2tig and 2tig + 1; lim_lo: the smallest over the rows.
struct Cols {
  int row0, nrows, qh0, lim0, lim1, lim_lo;
};

__device__ __forceinline__ bool tok_ok(int t, int L, int sink, int window, int mode, int lim) {
  // mode 0: INT2 region; 1: BF16 region (sink + recent); 2: all tokens; lim: the
  // row sees positions below lim only (lim <= L)
  if (mode == 0) return t >= sink && t < L - window && t < lim;
  if (mode == 1) return t < lim && (t < sink || t >= L - window);
  return t < L;
}

// Bounded wait on one stage; a timeout drains the copies still in flight (with
// the same bound) and reports false so the caller stops.
// kAllIssued: every page of the warp was copied (INT2 rings copy page 0 for an
// invalid id); otherwise only pages with a valid id were.
template <int NS, bool kAllIssued = false>
__device__ __forceinline__ bool wait_stage(uint64_t* wbar, int s, uint32_t& phase, int i, int my_n,
                                           const int* ids, int warp, int32_t* status) {
  const bool ok = mbar_wait(&wbar[s], (phase >> s) & 1u, status);
  phase ^= 1u << s;
  if (__all_sync(0xffffffffu, ok)) return true;
  for (int j = i + 1; j < min(i + NS, my_n); ++j) {
    if (kAllIssued || ids[warp + kDWarps * j] >= 0) {
      const int sj = j % NS;
      mbar_wait(&wbar[sj], (phase >> sj) & 1u, status);
      phase ^= 1u << sj;
    }
  }
  return false;
}

// q.K for one INT2 page-head staged at st: log2-domain logits in the m16n8
// accumulator layout (rows = tokens gid / gid+8, cols = query heads 2tig / 2tig+1).
// A lane's code words of one plane (d/32 words: one per 32-channel group).
template <int NG>
__device__ __forceinline__ void load_words(const uint8_t* base, int lane, uint32_t (&w)[NG]) {
  if constexpr (NG == 4) {
    const uint4 v = reinterpret_cast<const uint4*>(base)[lane];
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    const uint2 v = reinterpret_cast<const uint2*>(base)[lane];
    w[0] = v.x; w[1] = v.y;
  }
}

// q.K for NPG code page-heads at once (one or two: the query operand is read
// once for both).  P = 2 (INT4 variant): the code is 4 * hi + lo, each plane
// read as INT2 codes; the high plane's dot products weigh 4.  Each group's dot
// products are weighed by the token's key scale, and the sum is brought to
// log2-domain logits by one multiply-add onto the zero term.
// kPrecise: the query enters as an fp16 pair, q' = hi + lo (lo the fp16
// rounding of what hi leaves): both products with a code are exact and the pair
// carries q' to ~2^-22.  Otherwise q' enters as fp16 alone (2^-12 relative),
// which the split CTA allows only for logits of moderate size (split_precise).
template <int D, int P, int NPG, bool kPrecise>
__device__ __forceinline__ void int2_qk(const uint8_t* const (&st)[NPG], const uint2* qbs,
                                        const uint2* qbl, uint32_t qz, float ks, int lane,
                                        float (&lg)[NPG][4]) {
  using F = Fmt<D, P>;
  constexpr int NG = D / 32;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t kw[NPG][P][NG], sa[NPG][NG], sb[NPG][NG];
  float zt[NPG][4], acc[NPG][4];
#pragma unroll
  for (int pg = 0; pg < NPG; ++pg) {
#pragma unroll
    for (int pl = 0; pl < P; ++pl) load_words<NG>(st[pg] + F::kKc + pl * F::kPlane, lane, kw[pg][pl]);
    const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st[pg] + F::kKsz);
    uint32_t za = 0, zb = 0;
    if (tig < NG) {
      const uint32_t e0 = ksz[gid * NG + tig], e1 = ksz[(gid + 8) * NG + tig];
      za = __byte_perm(e0, e0, 0x3232);
      zb = __byte_perm(e1, e1, 0x3232);
    }
    mma_f16_z(zt[pg], za, zb, 0u, 0u, qz, 0u);     // zero term, already in log2 units
    if constexpr (NG == 4) {
      const uint4 a = reinterpret_cast<const uint4*>(ksz)[gid];
      const uint4 c = reinterpret_cast<const uint4*>(ksz)[gid + 8];
      sa[pg][0] = a.x; sa[pg][1] = a.y; sa[pg][2] = a.z; sa[pg][3] = a.w;
      sb[pg][0] = c.x; sb[pg][1] = c.y; sb[pg][2] = c.z; sb[pg][3] = c.w;
    } else {
      const uint2 a = reinterpret_cast<const uint2*>(ksz)[gid];
      const uint2 c = reinterpret_cast<const uint2*>(ksz)[gid + 8];
      sa[pg][0] = a.x; sa[pg][1] = a.y;
      sb[pg][0] = c.x; sb[pg][1] = c.y;
    }
  }
#pragma unroll
  for (int m = 0; m < NG; ++m) {
    // pair (s, i) sits at bits 4s+2i (+16); s = 2, 3 are reached with one shift
    // by 8, so every extracted half is code * 4^i * 16^(s&1) * 2^-24
    const uint32_t m0 = 0x00030003u, m1 = 0x00300030u;
    const uint2 b0 = qbs[(2 * m) * 32 + lane], b1 = qbs[(2 * m + 1) * 32 + lane];
    uint2 c0 = make_uint2(0u, 0u), c1 = make_uint2(0u, 0u);
    if constexpr (kPrecise) {
      c0 = qbl[(2 * m) * 32 + lane];
      c1 = qbl[(2 * m + 1) * 32 + lane];
    }
#pragma unroll
    for (int pg = 0; pg < NPG; ++pg) {
      float dg[4];
      {   // A registers a0..a3 hold key pairs s = 0, 2, 1, 3 (lowest plane)
        const uint32_t wl = kw[pg][P - 1][m], wh = kw[pg][P - 1][m] >> 8;
        const uint32_t a0 = wl & m0, a1 = wh & m0, a2 = wl & m1, a3 = wh & m1;
        const uint32_t e0 = wl & (m0 << 2), e1 = wh & (m0 << 2), e2 = wl & (m1 << 2),
                       e3 = wh & (m1 << 2);
        mma_f16_z(dg, a0, a1, a2, a3, b0.x, b0.y);
        mma_f16(dg, e0, e1, e2, e3, b1.x, b1.y);
        if constexpr (kPrecise) {
          mma_f16(dg, a0, a1, a2, a3, c0.x, c0.y);
          mma_f16(dg, e0, e1, e2, e3, c1.x, c1.y);
        }
      }
      if constexpr (P == 2) {   // high plane: code bits 3..2
        const uint32_t wl = kw[pg][0][m], wh = kw[pg][0][m] >> 8;
        const uint32_t a0 = wl & m0, a1 = wh & m0, a2 = wl & m1, a3 = wh & m1;
        const uint32_t e0 = wl & (m0 << 2), e1 = wh & (m0 << 2), e2 = wl & (m1 << 2),
                       e3 = wh & (m1 << 2);
        float dh[4];
        mma_f16_z(dh, a0, a1, a2, a3, b0.x, b0.y);
        mma_f16(dh, e0, e1, e2, e3, b1.x, b1.y);
        if constexpr (kPrecise) {
          mma_f16(dh, a0, a1, a2, a3, c0.x, c0.y);
          mma_f16(dh, e0, e1, e2, e3, c1.x, c1.y);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) dg[k] = fmaf(4.f, dh[k], dg[k]);
      }
      const float fa = half_lo(sa[pg][m]), fb = half_lo(sb[pg][m]);
      if (m == 0) {
        acc[pg][0] = fa * dg[0]; acc[pg][1] = fa * dg[1];
        acc[pg][2] = fb * dg[2]; acc[pg][3] = fb * dg[3];
      } else {
        acc[pg][0] = fmaf(fa, dg[0], acc[pg][0]);
        acc[pg][1] = fmaf(fa, dg[1], acc[pg][1]);
        acc[pg][2] = fmaf(fb, dg[2], acc[pg][2]);
        acc[pg][3] = fmaf(fb, dg[3], acc[pg][3]);
      }
    }
  }
#pragma unroll
  for (int pg = 0; pg < NPG; ++pg)
#pragma unroll
    for (int k = 0; k < 4; ++k) lg[pg][k] = fmaf(acc[pg][k], ks, zt[pg][k]);
}

// p.V for one INT2 page-head: o (channel x query head) += codes^T (p * s), plus
// the zero term and, on the spare row NG, the probability sum (ones row).
// kPrecise: p enters as an fp16 pair p = hi + lo, and p * s as the pair
// (fp16(hi s), the rounding of (hi s - fp16(hi s)) + lo s), the first residual
// exact by a fused multiply-add: both to ~2^-22 instead of fp16's 2^-12.
template <int D, int P, bool kPrecise>
__device__ __forceinline__ void int2_pv(const uint8_t* st, const float (&pr)[4], int lane,
                                        float (&o)[D / 16][4], float (&zacc)[4]) {
  using F = Fmt<D, P>;
  constexpr int NG = D / 32;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t h01 = pack_half2(pr[0], pr[1]), h23 = pack_half2(pr[2], pr[3]);
  const uint32_t pb0 = movmatrix_trans(h01);
  const uint32_t pb1 = movmatrix_trans(h23);
  uint32_t pl0 = 0u, pl1 = 0u;
  if constexpr (kPrecise) {
    pl0 = movmatrix_trans(pack_half2(pr[0] - half_lo(h01), pr[1] - half_hi(h01)));
    pl1 = movmatrix_trans(pack_half2(pr[2] - half_lo(h23), pr[3] - half_hi(h23)));
  }
  uint32_t vw[P][NG], vs0[NG], vs1[NG];
#pragma unroll
  for (int pl = 0; pl < P; ++pl) load_words<NG>(st + F::kVc + pl * F::kPlane, lane, vw[pl]);
  const uint32_t* vsw = reinterpret_cast<const uint32_t*>(st + F::kVs);
  if constexpr (NG == 4) {
    const uint4 a = reinterpret_cast<const uint4*>(vsw)[tig * 2];
    const uint4 c = reinterpret_cast<const uint4*>(vsw)[tig * 2 + 1];
    vs0[0] = a.x; vs0[1] = a.y; vs0[2] = a.z; vs0[3] = a.w;
    vs1[0] = c.x; vs1[1] = c.y; vs1[2] = c.z; vs1[3] = c.w;
  } else {
    const uint2 a = reinterpret_cast<const uint2*>(vsw)[tig * 2];
    const uint2 c = reinterpret_cast<const uint2*>(vsw)[tig * 2 + 1];
    vs0[0] = a.x; vs0[1] = a.y;
    vs1[0] = c.x; vs1[1] = c.y;
  }
#pragma unroll
  for (int m = 0; m < NG; ++m) {
    const uint32_t bb0 = hmul2_u32(pb0, vs0[m]);
    const uint32_t bb1 = hmul2_u32(pb1, vs1[m]);
    uint32_t bl0 = 0u, bl1 = 0u;
    if constexpr (kPrecise) {
      bl0 = hfma2_u32(pl0, vs0[m], hfma2_u32(pb0, vs0[m], bb0 ^ 0x80008000u));
      bl1 = hfma2_u32(pl1, vs1[m], hfma2_u32(pb1, vs1[m], bb1 ^ 0x80008000u));
    }
    // value pair s = r: rows gid (s = 0, 2) read at 4^i, rows gid+8 (s = 1, 3) at 16 * 4^i
    const uint32_t m0 = 0x00030003u, m1 = 0x00300030u;
    {   // lowest plane
      const uint32_t wl = vw[P - 1][m], wh = vw[P - 1][m] >> 8;
      const uint32_t a0 = wl & m0, a1 = wl & m1, a2 = wh & m0, a3 = wh & m1;
      const uint32_t e0 = wl & (m0 << 2), e1 = wl & (m1 << 2), e2 = wh & (m0 << 2),
                     e3 = wh & (m1 << 2);
      mma_f16(o[2 * m], a0, a1, a2, a3, bb0, bb1);
      mma_f16(o[2 * m + 1], e0, e1, e2, e3, bb0, bb1);
      if constexpr (kPrecise) {
        mma_f16(o[2 * m], a0, a1, a2, a3, bl0, bl1);
        mma_f16(o[2 * m + 1], e0, e1, e2, e3, bl0, bl1);
      }
    }
    if constexpr (P == 2) {   // high plane, weighed by 4 (exact in fp16)
      const uint32_t four = 0x44004400u;
      const uint32_t bh0 = hmul2_u32(bb0, four), bh1 = hmul2_u32(bb1, four);
      const uint32_t wl = vw[0][m], wh = vw[0][m] >> 8;
      const uint32_t a0 = wl & m0, a1 = wl & m1, a2 = wh & m0, a3 = wh & m1;
      const uint32_t e0 = wl & (m0 << 2), e1 = wl & (m1 << 2), e2 = wh & (m0 << 2),
                     e3 = wh & (m1 << 2);
      mma_f16(o[2 * m], a0, a1, a2, a3, bh0, bh1);
      mma_f16(o[2 * m + 1], e0, e1, e2, e3, bh0, bh1);
      if constexpr (kPrecise) {
        const uint32_t bm0 = hmul2_u32(bl0, four), bm1 = hmul2_u32(bl1, four);
        mma_f16(o[2 * m], a0, a1, a2, a3, bm0, bm1);
        mma_f16(o[2 * m + 1], e0, e1, e2, e3, bm0, bm1);
      }
    }
  }
  const uint32_t* vz = reinterpret_cast<const uint32_t*>(st + F::kVz);
  uint32_t za0 = 0, za2 = 0;
  if (gid < NG) {
    za0 = vz[(tig * 2) * NG + gid];
    za2 = vz[(tig * 2 + 1) * NG + gid];
  } else if (gid == NG) {
    za0 = za2 = 0x3C003C00u;   // ones: row NG accumulates sum_t p
  }
  mma_f16(zacc, za0, 0u, za2, 0u, pb0, pb1);
  if constexpr (kPrecise) mma_f16(zacc, za0, 0u, za2, 0u, pl0, pl1);
}

// INT2 pages [lo, lo + n) of one (sequence, KV head): warp w takes pages
// w, w + 8, ... through its own ring of NS bulk-copied page-head blocks, two
// pages per step so their dependency chains overlap and share one softmax
// update.  Invalid page ids (negative) copy page 0 and are masked out.
template <int D, int NS, int P, bool kPacked>
__device__ __forceinline__ void int2_pages(const DecodeParams& p, int b, int h, int warp, int lane,
                                           const int* ids, int lo, int n, int L, uint8_t* ring,
                                           uint64_t* bars, uint2* qbs, float (&o)[D / 16][4],
                                           float (&zacc)[4], Softmax& sm, int defer_lp,
                                           const Cols& cs) {
  static_assert(NS % 2 == 0, "pages are consumed in pairs of stages");
  constexpr int NG = D / 32, NK = D / 16;
  constexpr int SB = Fmt<D, P>::kInt2Block;
  const int gid = lane >> 2, tig = lane & 3, G = p.gq;
  uint8_t* wring = ring + warp * NS * SB;
  uint64_t* wbar = bars + warp * 8;
  const uint8_t* pool_h = p.int2_pool + static_cast<size_t>(h) * SB;
  const size_t pstride = static_cast<size_t>(p.hkv) * SB;
  const int my_n = n > warp ? (n - warp + kDWarps - 1) / kDWarps : 0;
  const int* wids = ids + warp;                   // page i of this warp: wids[8 i]
  // Only kPreStages pages per warp are requested before the rotated query is
  // read: a full ring from every CTA at once queues the small q' loads behind
  // megabytes of page copies.  The rest of the ring follows the staging.
  // A page the predecessor grid may still be writing (defer_lp) waits for the
  // second batch.
  constexpr int kPreStages = 2;
  int deferred = -1;
  if (lane == 0) {
    for (int i = 0; i < min(kPreStages, my_n); ++i) {
      if (lo + warp + kDWarps * i == defer_lp) {
        deferred = i;
        continue;
      }
      mbar_arrive_expect_tx(&wbar[i], SB);
      bulk_g2s(wring + i * SB, pool_h + max(wids[kDWarps * i], 0) * pstride, SB, &wbar[i]);
    }
  }
  // ---- query operand, once the rotated query is complete: warp 0 reads q'
  // once and stages the MMA operand and the zero-term operand for every warp
  pdl_wait();
  uint2* qbl = qbs + NK * 32;                                 // the lo halves of the pair
  uint32_t* qzs = reinterpret_cast<uint32_t*>(qbs + 2 * NK * 32);
  if (warp == 0) {
    uint32_t qz = 0;
    // this lane's column gid: head qh0 + gid % G of row row0 + gid / G when
    // rows are packed, head qh0 + gid of row row0 otherwise
    const bool cvalid = kPacked ? gid < G * cs.nrows : gid < G;
    const int crow = kPacked && cvalid ? gid / G : 0;
    const int chead = kPacked ? gid % G : gid;
    const float* qr = p.qrot + (static_cast<size_t>(cs.row0 + crow) * p.hq + cs.qh0 + chead) * D;
    float gs[NG];
    float qmax = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) gs[g] = 0.f;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
      if (cvalid) {
        v0 = __ldcg(reinterpret_cast<const float2*>(qr + 16 * kk + 2 * tig));
        v1 = __ldcg(reinterpret_cast<const float2*>(qr + 16 * kk + 2 * tig + 8));
      }
      qmax = fmax_nan(qmax, fmax_nan(fmax_nan(fabsf(v0.x), fabsf(v0.y)),
                                     fmax_nan(fabsf(v1.x), fabsf(v1.y))));
      gs[kk >> 1] += (v0.x + v0.y) + (v1.x + v1.y);
      // codes of k-step parity i and channel half h are read at 4^i * 16^h
      // (exact power-of-two weights); each weighted value becomes an fp16 pair
      const float sc = (kk & 1) ? 0.25f : 1.f;
      const float w0 = v0.x * sc, w1 = v0.y * sc;
      const float w2 = v1.x * sc * 0.0625f, w3 = v1.y * sc * 0.0625f;
      const uint32_t h01 = pack_half2(w0, w1), h23 = pack_half2(w2, w3);
      qbs[kk * 32 + lane] = make_uint2(h01, h23);
      qbl[kk * 32 + lane] = make_uint2(pack_half2(w0 - half_lo(h01), w1 - half_hi(h01)),
                                       pack_half2(w2 - half_lo(h23), w3 - half_hi(h23)));
    }
    float mine = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      gs[g] += __shfl_xor_sync(0xffffffffu, gs[g], 1);
      gs[g] += __shfl_xor_sync(0xffffffffu, gs[g], 2);
      if (g == tig) mine = gs[g];
    }
    if (tig < NG) {   // zero-term operand, pre-scaled to log2-domain logits
      mine *= p.scale_log2;
      const __half hi = __float2half_rn(mine);
      const __half lo16 = __float2half_rn(mine - __half2float(hi));
      qz = static_cast<uint32_t>(__half_as_ushort(hi)) |
           (static_cast<uint32_t>(__half_as_ushort(lo16)) << 16);
    }
    qzs[lane] = qz;
    // a NaN query takes the precise loop (either propagates it)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      qmax = fmax_nan(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
    if (lane == 0)
      qzs[32] = split_precise(qmax, p.clip_k[h], p.clip_v[h], p.scale_log2) ? 1u : 0u;
  }
  __syncthreads();
  const uint32_t qz = qzs[lane];
  const bool precise = qzs[32] != 0u;
  if (lane == 0) {
    if (deferred >= 0) {
      mbar_arrive_expect_tx(&wbar[deferred], SB);
      bulk_g2s(wring + deferred * SB, pool_h + max(wids[kDWarps * deferred], 0) * pstride, SB,
               &wbar[deferred]);
    }
    for (int i = kPreStages; i < min(NS, my_n); ++i) {
      mbar_arrive_expect_tx(&wbar[i], SB);
      bulk_g2s(wring + i * SB, pool_h + max(wids[kDWarps * i], 0) * pstride, SB, &wbar[i]);
    }
  }
  // the page loop in the precision the CTA chose (two instantiations)
  auto loop = [&](auto precise_tag) {
    constexpr bool kPrecise = decltype(precise_tag)::value;
    const float ks = p.scale_log2 * 16777216.f;   // codes are read as code * 2^-24
    const float pe = int2_pscale_log2(p.clip_v[h]);
    // the merge divides the weight 2^pe out again: it finds pe in shared
    // memory (qzs[33] is read once every warp has left the loop)
    if (warp == 0 && lane == 0) qzs[33] = __float_as_uint(pe);
    // every column sees INT2 tokens in [tok_lo, tok_hi); column 2tig (2tig+1)
    // sees them below min(L - window, lim0 (lim1)), worked out where a page needs masking
    const int tok_lo = p.sink, tok_hi = min(L - p.window, cs.lim_lo);
    uint32_t phase = 0;
    int s = 0;
    int i = 0;
    for (; i + 1 < my_n; i += 2) {
      const int idA = wids[kDWarps * i], idB = wids[kDWarps * (i + 1)];
      if (!wait_stage<NS, true>(wbar, s, phase, i, my_n, ids, warp, p.status)) return;
      if (!wait_stage<NS, true>(wbar, s + 1, phase, i + 1, my_n, ids, warp, p.status)) return;
      const uint8_t* stA = wring + s * SB;
      const uint8_t* stB = stA + SB;
      float lab[2][4];
      {
        const uint8_t* const sts[2] = {stA, stB};
        int2_qk<D, P, 2, kPrecise>(sts, qbs, qbl, qz, ks, lane, lab);
      }
      float (&la)[4] = lab[0];
      float (&lb)[4] = lab[1];
      const int pA = (lo + warp + kDWarps * i) * kPage, pB = pA + kDWarps * kPage;
      if (pA < tok_lo || pB + kPage > tok_hi || (idA | idB) < 0) {
        const int t0 = pA + gid, t1 = t0 + 8, u0 = pB + gid, u1 = u0 + 8;
        if constexpr (kPacked) {   // each column its own row's limit
          const int hi0 = min(L - p.window, cs.lim0), hi1 = min(L - p.window, cs.lim1);
          const bool a0 = idA >= 0 && t0 >= tok_lo, a1 = idA >= 0 && t1 >= tok_lo;
          const bool c0 = idB >= 0 && u0 >= tok_lo, c1 = idB >= 0 && u1 >= tok_lo;
          if (!(a0 && t0 < hi0)) la[0] = -INFINITY;
          if (!(a0 && t0 < hi1)) la[1] = -INFINITY;
          if (!(a1 && t1 < hi0)) la[2] = -INFINITY;
          if (!(a1 && t1 < hi1)) la[3] = -INFINITY;
          if (!(c0 && u0 < hi0)) lb[0] = -INFINITY;
          if (!(c0 && u0 < hi1)) lb[1] = -INFINITY;
          if (!(c1 && u1 < hi0)) lb[2] = -INFINITY;
          if (!(c1 && u1 < hi1)) lb[3] = -INFINITY;
        } else {
          if (idA < 0 || t0 < tok_lo || t0 >= tok_hi) la[0] = la[1] = -INFINITY;
          if (idA < 0 || t1 < tok_lo || t1 >= tok_hi) la[2] = la[3] = -INFINITY;
          if (idB < 0 || u0 < tok_lo || u0 >= tok_hi) lb[0] = lb[1] = -INFINITY;
          if (idB < 0 || u1 < tok_lo || u1 >= tok_hi) lb[2] = lb[3] = -INFINITY;
        }
      }
      float pa[4], pbv[4];
      softmax_pair<NK>(sm, la, lb, o, zacc, pa, pbv, pe);
      int2_pv<D, P, kPrecise>(stA, pa, lane, o, zacc);
      int2_pv<D, P, kPrecise>(stB, pbv, lane, o, zacc);
      __syncwarp();
      if (lane == 0) {
        if (i + NS < my_n) {
          mbar_arrive_expect_tx(&wbar[s], SB);
          bulk_g2s(wring + s * SB, pool_h + max(wids[kDWarps * (i + NS)], 0) * pstride, SB, &wbar[s]);
        }
        if (i + 1 + NS < my_n) {
          mbar_arrive_expect_tx(&wbar[s + 1], SB);
          bulk_g2s(wring + (s + 1) * SB, pool_h + max(wids[kDWarps * (i + 1 + NS)], 0) * pstride,
                   SB, &wbar[s + 1]);
        }
      }
      s = (s + 2 == NS) ? 0 : s + 2;
    }
    if (i < my_n) {   // odd tail: one page
      const int idA = wids[kDWarps * i];
      if (!wait_stage<NS, true>(wbar, s, phase, i, my_n, ids, warp, p.status)) return;
      const uint8_t* stA = wring + s * SB;
      float l1[1][4];
      {
        const uint8_t* const sts[1] = {stA};
        int2_qk<D, P, 1, kPrecise>(sts, qbs, qbl, qz, ks, lane, l1);
      }
      float (&la)[4] = l1[0];
      const int pA = (lo + warp + kDWarps * i) * kPage;
      const int t0 = pA + gid, t1 = t0 + 8;
      if constexpr (kPacked) {
        const int hi0 = min(L - p.window, cs.lim0), hi1 = min(L - p.window, cs.lim1);
        const bool a0 = idA >= 0 && t0 >= tok_lo, a1 = idA >= 0 && t1 >= tok_lo;
        if (!(a0 && t0 < hi0)) la[0] = -INFINITY;
        if (!(a0 && t0 < hi1)) la[1] = -INFINITY;
        if (!(a1 && t1 < hi0)) la[2] = -INFINITY;
        if (!(a1 && t1 < hi1)) la[3] = -INFINITY;
      } else {
        if (idA < 0 || t0 < tok_lo || t0 >= tok_hi) la[0] = la[1] = -INFINITY;
        if (idA < 0 || t1 < tok_lo || t1 >= tok_hi) la[2] = la[3] = -INFINITY;
      }
      float pa[4];
      float dummy[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY}, pd[4];
      softmax_pair<NK>(sm, la, dummy, o, zacc, pa, pd, pe);
      int2_pv<D, P, kPrecise>(stA, pa, lane, o, zacc);
    }

  };
  if (precise)
    loop(std::true_type{});
  else
    loop(std::false_type{});
}

// BF16 pages (the sink + recent split, or every page of the BF16 baseline):
// raw q against bf16 keys and values in the same fragment-native order.
// kSplitP: the probabilities enter p.V as a bf16 pair (p = hi + mid, two MMAs),
// exact to ~2^-17 instead of bf16's 2^-9, and for layers with large values
// (value clip above 32) as three pieces (a third MMA: ~2^-25), each piece the
// bf16 rounding of what the earlier ones leave.  Used for the sink + recent
// split of the mixed cache, where a query row may see only a few tokens (a row
// early in a chunk) or the window may hold most of the weight; the all-BF16
// baseline keeps one MMA.
template <int D, int NS, bool kSplitP, bool kPacked>
__device__ __forceinline__ void bf16_pages(const DecodeParams& p, int b, int h, int warp, int lane,
                                           const int* ids, const int* lps, int n, int L, int mode,
                                           uint8_t* ring, uint64_t* bars, float (&o)[D / 16][4],
                                           Softmax& sm, const Cols& cs) {
  constexpr int NK = D / 16;
  constexpr int SB = Fmt<D>::kBf16Block;
  const int gid = lane >> 2, tig = lane & 3, G = p.gq;
  uint8_t* wring = ring + warp * NS * SB;
  uint64_t* wbar = bars + warp * 8;
  const uint8_t* pool_h = p.bf16_pool + static_cast<size_t>(h) * SB;
  const size_t pstride = static_cast<size_t>(p.hkv) * SB;
  const int my_n = n > warp ? (n - warp + kDWarps - 1) / kDWarps : 0;
  auto prefill = [&] {
    if (lane == 0) {
      for (int i = 0; i < min(NS, my_n); ++i) {
        const int id = ids[warp + kDWarps * i];
        if (id >= 0) {
          mbar_arrive_expect_tx(&wbar[i], SB);
          bulk_g2s(wring + i * SB, pool_h + id * pstride, SB, &wbar[i]);
        }
      }
    }
  };
  if (!p.after_append) prefill();   // the new token's BF16 page may still be in writing
  pdl_wait();
  if (p.after_append) prefill();
  uint32_t qb[NK][2];
  {
    // column gid: head qh0 + gid % G of row row0 + gid / G when rows are packed
    const bool cvalid = kPacked ? gid < G * cs.nrows : gid < G;
    const int crow = kPacked && cvalid ? gid / G : 0;
    const int chead = kPacked ? gid % G : gid;
    const uint16_t* qr = p.q + (static_cast<size_t>(cs.row0 + crow) * p.hq + cs.qh0 + chead) * D;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      qb[kk][0] = cvalid ? *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * tig) : 0u;
      qb[kk][1] = cvalid ? *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * tig + 8) : 0u;
    }
  }
  const float scale_log2 = p.scale_log2;
  // the third piece of p only for layers with large values (the value clip
  // beyond the INT2 loop's fast-path bound; a NaN clip takes it too)
  const bool p3 = kSplitP && !(fabsf(p.clip_v[h]) <= kFastValueClip);
  float zdummy[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t phase = 0;
  int s = 0;
  for (int i = 0; i < my_n; ++i) {
    const int k = warp + kDWarps * i;
    if (ids[k] >= 0) {
      if (!wait_stage<NS>(wbar, s, phase, i, my_n, ids, warp, p.status)) return;
      const uint8_t* st = wring + s * SB;
      float dk[4] = {0.f, 0.f, 0.f, 0.f};
      const uint4* kb = reinterpret_cast<const uint4*>(st);
#pragma unroll
      for (int kk = 0; kk < NK; ++kk) {
        const uint4 a = kb[kk * 32 + lane];
        mma_bf16(dk, a.x, a.y, a.z, a.w, qb[kk][0], qb[kk][1]);
      }
      float lg[4] = {dk[0] * scale_log2, dk[1] * scale_log2, dk[2] * scale_log2, dk[3] * scale_log2};
      const int pbeg = lps[k] * kPage;
      const bool whole = mode == 2 && pbeg + kPage <= L && p.limits == nullptr;
      if (!whole) {
        const int t0 = pbeg + gid, t1 = t0 + 8;
        if constexpr (kPacked) {   // each column its own row's limit
          if (!tok_ok(t0, L, p.sink, p.window, mode, cs.lim0)) lg[0] = -INFINITY;
          if (!tok_ok(t0, L, p.sink, p.window, mode, cs.lim1)) lg[1] = -INFINITY;
          if (!tok_ok(t1, L, p.sink, p.window, mode, cs.lim0)) lg[2] = -INFINITY;
          if (!tok_ok(t1, L, p.sink, p.window, mode, cs.lim1)) lg[3] = -INFINITY;
        } else {
          if (!tok_ok(t0, L, p.sink, p.window, mode, cs.lim_lo)) lg[0] = lg[1] = -INFINITY;
          if (!tok_ok(t1, L, p.sink, p.window, mode, cs.lim_lo)) lg[2] = lg[3] = -INFINITY;
        }
      }
      float pr[4];
      softmax_tile<NK>(sm, lg, o, zdummy, pr);
      const uint32_t h01 = pack_bf162(pr[0], pr[1]);
      const uint32_t h23 = pack_bf162(pr[2], pr[3]);
      const uint32_t pb0 = movmatrix_trans(h01);
      const uint32_t pb1 = movmatrix_trans(h23);
      const uint4* vb = reinterpret_cast<const uint4*>(st + Fmt<D>::kBf16V);
#pragma unroll
      for (int mt = 0; mt < NK; ++mt) {
        const uint4 a = vb[mt * 32 + lane];
        mma_bf16(o[mt], a.x, a.y, a.z, a.w, pb0, pb1);
      }
      if constexpr (kSplitP) {
        // the parts of p the bf16 roundings dropped (each residual exact in fp32)
        const float e0 = pr[0] - bf16_lo_value(h01), e1 = pr[1] - bf16_hi_value(h01);
        const float e2 = pr[2] - bf16_lo_value(h23), e3 = pr[3] - bf16_hi_value(h23);
        const uint32_t m01 = pack_bf162(e0, e1), m23 = pack_bf162(e2, e3);
        const uint32_t pm0 = movmatrix_trans(m01), pm1 = movmatrix_trans(m23);
#pragma unroll
        for (int mt = 0; mt < NK; ++mt) {
          const uint4 a = vb[mt * 32 + lane];
          mma_bf16(o[mt], a.x, a.y, a.z, a.w, pm0, pm1);
        }
        if (p3) {
          const uint32_t pl0 =
              movmatrix_trans(pack_bf162(e0 - bf16_lo_value(m01), e1 - bf16_hi_value(m01)));
          const uint32_t pl1 =
              movmatrix_trans(pack_bf162(e2 - bf16_lo_value(m23), e3 - bf16_hi_value(m23)));
#pragma unroll
          for (int mt = 0; mt < NK; ++mt) {
            const uint4 a = vb[mt * 32 + lane];
            mma_bf16(o[mt], a.x, a.y, a.z, a.w, pl0, pl1);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + NS < my_n) {
      const int id = ids[k + kDWarps * NS];
      if (id >= 0) {
        mbar_arrive_expect_tx(&wbar[s], SB);
        bulk_g2s(wring + s * SB, pool_h + id * pstride, SB, &wbar[s]);
      }
    }
    s = (s + 1 == NS) ? 0 : s + 1;
  }
}

// kPacked: several rows of a sequence share the CTA's query columns (multi-row
// calls with G < 8); the decode and single-row calls use kPacked = false.
template <int D, bool kBf16Only, int P, bool kPacked>
__global__ void __launch_bounds__(kDThreads, SplitCfg<D, kBf16Only, P>::kCtasPerSm)
    split_kernel(const DecodeParams p) {
  using C = SplitCfg<D, kBf16Only, P>;
  constexpr int NG = D / 32;     // groups = code words per lane
  constexpr int NK = D / 16;     // k-steps / channel tiles
  extern __shared__ __align__(128) uint8_t smem[];
  int* ids = reinterpret_cast<int*>(smem + C::kIds);
  int* lps = reinterpret_cast<int*>(smem + C::kLps);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint8_t* ring = smem + C::kRingOff;

  const int split = blockIdx.x, h = blockIdx.y / p.halves, unit = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int G = p.gq;
  const int qh0 = h * p.G + (blockIdx.y % p.halves) * p.gq;   // first query head of this CTA

  // Without a gate kernel in front (the BF16-only call), nothing may be read
  // before the predecessor grid completes.
  if (p.wait_first) pdl_wait();
  // main splits know their page span without the length, so the page ids are
  // fetched in the same round trip as the length
  const bool bf16_split = kBf16Only || split == p.n_main;
  const int mode = kBf16Only ? 2 : (bf16_split ? 1 : 0);
  const int first = mode == 0 ? p.sink / kPage : 0;
  const int lo = first + split * p.pps;
  int sb, b, nrows;   // the sequence read, the CTA's first batch row, its rows
  if constexpr (kPacked) {
    const int ups = (p.rows_per_seq + p.rpu - 1) / p.rpu;   // CTA units per sequence
    sb = unit / ups;
    const int r_in = (unit % ups) * p.rpu;                   // first row within the sequence
    nrows = min(p.rpu, p.rows_per_seq - r_in);
    b = sb * p.rows_per_seq + r_in;
  } else {
    b = unit;
    sb = b / p.rows_per_seq;
    nrows = 1;
  }
  const int32_t* pt = (mode == 0 ? p.int2_pt : p.bf16_pt) + static_cast<size_t>(sb) * p.max_pages;
  const int64_t npages = mode == 0 ? p.n_int2_pages : p.n_bf16_pages;
  int spec[(kMaxCtaPages + kDThreads - 1) / kDThreads];
  if (mode != 1) {
#pragma unroll
    for (int r = 0; r < (kMaxCtaPages + kDThreads - 1) / kDThreads; ++r) {
      const int k = tid + r * kDThreads;
      spec[r] = (k < p.pps && lo + k < p.max_pages) ? pt[lo + k] : -1;
    }
  }
  int L = p.seq_lens[sb];
  if (L < 1 || L > p.max_len) {
    if (tid == 0 && p.status) atomicOr(p.status, OSCAR_DEVERR_SEQ_LEN);
    L = 0;
  }
  // visibility limits (positions below): the whole cache for a decode, per row
  // for several rows of a sequence; lim is the widest over the CTA's rows
  auto row_lim = [&](int r) -> int {
    if (!p.limits) return L;
    const int qp = p.limits[b + r];
    return (qp < 0 || qp >= L) ? 0 : qp + 1;
  };
  int lim = L, lim_lo = L;
  if (p.limits) {
    lim = 0;
    for (int r = 0; r < nrows; ++r) {
      const int lr = row_lim(r);
      if (lr == 0 && tid == 0 && p.status && L > 0) atomicOr(p.status, OSCAR_DEVERR_SEQ_LEN);
      lim = max(lim, lr);
      lim_lo = min(lim_lo, lr);
    }
  }
  Cols cs;
  cs.row0 = b;
  cs.nrows = nrows;
  cs.qh0 = qh0;
  cs.lim_lo = lim_lo;
  cs.lim0 = cs.lim1 = lim;
  if constexpr (kPacked) {   // this thread's columns 2tig, 2tig + 1 (unused columns: any finite limit)
    if (2 * tig < G * nrows) cs.lim0 = row_lim((2 * tig) / G);
    if (2 * tig + 1 < G * nrows) cs.lim1 = row_lim((2 * tig + 1) / G);
  }
  int n = 0;
  if (mode == 1) {
    // sink pages, then recent pages not already listed
    const int s_end = (min(p.sink, L) + kPage - 1) / kPage;
    const int r_beg = max(p.sink, L - p.window) / kPage;
    const int r_end = (L + kPage - 1) / kPage;
    const int r0 = max(r_beg, s_end);
    const int n_sink = s_end, n_rec = max(0, r_end - r0);
    n = min(n_sink + n_rec, kMaxCtaPages);
    for (int k = tid; k < n; k += kDThreads) {
      const int lp = k < n_sink ? k : r0 + (k - n_sink);
      lps[k] = lp;
      int id = lp < p.max_pages ? pt[lp] : -1;
      if (id < 0 || id >= npages) {
        if (p.status) atomicOr(p.status, OSCAR_DEVERR_PAGE_ID);
        id = -1;
      }
      ids[k] = id;
    }
  } else {
    const int hi = min(L - p.window, lim);   // INT2 tokens this row sees end below hi
    const int last = mode == 0
        ? ((hi > p.sink) ? (hi + kPage - 1) / kPage : first)
        : (L + kPage - 1) / kPage;
    n = max(0, min(min(last, lo + p.pps) - lo, kMaxCtaPages));
#pragma unroll
    for (int r = 0; r < (kMaxCtaPages + kDThreads - 1) / kDThreads; ++r) {
      const int k = tid + r * kDThreads;
      if (k < n) {
        int id = spec[r];
        if (id < 0 || id >= npages) {
          if (p.status) atomicOr(p.status, OSCAR_DEVERR_PAGE_ID);
          id = -1;
        }
        ids[k] = id;
        lps[k] = lo + k;
      }
    }
  }
  if (tid < kDWarps * 8) mbar_init(&bars[tid], 1);
  fence_mbar_init();
  __syncthreads();

  float o[NK][4];
#pragma unroll
  for (int t = 0; t < NK; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float zacc[4] = {0.f, 0.f, 0.f, 0.f};
  Softmax sm{-INFINITY, -INFINITY, 0.f, 0.f};
  // the INT2 page receiving the token that leaves the window in this step
  const int defer_lp = (p.after_append && L - 1 - p.window >= p.sink) ? (L - 1 - p.window) / kPage : -1;
  if (mode == 0)
    int2_pages<D, C::kStagesI, P, kPacked>(p, b, h, warp, lane, ids, lo, n, L, ring, bars,
                               reinterpret_cast<uint2*>(lps), o, zacc, sm, defer_lp, cs);
  else
    bf16_pages<D, C::kStagesB, !kBf16Only, kPacked>(p, b, h, warp, lane, ids, lps, n, L, mode, ring,
                                                    bars, o, sm, cs);

  pdl_trigger();

  // ---- warp result -> shared scratch (the ring is idle once every warp is here)
  float l0 = sm.l0, l1 = sm.l1;
  // INT2 pages: every probability carried the weight 2^pe (staged with q')
  const float unw =
      mode == 0 ? exp2f(-__uint_as_float(reinterpret_cast<const uint32_t*>(smem + C::kLps + C::kQzOff)[33]))
                : 1.f;
  if (mode == 0) {
    // INT2 pages: the probability sum sits on row NG of the zero-term accumulator
    l0 = __shfl_sync(0xffffffffu, zacc[0], NG * 4 + tig) * unw;
    l1 = __shfl_sync(0xffffffffu, zacc[1], NG * 4 + tig) * unw;
  } else {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
  }
  float zz0[NG], zz1[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    zz0[g] = __shfl_sync(0xffffffffu, zacc[0], g * 4 + tig);
    zz1[g] = __shfl_sync(0xffffffffu, zacc[1], g * 4 + tig);
  }
  __syncthreads();
  // per warp: [8] max, [8] sum, then the output channel-major, [D][8], so that
  // a lane's two columns are one 8-byte store (a warp's stores fill 256
  // consecutive bytes: no bank conflicts)
  float* scr = reinterpret_cast<float*>(ring);
  float* wm = scr + warp * (16 + 8 * D);
  float* wl = wm + 8;
  float* wo = wm + 16;
  if (gid == 0) {
    wm[2 * tig] = sm.m0; wm[2 * tig + 1] = sm.m1;
    wl[2 * tig] = l0; wl[2 * tig + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < NK; ++mt) {
    const int c0 = 16 * mt + gid, c1 = c0 + 8;
    float v0 = o[mt][0], v1 = o[mt][1], v2 = o[mt][2], v3 = o[mt][3];
    if (mode == 0) {
      // undo the code read-out scale: 2^24 / 4^(mt&1), and / 16 for rows gid+8,
      // and the probabilities' weight
      const float sc = ((mt & 1) ? 4194304.f : 16777216.f) * unw;
      const float za = zz0[mt >> 1] * unw, zb = zz1[mt >> 1] * unw;
      v0 = fmaf(v0, sc, za); v1 = fmaf(v1, sc, zb);
      v2 = fmaf(v2, sc * 0.0625f, za); v3 = fmaf(v3, sc * 0.0625f, zb);
    }
    *reinterpret_cast<float2*>(wo + c0 * 8 + 2 * tig) = make_float2(v0, v1);
    *reinterpret_cast<float2*>(wo + c1 * 8 + 2 * tig) = make_float2(v2, v3);
  }
  __syncthreads();
  // per-warp weights 2^(m_w - M) once, then a plain weighted sum per element
  float* esc = reinterpret_cast<float*>(smem + C::kLps);      // [warps][8] (page list no longer needed)
  float* gmax = esc + kDWarps * 8;                              // [8]
  if (tid < kDWarps * 8) {
    const int w = tid >> 3, g = tid & 7;
    float M = -INFINITY;
#pragma unroll
    for (int v = 0; v < kDWarps; ++v) M = fmaxf(M, scr[v * (16 + 8 * D) + g]);
    const float mw = scr[w * (16 + 8 * D) + g];
    esc[tid] = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
    if (w == 0) gmax[g] = M;
  }
  __syncthreads();
  // element (column g, channel ch), g fastest: the reads follow the [D][8]
  // order, and each warp's stores fill 32-byte runs of a few partial rows
  const int gv = kPacked ? G * cs.nrows : G;              // columns in use (<= 8)
  const int gsh = gv > 4 ? 3 : (gv > 2 ? 2 : (gv > 1 ? 1 : 0));
  for (int idx = tid; idx < (D << gsh); idx += kDThreads) {
    const int g = idx & ((1 << gsh) - 1), ch = idx >> gsh;
    if (g >= gv) continue;
    float Os = 0.f;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) Os = fmaf(esc[w * 8 + g], scr[w * (16 + 8 * D) + 16 + ch * 8 + g], Os);
    float* dst = p.part +
                 ((static_cast<size_t>(kPacked ? b + g / G : b) * p.hq + qh0 + (kPacked ? g % G : g)) *
                      p.n_splits + split) * (D + 2);
    if (ch == 0) {
      float Ls = 0.f;
#pragma unroll
      for (int w = 0; w < kDWarps; ++w) Ls = fmaf(esc[w * 8 + g], scr[w * (16 + 8 * D) + 8 + g], Ls);
      dst[0] = gmax[g];
      dst[1] = Ls;
    }
    dst[2 + ch] = Os;
  }
}

// ---------------------------------------------------------------- combine

constexpr int kMaxSplits = 2048;

// One CTA per KV head h and (batch row, query head of h) pair, or, with
// kMulti, per run of pairs: then the CTA loads its share of R_V once and merges
// its pairs one after another (many rows per KV head).  Per pair, warp 0 finds the global max and the split weights w_s = 2^(m_s - M);
// all threads then sum the weighted split outputs channel by channel
// (coalesced, many loads in flight), and the INT2 part is rotated back once:
// out = (o_raw + o_rot R_V^T) / l.  With kMulti the next pair's partials are
// requested while the current pair is summed and rotated.  For the rotation each warp
// holds RPW rows of R_V (a lane VPL columns of each) and reduces its RPW
// partial dot products across the lanes by halving: at every exchange a lane
// keeps half of its rows and adds the partner's half, so RPW sums take
// RPW - 1 + log2(32 / RPW) + 1 shuffles instead of 5 RPW.
template <int D, bool kBf16Only, bool kMulti>
__global__ void __launch_bounds__(256, kBf16Only ? 4 : 2) combine_kernel(const DecodeParams p) {
  constexpr int RPW = D / 8;              // output rows per warp
  constexpr int VPL = D / 32;             // R_V entries per lane per row
  constexpr int SG = 256 / D;             // split groups summed in parallel
  constexpr int MAXR = 24;                // split outputs a thread holds in registers
  __shared__ float wsplit[kMaxSplits];
  __shared__ float acc_rot[SG][D];
  __shared__ float acc_raw[SG][D];
  __shared__ float orot[D];
  __shared__ float lsum[2];               // by pair parity (read after the next pair began)
  const int h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // this CTA's pairs [q0, q1): pair q is query head h * G + q % G of row q / G
  const int npairs = p.batch * p.G;
  const int q0 = kMulti ? static_cast<int>(static_cast<int64_t>(blockIdx.x) * npairs / gridDim.x)
                        : static_cast<int>(blockIdx.x);
  const int q1 = kMulti ? static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * npairs / gridDim.x)
                        : q0 + 1;
  float rv[kBf16Only ? 1 : RPW][VPL];
  if (!kBf16Only) {   // R_V does not depend on the previous kernel
    const float* r = p.r_v + static_cast<size_t>(h) * D * D;
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const int i = warp * RPW + k;
#pragma unroll
      for (int u = 0; u < VPL; ++u) rv[k][u] = r[i * D + lane * VPL + u];
    }
  }
  pdl_wait();
  pdl_trigger();
  if (q0 >= q1) return;
  const int ns = p.n_splits;
  const int n_rot = kBf16Only ? 0 : p.n_main;
  const int ch = tid % D, sg = tid / D;
  auto part_of = [&](int q) {
    return p.part + (static_cast<size_t>(q / p.G) * p.hq + h * p.G + q % p.G) * ns * (D + 2);
  };
  // every load of a pair that does not need its weights, in one round trip
  float ov[MAXR], mv[2], lv[2];
  auto request = [&](const float* base) {
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
      const int sp = sg + r * SG;
      ov[r] = sp < ns ? base[sp * (D + 2) + 2 + ch] : 0.f;
    }
    if (warp == 0) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int sp = lane + 32 * r;
        mv[r] = sp < ns ? base[sp * (D + 2)] : -INFINITY;
        lv[r] = sp < ns ? base[sp * (D + 2) + 1] : 0.f;
      }
    }
  };
  request(part_of(q0));
  for (int q = q0; q < q1; ++q) {
    const float* base = part_of(q);
    if (warp == 0) {
      float M = fmaxf(mv[0], mv[1]);
      for (int sp = lane + 64; sp < ns; sp += 32) M = fmaxf(M, base[sp * (D + 2)]);
      M = warp_max(M);
      float Ls = 0.f;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int sp = lane + 32 * r;
        if (sp < ns) {
          const float w = (mv[r] == -INFINITY) ? 0.f : exp2f(mv[r] - M);
          wsplit[sp] = w;
          Ls = fmaf(w, lv[r], Ls);
        }
      }
      for (int sp = lane + 64; sp < ns; sp += 32) {
        const float ms = base[sp * (D + 2)];
        const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
        wsplit[sp] = w;
        Ls = fmaf(w, base[sp * (D + 2) + 1], Ls);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      if (lane == 0) lsum[q & 1] = Ls;
    }
    __syncthreads();
    {
      float ar = 0.f, aw = 0.f;
#pragma unroll
      for (int r = 0; r < MAXR; ++r) {
        const int sp = sg + r * SG;
        if (sp < ns) {
          const float v = wsplit[sp] * ov[r];
          if (sp < n_rot) ar += v; else aw += v;
        }
      }
      for (int sp = sg + MAXR * SG; sp < ns; sp += SG) {
        const float v = wsplit[sp] * base[sp * (D + 2) + 2 + ch];
        if (sp < n_rot) ar += v; else aw += v;
      }
      acc_rot[sg][ch] = ar;
      acc_raw[sg][ch] = aw;
    }
    if (kMulti && q + 1 < q1) request(part_of(q + 1));   // in flight while this pair finishes
    __syncthreads();
    if (tid < D) {
      float ar = 0.f, aw = 0.f;
#pragma unroll
      for (int k = 0; k < SG; ++k) { ar += acc_rot[k][tid]; aw += acc_raw[k][tid]; }
      orot[tid] = ar;
      acc_raw[0][tid] = aw;
    }
    __syncthreads();
    const float l = lsum[q & 1];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint16_t* dst = p.out + (static_cast<size_t>(q / p.G) * p.hq + h * p.G + q % p.G) * D;
    if (kBf16Only) {
      if (tid < D) dst[tid] = __bfloat16_as_ushort(__float2bfloat16_rn(acc_raw[0][tid] * inv));
    } else {
      static_assert(RPW == 16 || RPW == 8, "the halving below takes 16 or 8 rows per warp");
      float a[RPW];
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        a[k] = 0.f;
#pragma unroll
        for (int u = 0; u < VPL; ++u) a[k] = fmaf(orot[lane * VPL + u], rv[k][u], a[k]);
      }
      // halving: with n rows left, the lane whose bit `off` is set keeps rows
      // n/2 .. n-1 (its partner rows 0 .. n/2-1) and receives the partner's
      // partial sums of them.  After the exchange at off, row k of the n/2 kept
      // rows is row k + (bit ? n/2 : 0) of the n; in the end lane l holds row
      // (l >> 1) of the warp's (16 rows) or row (l >> 2) (8 rows).
#pragma unroll
      for (int n = RPW, off = 16; n > 1; n >>= 1, off >>= 1) {
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < n / 2; ++k) {
          const float send = up ? a[k] : a[k + n / 2];
          const float keep = up ? a[k + n / 2] : a[k];
          a[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      constexpr int kRest = 32 / RPW;   // lanes still sharing a row: 2 or 4
      float s = a[0];
#pragma unroll
      for (int off = 1; off < kRest; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if ((lane & (kRest - 1)) == 0) {
        const int i = warp * RPW + lane / kRest;
        dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn((acc_raw[0][i] + s) * inv));
      }
    }
    // the next pair rewrites acc_rot / acc_raw / orot only after its first
    // barrier, which every warp reaches after finishing this pair
  }
}

// The combine for many (row, query head) pairs that each have few splits
// (ns <= kRowsMaxSplits: large batches): one CTA per KV head h and run of
// pairs keeps R_V^T in shared memory, and a warp merges kRowsPairs pairs at a
// time entirely in registers.  Lane l owns channels and output rows
// l*CPL .. l*CPL + CPL-1: it reads every split's max and sum (the same words
// for all lanes), weighs its channels of each split output, and forms
// out_i = (o_raw_i + sum_j o_rot_j R_V[i][j]) / l from row j of R_V^T (one
// conflict-free vector read per j, shared by the warp's pairs) and o_rot_j
// broadcast from the warp's shared row.
constexpr int kRowsPairs = 2;
constexpr int kRowsMaxSplits = 4;

template <int D>
constexpr int rows_smem_bytes() {
  return (D * (D + 4) + kDWarps * kRowsPairs * D) * 4;
}

template <int D>
__global__ void __launch_bounds__(256, 2) combine_rows_kernel(const DecodeParams p) {
  constexpr int CPL = D / 32;             // channels (and output rows) per lane
  constexpr int RS = D + 4;               // row stride of R_V^T (spreads the transposing stores)
  constexpr int TP = kRowsPairs;
  constexpr int NSX = kRowsMaxSplits;
  extern __shared__ __align__(16) float rsm[];
  float* rt = rsm;                        // [D][RS]: rt[j][i] = R_V[i][j]
  const int h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  float* orow = rsm + D * RS + warp * TP * D;   // this warp's o_rot rows [TP][D]
  {   // R_V is a constant of the layer: staged before the wait
    const float* r = p.r_v + static_cast<size_t>(h) * D * D;
    for (int e = tid; e < D * D; e += 256) rt[(e % D) * RS + e / D] = r[e];
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int npairs = p.batch * p.G;
  const int q0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * npairs / gridDim.x);
  const int q1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * npairs / gridDim.x);
  const int ns = p.n_splits, n_rot = p.n_main;
  for (int qb = q0 + warp * TP; qb < q1; qb += kDWarps * TP) {
    float ml[TP][NSX][2], ov[TP][NSX][CPL];
    // every load of the warp's pairs in one round trip
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      const int q = qb + t < q1 ? qb + t : qb;   // a spare slot repeats the first pair
      const float* base = p.part + (static_cast<size_t>(q / p.G) * p.hq + h * p.G + q % p.G) * ns * (D + 2);
#pragma unroll
      for (int sx = 0; sx < NSX; ++sx) {
        if (sx < ns) {
          const float* ps = base + sx * (D + 2);
          ml[t][sx][0] = ps[0];
          ml[t][sx][1] = ps[1];
#pragma unroll
          for (int c = 0; c < CPL; c += 2) {
            const float2 v = *reinterpret_cast<const float2*>(ps + 2 + lane * CPL + c);
            ov[t][sx][c] = v.x;
            ov[t][sx][c + 1] = v.y;
          }
        } else {
          ml[t][sx][0] = -INFINITY;
          ml[t][sx][1] = 0.f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) ov[t][sx][c] = 0.f;
        }
      }
    }
    float oraw[TP][CPL], inv[TP];
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      float M = -INFINITY;
#pragma unroll
      for (int sx = 0; sx < NSX; ++sx) M = fmaxf(M, ml[t][sx][0]);
      float L = 0.f, orot[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) orot[c] = oraw[t][c] = 0.f;
#pragma unroll
      for (int sx = 0; sx < NSX; ++sx) {
        const float w = (ml[t][sx][0] == -INFINITY) ? 0.f : exp2f(ml[t][sx][0] - M);
        L = fmaf(w, ml[t][sx][1], L);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          if (sx < n_rot) orot[c] = fmaf(w, ov[t][sx][c], orot[c]);
          else oraw[t][c] = fmaf(w, ov[t][sx][c], oraw[t][c]);
        }
      }
      inv[t] = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int c = 0; c < CPL; c += 2)
        *reinterpret_cast<float2*>(orow + t * D + lane * CPL + c) = make_float2(orot[c], orot[c + 1]);
    }
    __syncwarp();
    float acc[TP][CPL];
#pragma unroll
    for (int t = 0; t < TP; ++t)
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[t][c] = 0.f;
#pragma unroll 2
    for (int j4 = 0; j4 < D; j4 += 4) {
      float4 oj[TP];
#pragma unroll
      for (int t = 0; t < TP; ++t) oj[t] = *reinterpret_cast<const float4*>(orow + t * D + j4);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        float r[CPL];
        if constexpr (CPL == 4) {
          const float4 v = *reinterpret_cast<const float4*>(rt + (j4 + jj) * RS + lane * 4);
          r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(rt + (j4 + jj) * RS + lane * 2);
          r[0] = v.x; r[1] = v.y;
        }
#pragma unroll
        for (int t = 0; t < TP; ++t) {
          const float o = jj == 0 ? oj[t].x : jj == 1 ? oj[t].y : jj == 2 ? oj[t].z : oj[t].w;
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[t][c] = fmaf(o, r[c], acc[t][c]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      const int q = qb + t;
      if (q < q1) {
        uint16_t* dst = p.out + (static_cast<size_t>(q / p.G) * p.hq + h * p.G + q % p.G) * D + lane * CPL;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
          dst[c] = __bfloat16_as_ushort(__float2bfloat16_rn((oraw[t][c] + acc[t][c]) * inv[t]));
      }
    }
    __syncwarp();   // the o_rot rows are rewritten by the next pass
  }
}

// The combine's CTAs per KV head in one wave of resident CTAs (two per SM).
// A head with more (row, query head) pairs than that takes the multi-pair
// form (INT2 only: the BF16 merge has no R_V to share).
inline int combine_wave_per_head(int hkv) {
  return std::max(1, (2 * oscar_host::sm_count() + hkv - 1) / hkv);
}

// ------------------------------------------------------------------- host

struct Plan {
  int n_main, pps, n_splits;
  size_t qrot_bytes, part_off, part_bytes, qrope_off, total;
};

// Split-CTA units per KV head slice for `rows` batch rows of rows_per_seq rows
// per sequence: rows of one sequence share a CTA's 8 query columns, 8 / gq of
// them (gq = query heads per CTA); *rpu receives the rows per unit.
int64_t split_units(const oscar_cache_desc* c, int rows, int rows_per_seq, int* rpu) {
  const int g = c->num_q_heads / c->num_kv_heads;
  const int gq = g < 8 ? g : 8;
  *rpu = rows_per_seq > 1 ? std::max(1, std::min(8 / gq, rows_per_seq)) : 1;
  return static_cast<int64_t>(rows / rows_per_seq) * ((rows_per_seq + *rpu - 1) / *rpu);
}

// n_units: split-CTA units per KV head slice (the batch rows for a decode; fewer
// when rows of a sequence share a CTA)
Plan make_plan(const oscar_cache_desc* c, int batch, int max_len, bool bf16_only,
               int64_t n_units = -1) {
  Plan pl{};
  const int D = c->head_dim;
  int main_pages;
  if (bf16_only) {
    main_pages = (max_len + kPage - 1) / kPage;
  } else {
    const int last = (max_len - c->window > c->sink)
                         ? (max_len - c->window + kPage - 1) / kPage : c->sink / kPage;
    main_pages = last - c->sink / kPage;
  }
  main_pages = std::max(main_pages, 1);
  const int per_sm = bf16_only ? SplitCfg<128, true>::kCtasPerSm : SplitCfg<128, false>::kCtasPerSm;
  // one wave: units * (main splits + the BF16 split) CTAs fill every resident slot
  const int g_all = c->num_q_heads / c->num_kv_heads;
  const int64_t units = (n_units < 0 ? batch : n_units) * c->num_kv_heads * (g_all > 8 ? g_all / 8 : 1);
  const int64_t slots = static_cast<int64_t>(per_sm) * oscar_host::sm_count();
  int n_main = static_cast<int>(std::max<int64_t>(1, slots / units - (bf16_only ? 0 : 1)));
  n_main = std::min(n_main, main_pages);
  n_main = std::max(n_main, (main_pages + kMaxCtaPages - 1) / kMaxCtaPages);
  pl.pps = (main_pages + n_main - 1) / n_main;
  pl.n_main = (main_pages + pl.pps - 1) / pl.pps;
  pl.n_splits = pl.n_main + (bf16_only ? 0 : 1);
  pl.qrot_bytes = bf16_only ? 0 : static_cast<size_t>(batch) * c->num_q_heads * D * 4;
  pl.part_off = (pl.qrot_bytes + 255) & ~static_cast<size_t>(255);
  pl.part_bytes = static_cast<size_t>(batch) * c->num_q_heads * pl.n_splits * (D + 2) * 4;
  // the rotated bf16 query of a step with rotary embedding
  pl.qrope_off = (pl.part_off + pl.part_bytes + 255) & ~static_cast<size_t>(255);
  pl.total = pl.qrope_off + static_cast<size_t>(batch) * c->num_q_heads * D * 2;
  return pl;
}

template <typename Kern>
cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       const DecodeParams& p) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int D, bool kBf16Only, int P, bool kPacked = false>
oscar_status run_decode(const DecodeParams& p, const Plan& pl, cudaStream_t st) {
  using C = SplitCfg<D, kBf16Only, P>;
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(split_kernel<D, kBf16Only, P, kPacked>),
                              C::kBytes))
    return OSCAR_ERR_CUDA;
  const dim3 sgrid(pl.n_splits, p.hkv * p.halves, p.units);
  cudaError_t e;
  // every kernel is launched with programmatic stream serialisation: it may
  // start while its predecessor drains, and waits (griddepcontrol.wait) before
  // touching anything the predecessor produces
  if (!kBf16Only) {
    if (!p.after_append) {   // a fused step's append kernel has written q' already
      e = launch_pdl(qrot_kernel<D>, dim3(p.hkv * p.halves, p.batch), dim3(1024), 0, st, p);
      if (e != cudaSuccess) return OSCAR_ERR_CUDA;
    }
    e = launch_pdl(split_kernel<D, kBf16Only, P, kPacked>, sgrid, dim3(kDThreads), C::kBytes, st, p);
  } else {
    e = launch_pdl(split_kernel<D, kBf16Only, P, kPacked>, sgrid, dim3(kDThreads), C::kBytes, st, p);
  }
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  const int npairs = p.batch * p.G, wave = combine_wave_per_head(p.hkv);
  bool multi = false;
  if constexpr (!kBf16Only) multi = npairs > wave;
  if constexpr (!kBf16Only) {
    if (multi && p.n_splits <= kRowsMaxSplits) {
      if (!oscar_host::allow_smem(reinterpret_cast<const void*>(combine_rows_kernel<D>), rows_smem_bytes<D>()))
        return OSCAR_ERR_CUDA;
      e = launch_pdl(combine_rows_kernel<D>, dim3(wave, p.hkv), dim3(256), rows_smem_bytes<D>(), st, p);
    } else if (multi) {
      e = launch_pdl(combine_kernel<D, false, true>, dim3(wave, p.hkv), dim3(256), 0, st, p);
    }
  }
  if (!multi)
    e = launch_pdl(combine_kernel<D, kBf16Only, false>, dim3(npairs, p.hkv), dim3(256), 0, st, p);
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status append_with_query(const oscar_cache_desc* desc, const void* q, const void* k_new,
                               const void* v_new, const int32_t* seq_lens_after, int32_t batch,
                               float* qrot, double rope_log2_base, uint16_t* qrope,
                               cudaStream_t st);

// Host buffers of a step whose inputs and result live in host memory: the
// inputs are copied in after every check has passed and before the first
// kernel, the result is copied out after the last, on the call's stream.
struct HostCopy {
  void* in_dst;
  const void* in_src;
  size_t in_bytes;
  void* out_dst;
  const void* out_src;
  size_t out_bytes;
};

// Argument checks of every decode entry point, in the order the callers rely
// on: descriptor, sizes, pointers and alignment, then the shape limits.  A
// batch of 0 passes (the caller returns OSCAR_OK without launching).
// with_ws: the caller passes a workspace pointer, checked too.
oscar_status decode_args(const oscar_cache_desc* c, const void* q, const int32_t* seq_lens,
                         int batch, int max_len, const void* out, const void* ws, bool bf16_only,
                         bool with_ws = true) {
  oscar_status s = oscar_host::check_desc(c, !bf16_only, true);
  if (s != OSCAR_OK) return s;
  if (batch < 0 || max_len < 1) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  if (!q || !seq_lens || !out) return OSCAR_ERR_INVALID_ARG;
  if (with_ws && (!ws || (reinterpret_cast<uintptr_t>(ws) & 15))) return OSCAR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 3)
    return OSCAR_ERR_INVALID_ARG;
  if (max_len > static_cast<int64_t>(c->max_pages_per_seq) * kPage) return OSCAR_ERR_INVALID_ARG;
  if (!bf16_only &&
      (c->sink + kPage - 1) / kPage + (c->window + kPage - 1) / kPage + 1 > kMaxCtaPages)
    return OSCAR_ERR_UNSUPPORTED;
  return OSCAR_OK;
}

oscar_status decode_entry(const oscar_cache_desc* c, const void* q, const int32_t* seq_lens,
                          int batch, int max_len, void* out, void* ws, size_t ws_bytes,
                          void* stream, bool bf16_only, const void* k_new = nullptr,
                          const void* v_new = nullptr, const int32_t* limits = nullptr,
                          int rows_per_seq = 1, double rope_log2_base = 0.0,
                          const HostCopy* hc = nullptr) {
  oscar_status s = decode_args(c, q, seq_lens, batch, max_len, out, ws, bf16_only);
  if (s != OSCAR_OK || batch == 0) return s;
  int rpu = 1;
  const int64_t n_units = split_units(c, batch, rows_per_seq, &rpu);
  const Plan pl = make_plan(c, batch, max_len, bf16_only, n_units);
  if (pl.n_splits > kMaxSplits) return OSCAR_ERR_UNSUPPORTED;
  if (ws_bytes < pl.total) return OSCAR_ERR_WORKSPACE;
  DecodeParams p{};
  p.hkv = c->num_kv_heads;
  p.hq = c->num_q_heads;
  p.G = c->num_q_heads / c->num_kv_heads;
  p.gq = p.G < 8 ? p.G : 8;
  p.halves = p.G / p.gq;
  p.sink = c->sink;
  p.window = c->window;
  p.max_pages = c->max_pages_per_seq;
  p.n_int2_pages = c->num_int2_pages;
  p.n_bf16_pages = c->num_bf16_pages;
  p.int2_pool = static_cast<const uint8_t*>(c->int2_pool);
  p.bf16_pool = static_cast<const uint8_t*>(c->bf16_pool);
  p.int2_pt = c->int2_page_table;
  p.bf16_pt = c->bf16_page_table;
  p.r_k = c->r_k;
  p.r_v = c->r_v;
  p.clip_k = c->clip_k;
  p.clip_v = c->clip_v;
  p.status = c->status;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.seq_lens = seq_lens;
  p.batch = batch;   // rows: sequences x rows_per_seq
  p.rows_per_seq = rows_per_seq;
  p.rpu = rpu;
  p.units = static_cast<int>(n_units);
  p.limits = limits;
  p.max_len = max_len;
  p.n_main = pl.n_main;
  p.pps = pl.pps;
  p.n_splits = pl.n_splits;
  p.qrot = reinterpret_cast<float*>(ws);
  p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.part_off);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c->head_dim)));
  p.wait_first = bf16_only ? 1 : 0;   // the INT2 call is gated by qrot_kernel
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (hc && cudaMemcpyAsync(hc->in_dst, hc->in_src, hc->in_bytes, cudaMemcpyHostToDevice, st) !=
                cudaSuccess)
    return OSCAR_ERR_CUDA;
  if (k_new) {   // fused step: the append kernel writes q' and gates the split kernel
    p.after_append = 1;
    uint16_t* qrope = nullptr;
    if (rope_log2_base > 0.0) {   // the split kernel's BF16 pages take the rotated query
      qrope = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + pl.qrope_off);
      p.q = qrope;
    }
    const oscar_status a =
        append_with_query(c, q, k_new, v_new, seq_lens, batch, p.qrot, rope_log2_base, qrope, st);
    if (a != OSCAR_OK) return a;
  }
  const bool int4 = oscar_host::code_planes(c) == 2;
  const bool packed = rpu > 1;
  oscar_status r;
  if (c->head_dim == 128) {
    if (bf16_only) r = run_decode<128, true, 1>(p, pl, st);
    else if (packed)
      r = int4 ? run_decode<128, false, 2, true>(p, pl, st) : run_decode<128, false, 1, true>(p, pl, st);
    else
      r = int4 ? run_decode<128, false, 2>(p, pl, st) : run_decode<128, false, 1>(p, pl, st);
  } else {
    if (bf16_only) r = run_decode<64, true, 1>(p, pl, st);
    else if (packed)
      r = int4 ? run_decode<64, false, 2, true>(p, pl, st) : run_decode<64, false, 1, true>(p, pl, st);
    else
      r = int4 ? run_decode<64, false, 2>(p, pl, st) : run_decode<64, false, 1>(p, pl, st);
  }
  if (r == OSCAR_OK && hc &&
      cudaMemcpyAsync(hc->out_dst, hc->out_src, hc->out_bytes, cudaMemcpyDeviceToHost, st) !=
          cudaSuccess)
    return OSCAR_ERR_CUDA;
  return r;
}

// Staging of a step with host buffers: the inputs (q, k_new, v_new, in the
// caller's host order) from byte 0, the output from the next multiple of 256.
struct HostStaging {
  size_t q_bytes, kv_bytes, in_bytes, out_off, out_bytes, total;
};

inline HostStaging host_staging(const oscar_cache_desc* c, int batch) {
  HostStaging h{};
  const size_t b = static_cast<size_t>(batch), d = static_cast<size_t>(c->head_dim);
  h.q_bytes = b * c->num_q_heads * d * 2;
  h.kv_bytes = b * c->num_kv_heads * d * 2;
  h.in_bytes = h.q_bytes + 2 * h.kv_bytes;
  h.out_off = (h.in_bytes + 255) / 256 * 256;
  h.out_bytes = h.q_bytes;
  h.total = h.out_off + h.out_bytes;
  return h;
}

}  // namespace oscar

namespace oscar_host {

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

// The device address of host range [p, p + bytes) when it is page-locked memory
// mapped into the device's address space (cudaHostAlloc memory under unified
// addressing, or cudaHostRegister'ed with mapping) and its first and last bytes
// map to one contiguous device range; null otherwise (a query error is cleared).
const void* mapped_range(const void* p, size_t bytes) {
  if (!p || bytes == 0) return nullptr;
  cudaPointerAttributes a{}, b{};
  const uint8_t* last = static_cast<const uint8_t*>(p) + (bytes - 1);
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess ||
      cudaPointerGetAttributes(&b, last) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || b.type != cudaMemoryTypeHost || !a.devicePointer ||
      !b.devicePointer)
    return nullptr;
  if (static_cast<const uint8_t*>(b.devicePointer) !=
      static_cast<const uint8_t*>(a.devicePointer) + (bytes - 1))
    return nullptr;
  return a.devicePointer;
}

bool allow_smem(const void* func, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;   // (function, device)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& d : done)
    if (d.first == func && d.second == dev) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  done.emplace_back(func, dev);
  return true;
}

}  // namespace oscar_host

// ------------------------------------------------ workspace without allocation
//
// Some callers cannot allocate device memory at the moment they need attention:
// plug-ins hosted by a runtime that owns every allocation, or latency-bound
// loops that must never enter the allocator (it may synchronise, or fail under
// memory pressure).  For them the library carries one fixed scratch buffer in
// its own image.  Every GPU that loads the library reserves it until the
// process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[size_t(16) << 20];   // 16 MiB

namespace oscar {

constexpr size_t kStaticScratchBytes = sizeof(g_decode_scratch);

// The current CUDA context's unique id (cuCtxGetId through the runtime's driver
// entry points, so the library does not link the driver library); 0 when it
// cannot be had.  Ids are never reused, unlike context handles.
unsigned long long current_context_id() {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static const std::pair<GetCurrent, GetId> fns = [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa{}, qb{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) !=
            cudaSuccess || qa != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
            cudaSuccess || qb != cudaDriverEntryPointSuccess)
      return std::make_pair(static_cast<GetCurrent>(nullptr), static_cast<GetId>(nullptr));
    return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
  }();
  if (!fns.first || !fns.second) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (fns.first(&ctx) != CUDA_SUCCESS || !ctx || fns.second(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch buffer in the current device's context.  In
// host code the symbol is only a handle; cudaGetSymbolAddress, called with the
// device current, yields the address the kernels are given.  It is looked up
// once per context: a context that was destroyed and created again (after
// cudaDeviceReset, say) reloads the library's module, so the address is looked
// up afresh rather than taken from a cache keyed on the device index alone.
void* decode_scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (addr[dev] && ctx != 0 && ctx_of[dev] == ctx) return addr[dev];
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
  addr[dev] = ptr;
  ctx_of[dev] = current_context_id();   // the lookup has made the context current
  return addr[dev];
}

}  // namespace oscar

extern "C" {

size_t oscar_decode_workspace_size(const oscar_cache_desc* desc, int32_t batch, int32_t max_seq_len) {
  if (oscar_host::check_desc(desc, false, false) != OSCAR_OK || batch < 1 || max_seq_len < 1)
    return 0;
  const oscar::Plan a = oscar::make_plan(desc, batch, max_seq_len, false);
  const oscar::Plan b = oscar::make_plan(desc, batch, max_seq_len, true);
  return std::max(a.total, b.total);
}

oscar_status oscar_decode_attention(const oscar_cache_desc* desc, const void* q,
                                    const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  return oscar::decode_entry(desc, q, seq_lens, batch, max_seq_len, out, workspace,
                             workspace_bytes, stream, false);
}

oscar_status oscar_decode_attention_bf16(const oscar_cache_desc* desc, const void* q,
                                         const int32_t* seq_lens, int32_t batch,
                                         int32_t max_seq_len, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  return oscar::decode_entry(desc, q, seq_lens, batch, max_seq_len, out, workspace,
                             workspace_bytes, stream, true);
}

int32_t oscar_device_sm_count(void) { return oscar_host::sm_count(); }

size_t oscar_multiquery_workspace_size(const oscar_cache_desc* desc, int32_t batch, int32_t m_rows,
                                       int32_t max_seq_len) {
  if (oscar_host::check_desc(desc, false, false) != OSCAR_OK || batch < 1 || m_rows < 1 ||
      max_seq_len < 1 || static_cast<int64_t>(batch) * m_rows > (int64_t(1) << 30))
    return 0;
  int rpu = 1;
  const int64_t units = oscar::split_units(desc, batch * m_rows, m_rows, &rpu);
  return oscar::make_plan(desc, batch * m_rows, max_seq_len, false, units).total;
}

oscar_status oscar_multiquery_attention(const oscar_cache_desc* desc, const void* q,
                                        const int32_t* seq_lens, const int32_t* q_pos,
                                        int32_t batch, int32_t m_rows, int32_t max_seq_len,
                                        void* out, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (batch < 0 || m_rows < 1 || !q_pos) return OSCAR_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * m_rows > (int64_t(1) << 30)) return OSCAR_ERR_INVALID_ARG;
  return oscar::decode_entry(desc, q, seq_lens, batch * m_rows, max_seq_len, out, workspace,
                             workspace_bytes, stream, false, nullptr, nullptr, q_pos, m_rows);
}

oscar_status oscar_decode_step(const oscar_cache_desc* desc, const void* q, const void* k_new,
                               const void* v_new, const int32_t* seq_lens_after, int32_t batch,
                               int32_t max_seq_len, void* out, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (batch > 0 && (!k_new || !v_new)) return OSCAR_ERR_INVALID_ARG;
  return oscar::decode_entry(desc, q, seq_lens_after, batch, max_seq_len, out, workspace,
                             workspace_bytes, stream, false, batch > 0 ? k_new : nullptr, v_new);
}

oscar_status oscar_decode_step_rope(const oscar_cache_desc* desc, const void* q, const void* k_new,
                                    const void* v_new, const int32_t* seq_lens_after,
                                    int32_t batch, int32_t max_seq_len, double rope_base,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!(rope_base > 1.0) || !std::isfinite(rope_base)) return OSCAR_ERR_INVALID_ARG;
  if (batch > 0 && (!k_new || !v_new)) return OSCAR_ERR_INVALID_ARG;
  return oscar::decode_entry(desc, q, seq_lens_after, batch, max_seq_len, out, workspace,
                             workspace_bytes, stream, false, batch > 0 ? k_new : nullptr, v_new,
                             nullptr, 1, std::log2(rope_base));
}

size_t oscar_decode_step_host_staging_size(const oscar_cache_desc* desc, int32_t batch) {
  if (oscar_host::check_desc(desc, false, false) != OSCAR_OK || batch < 1) return 0;
  return oscar::host_staging(desc, batch).total;
}

oscar_status oscar_decode_step_host(const oscar_cache_desc* desc, const void* in_host,
                                    const int32_t* seq_lens_after, int32_t batch,
                                    int32_t max_seq_len, double rope_base, void* out_host,
                                    void* staging, size_t staging_bytes, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  oscar_status st = oscar_host::check_desc(desc, true, true);
  if (st != OSCAR_OK) return st;
  if (batch < 0 || max_seq_len < 1) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  if (!(rope_base >= 0.0) || !std::isfinite(rope_base) || (rope_base > 0.0 && !(rope_base > 1.0)))
    return OSCAR_ERR_INVALID_ARG;
  if (!in_host || !out_host || !staging) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(staging) & 15) return OSCAR_ERR_INVALID_ARG;
  const oscar::HostStaging h = oscar::host_staging(desc, batch);
  if (staging_bytes < h.total) return OSCAR_ERR_WORKSPACE;
  const double lb = rope_base > 0.0 ? std::log2(rope_base) : 0.0;
  // Page-locked host buffers mapped into the device's address space are read
  // and written by the kernels in place (over the CPU-GPU link, no copy-engine
  // hop); any other host memory goes through the staging copies.
  const uint8_t* in_dev = static_cast<const uint8_t*>(oscar_host::mapped_range(in_host, h.in_bytes));
  uint8_t* out_dev =
      static_cast<uint8_t*>(const_cast<void*>(oscar_host::mapped_range(out_host, h.out_bytes)));
  uint8_t* sg = static_cast<uint8_t*>(staging);
  if (in_dev && out_dev && (reinterpret_cast<uintptr_t>(in_dev) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(out_dev) & 3) == 0)
    return oscar::decode_entry(desc, in_dev, seq_lens_after, batch, max_seq_len, out_dev,
                               workspace, workspace_bytes, stream, false, in_dev + h.q_bytes,
                               in_dev + h.q_bytes + h.kv_bytes, nullptr, 1, lb);
  const oscar::HostCopy hc{sg, in_host, h.in_bytes, out_host, sg + h.out_off, h.out_bytes};
  return oscar::decode_entry(desc, sg, seq_lens_after, batch, max_seq_len, sg + h.out_off,
                             workspace, workspace_bytes, stream, false, sg + h.q_bytes,
                             sg + h.q_bytes + h.kv_bytes, nullptr, 1, lb, &hc);
}

oscar_status oscar_decode_attention_static(const oscar_cache_desc* desc, const void* q,
                                           const int32_t* seq_lens, int32_t batch,
                                           int32_t max_seq_len, void* out, void* stream) {
  // the workspace call's argument checks first (the scratch stands in for the
  // workspace pointer), so an invalid argument is reported as such
  oscar_status st = oscar::decode_args(desc, q, seq_lens, batch, max_seq_len, out, nullptr, false,
                                       false);
  if (st != OSCAR_OK || batch == 0) return st;
  // the same plan the workspace call makes; refuse it if it needs more scratch
  const oscar::Plan pl = oscar::make_plan(desc, batch, max_seq_len, false);
  if (pl.total > oscar::kStaticScratchBytes) return OSCAR_ERR_WORKSPACE;
  void* ws = oscar::decode_scratch_address();
  if (!ws) return OSCAR_ERR_CUDA;
  // every byte the kernels read from the scratch is written earlier in the same
  // call (rotated queries, one partial per split), so nothing is cleared
  return oscar::decode_entry(desc, q, seq_lens, batch, max_seq_len, out, ws,
                             oscar::kStaticScratchBytes, stream, false);
}

}  // extern "C"
