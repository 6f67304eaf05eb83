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
  int64_t n_int2_pages, n_bf16_pages;
  const uint8_t* int2_pool;
  const uint8_t* bf16_pool;
  const int32_t* int2_pt;
  const int32_t* bf16_pt;
  const float* r_k;
  const float* r_v;
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
};

// ------------------------------------------------------------------ q R_K

template <int D>
__global__ void __launch_bounds__(1024) qrot_kernel(const DecodeParams p) {
  pdl_trigger();
  __shared__ float qs[8][D];
  __shared__ float partial[1024 / D][8][D];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int G = p.G;
  for (int i = tid; i < G * D; i += blockDim.x)
    qs[i / D][i % D] = bf16_to_float(p.q[(static_cast<size_t>(b) * p.hq + h * G) * D + i]);
  __syncthreads();
  constexpr int CH = 1024 / D;          // chunks of the contraction index
  constexpr int PER = D / CH;
  const int j = tid % D, c = tid / D;
  const float* r = p.r_k + static_cast<size_t>(h) * D * D;
  float rv[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) rv[u] = r[(c * PER + u) * D + j];
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
    p.qrot[(static_cast<size_t>(b) * p.hq + h * G + g) * D + jj] = acc;
  }
}

// ---------------------------------------------------------------- split-K

template <int D, bool kBf16Only>
struct SplitCfg {
  static constexpr int kStagesI = 6;                     // INT2 ring depth per warp
  static constexpr int kStagesB = kBf16Only ? 3 : 1;     // BF16 ring depth per warp
  static constexpr int kRingI = kDWarps * kStagesI * Fmt<D>::kInt2Block;
  static constexpr int kRingB = kDWarps * kStagesB * Fmt<D>::kBf16Block;
  static constexpr int kRing = kBf16Only ? kRingB : (kRingI > kRingB ? kRingI : kRingB);
  static constexpr int kScratch = kDWarps * (16 + 8 * D) * 4;
  static_assert(kScratch <= kRing, "merge scratch reuses the ring");
  static constexpr int kIds = 0;                                      // int [kMaxCtaPages]
  static constexpr int kLps = kIds + kMaxCtaPages * 4;               // int [kMaxCtaPages]
  static constexpr int kBars = kLps + kMaxCtaPages * 4;              // u64 [warps][stages]
  static constexpr int kRingOff = kBars + kDWarps * 8 * 8;
  static constexpr int kBytes = kRingOff + kRing;
  static constexpr int kCtasPerSm = kBf16Only ? 1 : 2;
};

struct Softmax {
  float m0, m1, l0, l1;   // running max (log2 domain) and partial sum for g = 2tig, 2tig+1
};

// Online-softmax update for one 16-token tile.  l[] are log2-domain logits in
// the m16n8 accumulator layout (rows = tokens gid / gid+8, cols = query heads
// 2tig / 2tig+1).  Rescales the output accumulators when the max grows and
// returns the probabilities in p[].
template <int NT>
__device__ __forceinline__ void softmax_tile(Softmax& st, float (&l)[4], float (&o)[NT][4],
                                             float (&z)[4], float (&pr)[4]) {
  float mx0 = fmaxf(l[0], l[2]), mx1 = fmaxf(l[1], l[3]);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const float n0 = fmaxf(st.m0, mx0), n1 = fmaxf(st.m1, mx1);
  if (n0 > st.m0 || n1 > st.m1) {
    const float a0 = (n0 == st.m0) ? 1.f : exp2f(st.m0 - n0);
    const float a1 = (n1 == st.m1) ? 1.f : exp2f(st.m1 - n1);
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
  pr[0] = exp2f(l[0] - b0);
  pr[1] = exp2f(l[1] - b1);
  pr[2] = exp2f(l[2] - b0);
  pr[3] = exp2f(l[3] - b1);
  st.l0 += pr[0] + pr[2];
  st.l1 += pr[1] + pr[3];
}

__device__ __forceinline__ bool tok_ok(int t, int L, int sink, int window, int mode) {
  // mode 0: INT2 region; 1: BF16 region (sink + recent); 2: all tokens
  if (mode == 0) return t >= sink && t < L - window;
  if (mode == 1) return t < L && (t < sink || t >= L - window);
  return t < L;
}

template <int D, bool kBf16Only>
__global__ void __launch_bounds__(kDThreads, SplitCfg<D, kBf16Only>::kCtasPerSm)
    split_kernel(const DecodeParams p) {
  using C = SplitCfg<D, kBf16Only>;
  constexpr int NG = D / 32;     // groups = code words per lane
  constexpr int NK = D / 16;     // k-steps / channel tiles
  extern __shared__ __align__(128) uint8_t smem[];
  int* ids = reinterpret_cast<int*>(smem + C::kIds);
  int* lps = reinterpret_cast<int*>(smem + C::kLps);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint8_t* ring = smem + C::kRingOff;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int G = p.G;

  int L = p.seq_lens[b];
  if (L < 1 || L > p.max_len) {
    if (tid == 0 && p.status) atomicOr(p.status, OSCAR_DEVERR_SEQ_LEN);
    L = 0;
  }
  // ---- which pages this CTA reads
  const bool bf16_split = kBf16Only || split == p.n_main;
  const int mode = kBf16Only ? 2 : (bf16_split ? 1 : 0);
  int n = 0;
  if (mode == 1) {
    // sink pages, then recent pages not already listed
    const int s_end = (min(p.sink, L) + kPage - 1) / kPage;
    const int r_beg = max(p.sink, L - p.window) / kPage;
    const int r_end = (L + kPage - 1) / kPage;
    const int r0 = max(r_beg, s_end);
    const int n_sink = s_end, n_rec = max(0, r_end - r0);
    n = min(n_sink + n_rec, kMaxCtaPages);
    for (int k = tid; k < n; k += kDThreads) lps[k] = k < n_sink ? k : r0 + (k - n_sink);
  } else {
    int first, last;   // logical page span of the main region
    if (mode == 0) {
      first = p.sink / kPage;
      last = (L - p.window > p.sink) ? (L - p.window + kPage - 1) / kPage : first;
    } else {
      first = 0;
      last = (L + kPage - 1) / kPage;
    }
    const int lo = first + split * p.pps;
    const int hi = min(last, lo + p.pps);
    n = max(0, min(hi - lo, kMaxCtaPages));
    for (int k = tid; k < n; k += kDThreads) lps[k] = lo + k;
  }
  __syncthreads();
  {
    const int32_t* pt = (mode == 0 ? p.int2_pt : p.bf16_pt) + static_cast<size_t>(b) * p.max_pages;
    const int64_t npages = mode == 0 ? p.n_int2_pages : p.n_bf16_pages;
    for (int k = tid; k < n; k += kDThreads) {
      const int lp = lps[k];
      int id = lp < p.max_pages ? pt[lp] : -1;
      if (id < 0 || id >= npages) {
        if (p.status) atomicOr(p.status, OSCAR_DEVERR_PAGE_ID);
        id = -1;
      }
      ids[k] = id;
    }
  }
  if (tid < kDWarps * 8) mbar_init(&bars[tid], 1);
  fence_mbar_init();
  __syncthreads();

  // ---- per-warp ring
  const int stage_bytes = mode == 0 ? Fmt<D>::kInt2Block : Fmt<D>::kBf16Block;
  const int n_stages = mode == 0 ? C::kStagesI : C::kStagesB;
  uint8_t* wring = ring + warp * n_stages * stage_bytes;
  uint64_t* wbar = bars + warp * 8;
  const uint8_t* pool = mode == 0 ? p.int2_pool : p.bf16_pool;
  const int my_n = n > warp ? (n - warp + kDWarps - 1) / kDWarps : 0;

  auto issue = [&](int i) {
    const int id = ids[warp + kDWarps * i];
    if (id < 0) return;
    const int s = i % n_stages;
    fence_proxy_async();
    mbar_arrive_expect_tx(&wbar[s], stage_bytes);
    bulk_g2s(wring + s * stage_bytes,
             pool + (static_cast<size_t>(id) * p.hkv + h) * stage_bytes, stage_bytes, &wbar[s]);
  };
  if (lane == 0)
    for (int i = 0; i < min(n_stages, my_n); ++i) issue(i);

  // ---- query operand (B fragments), after the producer of q' has finished
  pdl_wait();
  uint32_t qb[NK][2];
  uint32_t qz = 0;
  const float scale_log2 = p.scale_log2;
  if (mode == 0) {
    const float* qr = p.qrot + (static_cast<size_t>(b) * p.hq + h * G + gid) * D;
    float gs[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) gs[g] = 0.f;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
      if (gid < G) {
        v0 = *reinterpret_cast<const float2*>(qr + 16 * kk + 2 * tig);
        v1 = *reinterpret_cast<const float2*>(qr + 16 * kk + 2 * tig + 8);
      }
      gs[kk >> 1] += (v0.x + v0.y) + (v1.x + v1.y);
      const float sc = (kk & 1) ? 0.25f : 1.f;   // odd k-steps read codes at 4x
      qb[kk][0] = pack_half2(v0.x * sc, v0.y * sc);
      qb[kk][1] = pack_half2(v1.x * sc, v1.y * sc);
    }
    float mine = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      gs[g] += __shfl_xor_sync(0xffffffffu, gs[g], 1);
      gs[g] += __shfl_xor_sync(0xffffffffu, gs[g], 2);
      if (g == tig) mine = gs[g];
    }
    if (tig < NG) {
      const __half hi = __float2half_rn(mine);
      const __half lo = __float2half_rn(mine - __half2float(hi));
      qz = static_cast<uint32_t>(__half_as_ushort(hi)) |
           (static_cast<uint32_t>(__half_as_ushort(lo)) << 16);
    }
  } else {
    const uint16_t* qr = p.q + (static_cast<size_t>(b) * p.hq + h * G + gid) * D;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) {
      qb[kk][0] = gid < G ? *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * tig) : 0u;
      qb[kk][1] = gid < G ? *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * tig + 8) : 0u;
    }
  }

  float o[NK][4];
#pragma unroll
  for (int t = 0; t < NK; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float zacc[4] = {0.f, 0.f, 0.f, 0.f};
  Softmax sm{-INFINITY, -INFINITY, 0.f, 0.f};
  uint32_t phase = 0;
  const float ks = scale_log2 * 16777216.f;   // codes are read as code * 2^-24

  for (int i = 0; i < my_n; ++i) {
    const int k = warp + kDWarps * i;
    const int s = i % n_stages;
    if (ids[k] >= 0) {
      const bool ok = mbar_wait(&wbar[s], (phase >> s) & 1u, p.status);
      phase ^= 1u << s;
      if (__any_sync(0xffffffffu, !ok)) {
        // give the copies still in flight a bounded chance to land, then stop
        for (int j = i + 1; j < min(i + n_stages, my_n); ++j)
          if (ids[warp + kDWarps * j] >= 0) {
            const int sj = j % n_stages;
            mbar_wait(&wbar[sj], (phase >> sj) & 1u, p.status);
            phase ^= 1u << sj;
          }
        break;
      }
      const uint8_t* st = wring + s * stage_bytes;
      const int t0 = lps[k] * kPage + gid, t1 = t0 + 8;
      float lg[4], pr[4];
      if (mode == 0) {
        // ---- q.K over exact 2-bit codes, per-group accumulators
        uint32_t kw[NG];
        if constexpr (NG == 4) {
          const uint4 v = reinterpret_cast<const uint4*>(st + Fmt<D>::kKc)[lane];
          kw[0] = v.x; kw[1] = v.y; kw[2] = v.z; kw[3] = v.w;
        } else {
          const uint2 v = reinterpret_cast<const uint2*>(st + Fmt<D>::kKc)[lane];
          kw[0] = v.x; kw[1] = v.y;
        }
        float dg[NG][4];
#pragma unroll
        for (int m = 0; m < NG; ++m) {
          dg[m][0] = dg[m][1] = dg[m][2] = dg[m][3] = 0.f;
          const uint32_t w0 = kw[m], w1 = w0 >> 4, w2 = w0 >> 8, w3 = w0 >> 12;
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            const uint32_t mask = 0x00030003u << (2 * ii);
            // A registers a0..a3 hold (s = 0, 2, 1, 3) for keys
            mma_f16(dg[m], w0 & mask, w2 & mask, w1 & mask, w3 & mask, qb[2 * m + ii][0],
                    qb[2 * m + ii][1]);
          }
        }
        const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st + Fmt<D>::kKsz);
        uint32_t za = 0, zb = 0;
        if (tig < NG) {
          const uint32_t e0 = ksz[gid * NG + tig], e1 = ksz[(gid + 8) * NG + tig];
          za = __byte_perm(e0, e0, 0x3232);
          zb = __byte_perm(e1, e1, 0x3232);
        }
        float zq[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(zq, za, zb, 0u, 0u, qz, 0u);
        uint32_t sa[NG], sb[NG];
        if constexpr (NG == 4) {
          const uint4 a = reinterpret_cast<const uint4*>(ksz)[gid];
          const uint4 c = reinterpret_cast<const uint4*>(ksz)[gid + 8];
          sa[0] = a.x; sa[1] = a.y; sa[2] = a.z; sa[3] = a.w;
          sb[0] = c.x; sb[1] = c.y; sb[2] = c.z; sb[3] = c.w;
        } else {
          const uint2 a = reinterpret_cast<const uint2*>(ksz)[gid];
          const uint2 c = reinterpret_cast<const uint2*>(ksz)[gid + 8];
          sa[0] = a.x; sa[1] = a.y;
          sb[0] = c.x; sb[1] = c.y;
        }
        lg[0] = zq[0] * scale_log2; lg[1] = zq[1] * scale_log2;
        lg[2] = zq[2] * scale_log2; lg[3] = zq[3] * scale_log2;
#pragma unroll
        for (int m = 0; m < NG; ++m) {
          const float fa = half_lo(sa[m]) * ks, fb = half_lo(sb[m]) * ks;
          lg[0] = fmaf(fa, dg[m][0], lg[0]);
          lg[1] = fmaf(fa, dg[m][1], lg[1]);
          lg[2] = fmaf(fb, dg[m][2], lg[2]);
          lg[3] = fmaf(fb, dg[m][3], lg[3]);
        }
      } else {
        // ---- q.K over bf16 keys
        float dk[4] = {0.f, 0.f, 0.f, 0.f};
        const uint4* kb = reinterpret_cast<const uint4*>(st);
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
          const uint4 a = kb[kk * 32 + lane];
          mma_bf16(dk, a.x, a.y, a.z, a.w, qb[kk][0], qb[kk][1]);
        }
        lg[0] = dk[0] * scale_log2; lg[1] = dk[1] * scale_log2;
        lg[2] = dk[2] * scale_log2; lg[3] = dk[3] * scale_log2;
      }
      // mask tokens outside this CTA's region (only on boundary pages)
      const int pbeg = lps[k] * kPage;
      const bool whole = mode == 2 ? (pbeg + kPage <= L)
                       : mode == 0 ? (pbeg >= p.sink && pbeg + kPage <= L - p.window)
                                   : false;
      if (!whole) {
        if (!tok_ok(t0, L, p.sink, p.window, mode)) lg[0] = lg[1] = -INFINITY;
        if (!tok_ok(t1, L, p.sink, p.window, mode)) lg[2] = lg[3] = -INFINITY;
      }
      softmax_tile<NK>(sm, lg, o, zacc, pr);

      if (mode == 0) {
        const uint32_t pb0 = movmatrix_trans(pack_half2(pr[0], pr[1]));
        const uint32_t pb1 = movmatrix_trans(pack_half2(pr[2], pr[3]));
        uint32_t vw[NG], vs0[NG], vs1[NG];
        const uint32_t* vsw = reinterpret_cast<const uint32_t*>(st + Fmt<D>::kVs);
        if constexpr (NG == 4) {
          const uint4 v = reinterpret_cast<const uint4*>(st + Fmt<D>::kVc)[lane];
          vw[0] = v.x; vw[1] = v.y; vw[2] = v.z; vw[3] = v.w;
          const uint4 a = reinterpret_cast<const uint4*>(vsw)[tig * 2];
          const uint4 c = reinterpret_cast<const uint4*>(vsw)[tig * 2 + 1];
          vs0[0] = a.x; vs0[1] = a.y; vs0[2] = a.z; vs0[3] = a.w;
          vs1[0] = c.x; vs1[1] = c.y; vs1[2] = c.z; vs1[3] = c.w;
        } else {
          const uint2 v = reinterpret_cast<const uint2*>(st + Fmt<D>::kVc)[lane];
          vw[0] = v.x; vw[1] = v.y;
          const uint2 a = reinterpret_cast<const uint2*>(vsw)[tig * 2];
          const uint2 c = reinterpret_cast<const uint2*>(vsw)[tig * 2 + 1];
          vs0[0] = a.x; vs0[1] = a.y;
          vs1[0] = c.x; vs1[1] = c.y;
        }
#pragma unroll
        for (int m = 0; m < NG; ++m) {
          const uint32_t bb0 = hmul2_u32(pb0, vs0[m]);
          const uint32_t bb1 = hmul2_u32(pb1, vs1[m]);
          const uint32_t w0 = vw[m], w1 = w0 >> 4, w2 = w0 >> 8, w3 = w0 >> 12;
#pragma unroll
          for (int ii = 0; ii < 2; ++ii) {
            const uint32_t mask = 0x00030003u << (2 * ii);
            mma_f16(o[2 * m + ii], w0 & mask, w1 & mask, w2 & mask, w3 & mask, bb0, bb1);
          }
        }
        const uint32_t* vz = reinterpret_cast<const uint32_t*>(st + Fmt<D>::kVz);
        uint32_t za0 = 0, za2 = 0;
        if (gid < NG) {
          za0 = vz[(tig * 2) * NG + gid];
          za2 = vz[(tig * 2 + 1) * NG + gid];
        }
        mma_f16(zacc, za0, 0u, za2, 0u, pb0, pb1);
      } else {
        const uint32_t pb0 = movmatrix_trans(pack_bf162(pr[0], pr[1]));
        const uint32_t pb1 = movmatrix_trans(pack_bf162(pr[2], pr[3]));
        const uint4* vb = reinterpret_cast<const uint4*>(st + Fmt<D>::kBf16V);
#pragma unroll
        for (int mt = 0; mt < NK; ++mt) {
          const uint4 a = vb[mt * 32 + lane];
          mma_bf16(o[mt], a.x, a.y, a.z, a.w, pb0, pb1);
        }
      }
    }
    __syncwarp();
    if (lane == 0 && i + n_stages < my_n) issue(i + n_stages);
  }

  pdl_trigger();

  // ---- warp result -> shared scratch (the ring is idle once every warp is here)
  float l0 = sm.l0, l1 = sm.l1;
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  float zz0[NG], zz1[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    zz0[g] = __shfl_sync(0xffffffffu, zacc[0], g * 4 + tig);
    zz1[g] = __shfl_sync(0xffffffffu, zacc[1], g * 4 + tig);
  }
  __syncthreads();
  float* scr = reinterpret_cast<float*>(ring);
  float* wm = scr + warp * (16 + 8 * D);   // [8] max, [8] sum, [8][D] output
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
      const float sc = (mt & 1) ? 4194304.f : 16777216.f;   // 2^24 / 4^(mt&1)
      const float za = zz0[mt >> 1], zb = zz1[mt >> 1];
      v0 = fmaf(v0, sc, za); v1 = fmaf(v1, sc, zb);
      v2 = fmaf(v2, sc, za); v3 = fmaf(v3, sc, zb);
    }
    wo[(2 * tig) * D + c0] = v0;
    wo[(2 * tig + 1) * D + c0] = v1;
    wo[(2 * tig) * D + c1] = v2;
    wo[(2 * tig + 1) * D + c1] = v3;
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kDThreads) {
    const int g = idx / D, ch = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDWarps; ++w) M = fmaxf(M, scr[w * (16 + 8 * D) + g]);
    float Ls = 0.f, Os = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDWarps; ++w) {
        const float* base = scr + w * (16 + 8 * D);
        const float mw = base[g];
        if (mw != -INFINITY) {
          const float e = exp2f(mw - M);
          Ls = fmaf(e, base[8 + g], Ls);
          Os = fmaf(e, base[16 + g * D + ch], Os);
        }
      }
    }
    float* dst = p.part +
                 ((static_cast<size_t>(b) * p.hq + h * G + g) * p.n_splits + split) * (D + 2);
    if (ch == 0) { dst[0] = M; dst[1] = Ls; }
    dst[2 + ch] = Os;
  }
}

// ---------------------------------------------------------------- combine

constexpr int kMaxSplits = 2048;

// One CTA per (query head, KV head, sequence).  Warp 0 finds the global max
// and the split weights w_s = 2^(m_s - M); all threads then sum the weighted
// split outputs channel by channel (coalesced, many loads in flight), and the
// INT2 part is rotated back once: out = (o_raw + o_rot R_V^T) / l.
template <int D, bool kBf16Only>
__global__ void __launch_bounds__(256) combine_kernel(const DecodeParams p) {
  constexpr int RPW = D / 8;              // output rows per warp
  constexpr int VPL = D / 32;             // R_V entries per lane per row
  constexpr int SG = 256 / D;             // split groups summed in parallel
  __shared__ float wsplit[kMaxSplits];
  __shared__ float acc_rot[SG][D];
  __shared__ float acc_raw[SG][D];
  __shared__ float orot[D];
  __shared__ float lsum;
  const int g = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
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
  const int ns = p.n_splits;
  const float* base = p.part + (static_cast<size_t>(b) * p.hq + h * p.G + g) * ns * (D + 2);
  if (warp == 0) {
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, base[s * (D + 2)]);
    M = warp_max(M);
    float Ls = 0.f;
    for (int s = lane; s < ns; s += 32) {
      const float ms = base[s * (D + 2)];
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      wsplit[s] = w;
      Ls = fmaf(w, base[s * (D + 2) + 1], Ls);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane == 0) lsum = Ls;
  }
  __syncthreads();
  {
    const int ch = tid % D, sg = tid / D;
    float ar = 0.f, aw = 0.f;
    const int n_rot = kBf16Only ? 0 : p.n_main;
#pragma unroll 8
    for (int s = sg; s < ns; s += SG) {
      const float v = wsplit[s] * base[s * (D + 2) + 2 + ch];
      if (s < n_rot) ar += v; else aw += v;
    }
    acc_rot[sg][ch] = ar;
    acc_raw[sg][ch] = aw;
  }
  __syncthreads();
  if (tid < D) {
    float ar = 0.f, aw = 0.f;
#pragma unroll
    for (int k = 0; k < SG; ++k) { ar += acc_rot[k][tid]; aw += acc_raw[k][tid]; }
    orot[tid] = ar;
    acc_raw[0][tid] = aw;
  }
  __syncthreads();
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  uint16_t* dst = p.out + (static_cast<size_t>(b) * p.hq + h * p.G + g) * D;
  if (kBf16Only) {
    if (tid < D) dst[tid] = __bfloat16_as_ushort(__float2bfloat16_rn(acc_raw[0][tid] * inv));
  } else {
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const int i = warp * RPW + k;
      float a = 0.f;
#pragma unroll
      for (int u = 0; u < VPL; ++u) a = fmaf(orot[lane * VPL + u], rv[k][u], a);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
      if (lane == 0) dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn((acc_raw[0][i] + a) * inv));
    }
  }
}

// ------------------------------------------------------------------- host

struct Plan {
  int n_main, pps, n_splits;
  size_t qrot_bytes, part_off, part_bytes, total;
};

Plan make_plan(const oscar_cache_desc* c, int batch, int max_len, bool bf16_only) {
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
  const int64_t units = static_cast<int64_t>(batch) * c->num_kv_heads;
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
  pl.total = pl.part_off + pl.part_bytes;
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

template <int D, bool kBf16Only>
oscar_status run_decode(const DecodeParams& p, const Plan& pl, cudaStream_t st) {
  using C = SplitCfg<D, kBf16Only>;
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(split_kernel<D, kBf16Only>), C::kBytes))
    return OSCAR_ERR_CUDA;
  const dim3 sgrid(pl.n_splits, p.hkv, p.batch);
  cudaError_t e;
  if (!kBf16Only) {
    qrot_kernel<D><<<dim3(p.hkv, p.batch), 1024, 0, st>>>(p);
    if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_CUDA;
    e = launch_pdl(split_kernel<D, kBf16Only>, sgrid, dim3(kDThreads), C::kBytes, st, p);
  } else {
    split_kernel<D, kBf16Only><<<sgrid, kDThreads, C::kBytes, st>>>(p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return OSCAR_ERR_CUDA;
  e = launch_pdl(combine_kernel<D, kBf16Only>, dim3(p.G, p.hkv, p.batch), dim3(256), 0, st, p);
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

oscar_status decode_entry(const oscar_cache_desc* c, const void* q, const int32_t* seq_lens,
                          int batch, int max_len, void* out, void* ws, size_t ws_bytes,
                          void* stream, bool bf16_only) {
  oscar_status s = oscar_host::check_desc(c, !bf16_only, true);
  if (s != OSCAR_OK) return s;
  if (batch < 0 || max_len < 1) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  if (!q || !seq_lens || !out || !ws) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & 15) return OSCAR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 3)
    return OSCAR_ERR_INVALID_ARG;
  if (max_len > static_cast<int64_t>(c->max_pages_per_seq) * kPage) return OSCAR_ERR_INVALID_ARG;
  if (!bf16_only &&
      (c->sink + kPage - 1) / kPage + (c->window + kPage - 1) / kPage + 1 > kMaxCtaPages)
    return OSCAR_ERR_UNSUPPORTED;
  const Plan pl = make_plan(c, batch, max_len, bf16_only);
  if (pl.n_splits > kMaxSplits) return OSCAR_ERR_UNSUPPORTED;
  if (ws_bytes < pl.total) return OSCAR_ERR_WORKSPACE;
  DecodeParams p{};
  p.hkv = c->num_kv_heads;
  p.hq = c->num_q_heads;
  p.G = c->num_q_heads / c->num_kv_heads;
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
  p.status = c->status;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.max_len = max_len;
  p.n_main = pl.n_main;
  p.pps = pl.pps;
  p.n_splits = pl.n_splits;
  p.qrot = reinterpret_cast<float*>(ws);
  p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + pl.part_off);
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c->head_dim)));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->head_dim == 128)
    return bf16_only ? run_decode<128, true>(p, pl, st) : run_decode<128, false>(p, pl, st);
  return bf16_only ? run_decode<64, true>(p, pl, st) : run_decode<64, false>(p, pl, st);
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

}  // extern "C"
