// Rotate + clip + INT2-quantise + pack: moves tokens into the mixed cache.
//
// "Technical Summary: OSCAR ...", section 2.2B: the middle history is stored
// in INT2 after the fixed rotation and clipping; sink and recent tokens stay
// BF16.  One kernel serves both entry points:
//   prefill: a list of (sequence, position) tokens with their bf16 K/V; each is
//            copied to its BF16 slot or quantised into its INT2 slot;
//   append:  per sequence, the new token goes to its BF16 slot and the token
//            that just left the recent window is read back from its BF16 slot
//            and quantised into its INT2 slot.
// A CTA owns one (KV head, K-or-V) pair, keeps that head's d x d rotation in
// shared memory and walks tiles of 32 tokens: y = x R with fp32 FMAs in index
// order, then per group of 32 channels (one warp, one lane per channel) clip,
// min/max, s16 = fp16((max-min)/3), z16 = fp16(min), code =
// rint((y_c - z16)/s16) clamped to [0,3], each step rounded in fp32 exactly as
// written, then the codes are packed byte by byte into the page format of
// layout.cuh (every byte holds codes of one token, so slots never collide).
// Bulk prefill takes the tensor-core kernel of rotate_tc.cuh instead whenever
// its inputs suit TMA, and the per-step append has append_kernel (below); this
// kernel keeps the prefill inputs that do not suit TMA.
#include <algorithm>

#include "common.cuh"
#include "layout.cuh"

namespace oscar {

constexpr int kQTile = 32;
constexpr int kQThreads = 256;

struct QuantParams {
  int hkv, sink, window, max_pages;
  int64_t n_int2_pages, n_bf16_pages;
  uint8_t* int2_pool;
  uint16_t* bf16_pool;
  const int32_t* int2_pt;
  const int32_t* bf16_pt;
  const float* r_k;
  const float* r_v;
  const float* clip_k;
  const float* clip_v;
  int32_t* status;
  int append;
  int64_t n_items;
  int num_seqs;
  const uint16_t* k_src;
  const uint16_t* v_src;
  const int32_t* seq_ids;
  const int32_t* positions;
  const int32_t* seq_lens;
  // append only, optional: the step's rotated query q' = q R_K, written by the
  // K-side CTAs (each its 32 output channels) for the decode that follows
  const uint16_t* q;     // [B][Hq][D] bf16
  float* qrot;           // [B][Hq][D] fp32, or null
  int hq, G;
  int planes;            // 2-bit code planes: 1 (INT2) or 2 (the INT4 variant)
  // append only, optional: rotary position embedding of the new key and the
  // query at the new token's position (length - 1), log2 of its base (0: none);
  // the rotated query is also written, rounded to bf16, to qrope [B][Hq][D]
  double rope_log2_base;
  uint16_t* qrope;
  // optional diagnostic output: the fp32 rotated values y = x R each INT2
  // placement computed (before clipping), [item][Hkv][2 (K, V)][D]; entries of
  // items without an INT2 placement are not written
  float* y_out;
};

template <int D>
struct QuantSmem {
  static constexpr int kR = 0;                                    // float [D][D]
  static constexpr int kX = kR + D * D * 4;                       // float [T][D]
  static constexpr int kY = kX + kQTile * D * 4;                  // float [T][D]
  static constexpr int kCodes = kY + kQTile * D * 4;              // u8 [T][D]
  static constexpr int kSz = kCodes + kQTile * D;                 // u32 [T][ng]
  static constexpr int kMeta = kSz + kQTile * (D / 32) * 4;       // int [6][T]
  static constexpr int kBar = kMeta + 6 * kQTile * 4;             // u64 mbarrier
  static constexpr int kBytes = kBar + 16;
};

__device__ __forceinline__ void flag(int32_t* status, int bit) {
  if (status) atomicOr(status, bit);
}

}  // namespace oscar

#include "rotate_tc.cuh"
#include "append_group.cuh"

namespace oscar {

template <int D, int P>
__global__ void __launch_bounds__(kQThreads) quantize_kernel(const QuantParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  using S = QuantSmem<D>;
  using F = Fmt<D, P>;
  constexpr float kLevels = P == 2 ? 15.f : 3.f;   // largest code: INT4 variant / INT2
  constexpr int kMaxCode = P == 2 ? 15 : 3;
  constexpr int NG = D / 32;
  constexpr int NW = D / 32;    // code words per lane
  float* rs = reinterpret_cast<float*>(smem + S::kR);
  float* xs = reinterpret_cast<float*>(smem + S::kX);
  float* ys = reinterpret_cast<float*>(smem + S::kY);
  uint8_t* codes = smem + S::kCodes;
  uint32_t* szs = reinterpret_cast<uint32_t*>(smem + S::kSz);
  int* m_i2page = reinterpret_cast<int*>(smem + S::kMeta);   // INT2 destination page (-1: none)
  int* m_i2slot = m_i2page + kQTile;
  int* m_bfpage = m_i2slot + kQTile;                           // BF16 destination page (-1: none)
  int* m_bfslot = m_bfpage + kQTile;
  int* m_srcpage = m_bfslot + kQTile;                          // append: BF16 source page
  int* m_srcslot = m_srcpage + kQTile;

  const int h = blockIdx.y;
  const int kv = blockIdx.z;      // 0 keys, 1 values
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* rot = (kv ? p.r_v : p.r_k) + static_cast<size_t>(h) * D * D;
  const uint16_t* src = kv ? p.v_src : p.k_src;

  // the head's rotation arrives in shared memory by one bulk copy
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kBar);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  // launched with programmatic stream serialisation: inputs are read only after
  // the predecessor grid has completed (the clip too: a calibration kernel just
  // before this one may have written it); then the next kernel may launch
  pdl_wait();
  pdl_trigger();
  const float clip = (kv ? p.clip_v : p.clip_k)[h];
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, D * D * 4);
    bulk_g2s(rs, rot, D * D * 4, bar);
  }
  bool r_ready = false;

  const int64_t n_tiles = (p.n_items + kQTile - 1) / kQTile;
  for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    __syncthreads();   // previous tile's smem reads done (and R visible on the first pass)
    int need_rot = 0;
    if (tid < kQTile) {
      const int64_t item = tile * kQTile + tid;
      int i2page = -1, i2slot = 0, bfpage = -1, bfslot = 0, srcpage = -1, srcslot = 0;
      if (item < p.n_items) {
        if (!p.append) {
          const int seq = p.seq_ids[item];
          const int pos = p.positions[item];
          const int L = (seq >= 0 && seq < p.num_seqs) ? p.seq_lens[seq] : -1;
          if (seq < 0 || seq >= p.num_seqs || pos < 0 || pos >= L ||
              pos / kPage >= p.max_pages) {
            flag(p.status, OSCAR_DEVERR_SEQ_LEN);
          } else {
            const int64_t row = static_cast<int64_t>(seq) * p.max_pages + pos / kPage;
            if (pos >= p.sink && pos < L - p.window) {
              const int pg = p.int2_pt[row];
              if (pg < 0 || pg >= p.n_int2_pages) flag(p.status, OSCAR_DEVERR_PAGE_ID);
              else { i2page = pg; i2slot = pos % kPage; }
            } else {
              const int pg = p.bf16_pt[row];
              if (pg < 0 || pg >= p.n_bf16_pages) flag(p.status, OSCAR_DEVERR_PAGE_ID);
              else { bfpage = pg; bfslot = pos % kPage; }
            }
          }
        } else {
          const int b = static_cast<int>(item);
          const int L = p.seq_lens[b];
          if (L < 1 || (L - 1) / kPage >= p.max_pages) {
            flag(p.status, OSCAR_DEVERR_SEQ_LEN);
          } else {
            const int64_t base = static_cast<int64_t>(b) * p.max_pages;
            const int pn = L - 1;                      // new token -> BF16
            const int pg = p.bf16_pt[base + pn / kPage];
            if (pg < 0 || pg >= p.n_bf16_pages) flag(p.status, OSCAR_DEVERR_PAGE_ID);
            else { bfpage = pg; bfslot = pn % kPage; }
            const int po = L - 1 - p.window;           // token leaving the window
            if (po >= p.sink) {
              const int sp = p.bf16_pt[base + po / kPage];
              const int dp = p.int2_pt[base + po / kPage];
              if (sp < 0 || sp >= p.n_bf16_pages || dp < 0 || dp >= p.n_int2_pages) {
                flag(p.status, OSCAR_DEVERR_PAGE_ID);
              } else {
                srcpage = sp; srcslot = po % kPage;
                i2page = dp; i2slot = po % kPage;
              }
            }
          }
        }
      }
      m_i2page[tid] = i2page; m_i2slot[tid] = i2slot;
      m_bfpage[tid] = bfpage; m_bfslot[tid] = bfslot;
      m_srcpage[tid] = srcpage; m_srcslot[tid] = srcslot;
      need_rot = i2page >= 0;
    }
    need_rot = __syncthreads_or(need_rot);

    // --- load x rows (fp32) and perform the BF16 writes
    for (int idx = tid; idx < kQTile * D; idx += kQThreads) {
      const int t = idx / D, j = idx % D;
      const int64_t item = tile * kQTile + t;
      float x = 0.f;
      if (!p.append) {
        if (item < p.n_items) {
          const uint16_t v = src[(item * p.hkv + h) * D + j];
          x = bf16_to_float(v);
          const int bp = m_bfpage[t];
          if (bp >= 0) {
            const int e = kv ? 16 * D + bf16_value_elem(m_bfslot[t], j) : bf16_key_elem(m_bfslot[t], j);
            p.bf16_pool[(static_cast<int64_t>(bp) * p.hkv + h) * (32 * D) + e] = v;
          }
        }
      } else if (item < p.n_items) {
        // distinct slots: the leaving token's read and the new token's write
        // never touch the same element
        const int sp = m_srcpage[t];
        if (sp >= 0) {
          const int e = kv ? 16 * D + bf16_value_elem(m_srcslot[t], j) : bf16_key_elem(m_srcslot[t], j);
          x = bf16_to_float(p.bf16_pool[(static_cast<int64_t>(sp) * p.hkv + h) * (32 * D) + e]);
        }
        const int bp = m_bfpage[t];
        if (bp >= 0) {
          const uint16_t v = src[(item * p.hkv + h) * D + j];
          const int e = kv ? 16 * D + bf16_value_elem(m_bfslot[t], j) : bf16_key_elem(m_bfslot[t], j);
          p.bf16_pool[(static_cast<int64_t>(bp) * p.hkv + h) * (32 * D) + e] = v;
        }
      }
      xs[idx] = x;
    }
    if (!need_rot) continue;
    if (!r_ready) {
      r_ready = __syncthreads_and(mbar_wait(bar, 0, p.status));
      // recorded as a timeout; nothing usable to rotate with.  The copy may
      // still be in flight, so the CTA leaves through the bounded wait below.
      if (!r_ready) break;
    }
    __syncthreads();

    // --- rotation y = x R (fp32 FMA, i ascending); warps without an INT2 token idle
    const bool busy = m_i2page[4 * warp] >= 0 || m_i2page[4 * warp + 1] >= 0 ||
                      m_i2page[4 * warp + 2] >= 0 || m_i2page[4 * warp + 3] >= 0;
    if (busy) {
      constexpr int JPT = D / 32;
      const int jl = lane, tg = warp;
      float acc[4][JPT];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < JPT; ++c) acc[u][c] = 0.f;
      const float* x0 = xs + (4 * tg) * D;
#pragma unroll 4
      for (int i = 0; i < D; ++i) {
        float r[JPT];
        if constexpr (JPT == 4) {
          const float4 v = reinterpret_cast<const float4*>(rs + i * D)[jl];
          r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
        } else {
          const float2 v = reinterpret_cast<const float2*>(rs + i * D)[jl];
          r[0] = v.x; r[1] = v.y;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float xv = x0[u * D + i];
#pragma unroll
          for (int c = 0; c < JPT; ++c) acc[u][c] = fmaf(xv, r[c], acc[u][c]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < JPT; ++c) ys[(4 * tg + u) * D + JPT * jl + c] = acc[u][c];
    }
    __syncthreads();

    // --- clip + group quantisation: one warp per (token, group)
    for (int task = warp; task < kQTile * NG; task += kQThreads / 32) {
      const int t = task / NG, grp = task % NG;
      if (m_i2page[t] < 0) continue;
      float y = ys[t * D + 32 * grp + lane];
      if (p.y_out)
        p.y_out[((tile * kQTile + t) * p.hkv + h) * (2 * D) + kv * D + 32 * grp + lane] = y;
      if (__any_sync(0xffffffffu, !isfinite(y))) {   // stored as a zero group
        if (lane == 0) flag(p.status, OSCAR_DEVERR_NONFINITE);
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
      if (sf != 0.f) {
        code = __float2int_rn(__fdiv_rn(__fsub_rn(yc, zf), sf));
        code = min(max(code, 0), kMaxCode);
      }
      codes[t * D + 32 * grp + lane] = static_cast<uint8_t>(code);
      if (lane == 0)
        szs[t * NG + grp] = static_cast<uint32_t>(__half_as_ushort(s16)) |
                            (static_cast<uint32_t>(__half_as_ushort(z16)) << 16);
    }
    __syncthreads();

    // --- pack: one thread per (token, code plane, code byte); plane 0 holds the
    // highest two bits of each code
    for (int idx = tid; idx < kQTile * P * (D / 4); idx += kQThreads) {
      const int t = idx / (P * (D / 4)), rem = idx % (P * (D / 4));
      const int pl = rem / (D / 4), q = rem % (D / 4);
      const int shift = 2 * (P - 1 - pl);
      const int pg = m_i2page[t];
      if (pg < 0) continue;
      const int slot = m_i2slot[t];
      uint8_t* blk = p.int2_pool + (static_cast<int64_t>(pg) * p.hkv + h) * F::kInt2Block;
      const uint8_t* ct = codes + t * D;
      uint32_t byte = 0;
      if (kv == 0) {
        const int tig = q / (2 * NW), m = (q >> 1) % NW, e = q & 1;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int i = 0; i < 2; ++i)
            byte |= ((static_cast<uint32_t>(ct[16 * (2 * m + i) + 8 * hh + 2 * tig + e]) >> shift) & 3u)
                    << (4 * hh + 2 * i);
        blk[F::kKc + pl * F::kPlane + key_byte<D>(slot, tig, m, e)] = static_cast<uint8_t>(byte);
      } else {
        const int gid = q / NW, m = q % NW;
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int i = 0; i < 2; ++i)
            byte |= ((static_cast<uint32_t>(ct[16 * (2 * m + i) + 8 * ch + gid]) >> shift) & 3u)
                    << (4 * ch + 2 * i);
        blk[F::kVc + pl * F::kPlane + value_byte<D>(slot, gid, m)] = static_cast<uint8_t>(byte);
      }
    }
    for (int idx = tid; idx < kQTile * NG; idx += kQThreads) {
      const int t = idx / NG, grp = idx % NG;
      const int pg = m_i2page[t];
      if (pg < 0) continue;
      const int slot = m_i2slot[t];
      uint8_t* blk = p.int2_pool + (static_cast<int64_t>(pg) * p.hkv + h) * F::kInt2Block;
      const uint32_t sz = szs[t * NG + grp];
      if (kv == 0) {
        reinterpret_cast<uint32_t*>(blk + F::kKsz)[slot * NG + grp] = sz;
      } else {
        const int e = vsz_index<D>(slot, grp);
        reinterpret_cast<uint16_t*>(blk + F::kVs)[e] = static_cast<uint16_t>(sz & 0xffffu);
        reinterpret_cast<uint16_t*>(blk + F::kVz)[e] = static_cast<uint16_t>(sz >> 16);
      }
    }
  }
  if (!r_ready) mbar_wait(bar, 0, p.status);   // never leave with the copy in flight
}

template <int D, int P>
oscar_status launch_quantize_p(const QuantParams& p, cudaStream_t st) {
  const int smem = QuantSmem<D>::kBytes;
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(quantize_kernel<D, P>), smem))
    return OSCAR_ERR_CUDA;
  const int64_t tiles = (p.n_items + kQTile - 1) / kQTile;
  if (tiles == 0) return OSCAR_OK;
  const int sms = oscar_host::sm_count();
  const int64_t per_pair = std::max<int64_t>(1, (2LL * sms + 2 * p.hkv - 1) / (2 * p.hkv));
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>(tiles, per_pair)), p.hkv, 2);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_kernel<D, P>, p) == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

template <int D>
oscar_status launch_quantize(const QuantParams& p, cudaStream_t st) {
  return p.planes == 2 ? launch_quantize_p<D, 2>(p, st) : launch_quantize_p<D, 1>(p, st);
}

// ------------------------------------------------------------------ append

//
// One decode step's append: per sequence b, the new token goes to its BF16 slot
// (position L-1) and, once L-1-W >= S, the token at L-1-W leaves the window: it
// is read back from its BF16 slot, rotated, clipped, quantised and packed into
// its INT2 slot.  A batch has few tokens, so the work is spread over the
// channel groups: a CTA owns one group of 32 output channels of one (KV head,
// K/V) pair and up to 8 sequences, keeps the 16 KB column slice of R it needs,
// and a warp handles one sequence (lane j = output channel 32*grp + j).
constexpr int kAppendSeqs = 8;      // sequences per CTA: one per warp

// kGroup4 (batches of eight or more sequences): a warp rotates four queries
// per pass over the R slice.
template <int D, int P, bool kGroup4>
__global__ void __launch_bounds__(kQThreads) append_kernel(const QuantParams p) {
  constexpr int NG = D / 32;
  using F = Fmt<D, P>;
  __shared__ __align__(16) float rs[D][32];          // R[:, 32*grp .. 32*grp + 31]
  __shared__ __align__(16) float xs[kQThreads / 32][kGroup4 ? 4 : 1][D];   // per warp
  __shared__ uint8_t cs[kQThreads / 32][32];
  __shared__ double inv_freq[D / 2];                 // rotary base^(-2i/D)
  const int grp = blockIdx.x % NG, chunk = blockIdx.x / NG;
  const int h = blockIdx.y, kv = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool rope = p.rope_log2_base > 0.0;
  if (rope)
    for (int i = tid; i < D / 2; i += kQThreads) inv_freq[i] = exp2(-2.0 * i / D * p.rope_log2_base);
  // The layer's rotation is a constant of the cache and is read while the
  // predecessor grid may still run; every other input only after it has
  // completed (programmatic stream serialisation).
  const float* rot = (kv ? p.r_v : p.r_k) + static_cast<size_t>(h) * D * D + 32 * grp;
  for (int e = tid; e < D * 8; e += kQThreads) {       // float4 e%8 of row e/8
    const int i = e >> 3, c4 = e & 7;
    reinterpret_cast<float4*>(&rs[i][0])[c4] = reinterpret_cast<const float4*>(rot + i * D)[c4];
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const float clip = (kv ? p.clip_v : p.clip_k)[h];
  const uint16_t* src = kv ? p.v_src : p.k_src;
  const int j = 32 * grp + lane;                       // this lane's channel
  if (kv == 0 && p.qrot) {
    // the step's rotated query, (sequence, query head) tasks, lane j computing
    // channel 32*grp + j
    const int64_t left = p.n_items - static_cast<int64_t>(chunk) * kAppendSeqs;
    const int n_seq = static_cast<int>(left < kAppendSeqs ? left : kAppendSeqs);
    const int n_tasks = n_seq * p.G;
    constexpr int kWarps = kQThreads / 32;
    // the task's query (rotated to the new token's position with rotary
    // embedding, rounded to bf16) into row
    auto stage = [&](int task, float* row) {
      const int b = chunk * kAppendSeqs + task / p.G, g = task % p.G;
      const uint16_t* qg = p.q + (static_cast<int64_t>(b) * p.hq + h * p.G + g) * D;
      const int m = rope ? p.seq_lens[b] - 1 : 0;   // issued with the query loads, not after them
#pragma unroll
      for (int c = 0; c < NG; ++c) row[32 * c + lane] = bf16_to_float(qg[32 * c + lane]);
      __syncwarp();
      if (rope) {
        float v[NG];
#pragma unroll
        for (int c = 0; c < NG; ++c) {
          const int jj = 32 * c + lane;
          v[c] = rope_bf16<D>(row[jj], row[jj < D / 2 ? jj + D / 2 : jj - D / 2], jj, m, inv_freq);
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < NG; ++c) row[32 * c + lane] = v[c];
        __syncwarp();
        if (p.qrope)   // this CTA's 32 channels of the rotated query, for the BF16 split
          p.qrope[(static_cast<int64_t>(b) * p.hq + h * p.G + g) * D + j] =
              __bfloat16_as_ushort(__float2bfloat16_rn(row[j]));
      }
    };
    auto store = [&](int task, float v) {
      const int b = chunk * kAppendSeqs + task / p.G, g = task % p.G;
      p.qrot[(static_cast<int64_t>(b) * p.hq + h * p.G + g) * D + j] = v;
    };
    if (kGroup4 && n_tasks >= 4 * kWarps) {
      // many tasks: four per pass over the R slice, so each shared-memory read
      // of R serves four dot products (each task's sum in the same order as below)
      for (int t4 = 4 * warp; t4 < n_tasks; t4 += 4 * kWarps) {
        const int nt = min(4, n_tasks - t4);
        for (int t = 0; t < nt; ++t) stage(t4 + t, xs[warp][kGroup4 ? t : 0]);
        float acc[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll 4
        for (int i = 0; i < D; i += 4) {
          const float r0 = rs[i][lane], r1 = rs[i + 1][lane], r2 = rs[i + 2][lane],
                      r3 = rs[i + 3][lane];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float4 xv = *reinterpret_cast<const float4*>(&xs[warp][kGroup4 ? t : 0][i]);
            acc[t][0] = fmaf(xv.x, r0, acc[t][0]);
            acc[t][1] = fmaf(xv.y, r1, acc[t][1]);
            acc[t][2] = fmaf(xv.z, r2, acc[t][2]);
            acc[t][3] = fmaf(xv.w, r3, acc[t][3]);
          }
        }
        for (int t = 0; t < nt; ++t) store(t4 + t, (acc[t][0] + acc[t][1]) + (acc[t][2] + acc[t][3]));
        __syncwarp();
      }
    } else {
      // few tasks: one per warp, task t on warp (t + n_seq) mod 8: warps
      // 0 .. n_seq-1 also place a token each below, so with few sequences the
      // two chains run side by side
      const int t0 = ((warp - n_seq) % kWarps + kWarps) % kWarps;
      for (int task = t0; task < n_tasks; task += kWarps) {
        stage(task, xs[warp][0]);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int i = 0; i < D; i += 4) {
          const float4 xv = *reinterpret_cast<const float4*>(&xs[warp][0][i]);
          acc[0] = fmaf(xv.x, rs[i][lane], acc[0]);
          acc[1] = fmaf(xv.y, rs[i + 1][lane], acc[1]);
          acc[2] = fmaf(xv.z, rs[i + 2][lane], acc[2]);
          acc[3] = fmaf(xv.w, rs[i + 3][lane], acc[3]);
        }
        store(task, (acc[0] + acc[1]) + (acc[2] + acc[3]));
        __syncwarp();
      }
    }
  }
  for (int u = warp; u < kAppendSeqs; u += kQThreads / 32) {
    const int b = chunk * kAppendSeqs + u;
    if (b >= p.n_items) break;
    // loads are issued level by level: the length with the new token's values,
    // then every page-table entry the length selects, then the pages
    const int L = p.seq_lens[b];
    const uint16_t* xn = src + (static_cast<int64_t>(b) * p.hkv + h) * D;
    const uint16_t xv = xn[j];
    const uint16_t xr = (rope && kv == 0) ? xn[j < D / 2 ? j + D / 2 : j - D / 2] : 0;
    if (L < 1 || (L - 1) / kPage >= p.max_pages) {
      if (lane == 0 && grp == 0) flag(p.status, OSCAR_DEVERR_SEQ_LEN);
      continue;
    }
    const int64_t base = static_cast<int64_t>(b) * p.max_pages;
    const int pn = L - 1;                 // the new token -> its BF16 slot
    const int po = L - 1 - p.window;      // the token leaving the window
    const bool leaves = po >= p.sink;
    const int pg = p.bf16_pt[base + pn / kPage];
    const int sp = leaves ? p.bf16_pt[base + po / kPage] : -1;
    const int dp = leaves ? p.int2_pt[base + po / kPage] : -1;
    if (pg < 0 || pg >= p.n_bf16_pages) {
      if (lane == 0 && grp == 0) flag(p.status, OSCAR_DEVERR_PAGE_ID);
    } else {
      const int e = kv ? 16 * D + bf16_value_elem(pn % kPage, j) : bf16_key_elem(pn % kPage, j);
      uint16_t val = xv;
      if (rope && kv == 0)   // the new key at its position, rounded to bf16
        val = __bfloat16_as_ushort(__float2bfloat16_rn(rope_bf16<D>(
            bf16_to_float(xv), bf16_to_float(xr), j, pn, inv_freq)));
      p.bf16_pool[(static_cast<int64_t>(pg) * p.hkv + h) * (32 * D) + e] = val;
    }
    if (!leaves) continue;
    if (sp < 0 || sp >= p.n_bf16_pages || dp < 0 || dp >= p.n_int2_pages) {
      if (lane == 0 && grp == 0) flag(p.status, OSCAR_DEVERR_PAGE_ID);
      continue;
    }
    const int slot = po % kPage;
    const uint16_t* sblk = p.bf16_pool + (static_cast<int64_t>(sp) * p.hkv + h) * (32 * D);
#pragma unroll
    for (int c = 0; c < NG; ++c) {
      const int jj = 32 * c + lane;
      const int e = kv ? 16 * D + bf16_value_elem(slot, jj) : bf16_key_elem(slot, jj);
      xs[warp][0][jj] = bf16_to_float(sblk[e]);
    }
    __syncwarp();
    // y_j = sum_i x_i R[i][j], fp32, four partial chains over i
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int i = 0; i < D; i += 4) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[warp][0][i]);
      acc[0] = fmaf(xv.x, rs[i][lane], acc[0]);
      acc[1] = fmaf(xv.y, rs[i + 1][lane], acc[1]);
      acc[2] = fmaf(xv.z, rs[i + 2][lane], acc[2]);
      acc[3] = fmaf(xv.w, rs[i + 3][lane], acc[3]);
    }
    const float y = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    if (p.y_out) p.y_out[(static_cast<int64_t>(b) * p.hkv + h) * (2 * D) + kv * D + j] = y;
    uint8_t* blk = p.int2_pool + (static_cast<int64_t>(dp) * p.hkv + h) * F::kInt2Block;
    append_group<D, P>(y, clip, lane, grp, kv, slot, blk, cs[warp], p.status);
  }
}

template <int D, int P>
oscar_status launch_append_p(const QuantParams& p, cudaStream_t st) {
  const int64_t chunks = (p.n_items + kAppendSeqs - 1) / kAppendSeqs;
  if (chunks == 0) return OSCAR_OK;
  const dim3 grid(static_cast<unsigned>(chunks * (D / 32)), p.hkv, 2);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the grouped form only where a CTA has many query rotations to share R with
  const bool group4 = p.qrot && p.n_items >= kAppendSeqs;
  const cudaError_t e = group4 ? cudaLaunchKernelEx(&cfg, append_kernel<D, P, true>, p)
                               : cudaLaunchKernelEx(&cfg, append_kernel<D, P, false>, p);
  return e == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

template <int D>
oscar_status launch_append(const QuantParams& p, cudaStream_t st) {
  return p.planes == 2 ? launch_append_p<D, 2>(p, st) : launch_append_p<D, 1>(p, st);
}

QuantParams base_params(const oscar_cache_desc* c) {
  QuantParams p{};
  p.hkv = c->num_kv_heads;
  p.sink = c->sink;
  p.window = c->window;
  p.max_pages = c->max_pages_per_seq;
  p.n_int2_pages = c->num_int2_pages;
  p.n_bf16_pages = c->num_bf16_pages;
  p.int2_pool = static_cast<uint8_t*>(c->int2_pool);
  p.bf16_pool = static_cast<uint16_t*>(c->bf16_pool);
  p.int2_pt = c->int2_page_table;
  p.bf16_pt = c->bf16_page_table;
  p.r_k = c->r_k;
  p.r_v = c->r_v;
  p.clip_k = c->clip_k;
  p.clip_v = c->clip_v;
  p.status = c->status;
  p.planes = oscar_host::code_planes(c);
  return p;
}

oscar_status dispatch(const QuantParams& p, int d, cudaStream_t st) {
  return d == 128 ? launch_quantize<128>(p, st) : launch_quantize<64>(p, st);
}

// The append of a fused decode step: as oscar_quantize_append, and the K-side
// CTAs also write q' = q R_K for the decode that follows.
oscar_status append_with_query(const oscar_cache_desc* desc, const void* q, const void* k_new,
                               const void* v_new, const int32_t* seq_lens_after, int32_t batch,
                               float* qrot, double rope_log2_base, uint16_t* qrope,
                               cudaStream_t st) {
  QuantParams p = base_params(desc);
  p.append = 1;
  p.n_items = batch;
  p.num_seqs = batch;
  p.k_src = static_cast<const uint16_t*>(k_new);
  p.v_src = static_cast<const uint16_t*>(v_new);
  p.seq_lens = seq_lens_after;
  p.q = static_cast<const uint16_t*>(q);
  p.qrot = qrot;
  p.rope_log2_base = rope_log2_base;
  p.qrope = qrope;
  p.hq = desc->num_q_heads;
  p.G = desc->num_q_heads / desc->num_kv_heads;
  return desc->head_dim == 128 ? launch_append<128>(p, st) : launch_append<64>(p, st);
}

}  // namespace oscar

extern "C" {

oscar_status oscar_prefill_quantize_trace(const oscar_cache_desc* desc, const void* k,
                                          const void* v, const int32_t* seq_ids,
                                          const int32_t* positions, const int32_t* seq_lens_final,
                                          int32_t num_seqs, int64_t total_tokens, float* y_out,
                                          void* stream) {
  oscar_status s = oscar_host::check_desc(desc, true, true);
  if (s != OSCAR_OK) return s;
  if (total_tokens < 0 || num_seqs < 1) return OSCAR_ERR_INVALID_ARG;
  if (total_tokens == 0) return OSCAR_OK;
  if (!k || !v || !seq_ids || !positions || !seq_lens_final) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(y_out) & 15) return OSCAR_ERR_INVALID_ARG;
  oscar::QuantParams p = oscar::base_params(desc);
  p.append = 0;
  p.n_items = total_tokens;
  p.num_seqs = num_seqs;
  p.k_src = static_cast<const uint16_t*>(k);
  p.v_src = static_cast<const uint16_t*>(v);
  p.seq_ids = seq_ids;
  p.positions = positions;
  p.seq_lens = seq_lens_final;
  p.y_out = y_out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the rotation on the tensor cores whenever the inputs suit TMA; the
  // CUDA-core kernel otherwise (same bytes either way)
  oscar_status r = OSCAR_OK;
  const bool done = desc->head_dim == 128 ? oscar::launch_rotate_tc<128>(p, st, &r)
                                          : oscar::launch_rotate_tc<64>(p, st, &r);
  if (done) return r;
  return oscar::dispatch(p, desc->head_dim, st);
}

oscar_status oscar_prefill_quantize(const oscar_cache_desc* desc, const void* k, const void* v,
                                    const int32_t* seq_ids, const int32_t* positions,
                                    const int32_t* seq_lens_final, int32_t num_seqs,
                                    int64_t total_tokens, void* stream) {
  return oscar_prefill_quantize_trace(desc, k, v, seq_ids, positions, seq_lens_final, num_seqs,
                                      total_tokens, nullptr, stream);
}

oscar_status oscar_quantize_append_trace(const oscar_cache_desc* desc, const void* k_new,
                                         const void* v_new, const int32_t* seq_lens_after,
                                         int32_t batch, float* y_out, void* stream) {
  oscar_status s = oscar_host::check_desc(desc, true, true);
  if (s != OSCAR_OK) return s;
  if (batch < 0) return OSCAR_ERR_INVALID_ARG;
  if (batch == 0) return OSCAR_OK;
  if (!k_new || !v_new || !seq_lens_after) return OSCAR_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(y_out) & 15) return OSCAR_ERR_INVALID_ARG;
  oscar::QuantParams p = oscar::base_params(desc);
  p.append = 1;
  p.n_items = batch;
  p.num_seqs = batch;
  p.k_src = static_cast<const uint16_t*>(k_new);
  p.v_src = static_cast<const uint16_t*>(v_new);
  p.seq_lens = seq_lens_after;
  p.y_out = y_out;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return desc->head_dim == 128 ? oscar::launch_append<128>(p, st) : oscar::launch_append<64>(p, st);
}

oscar_status oscar_quantize_append(const oscar_cache_desc* desc, const void* k_new,
                                   const void* v_new, const int32_t* seq_lens_after,
                                   int32_t batch, void* stream) {
  return oscar_quantize_append_trace(desc, k_new, v_new, seq_lens_after, batch, nullptr, stream);
}

}  // extern "C"
