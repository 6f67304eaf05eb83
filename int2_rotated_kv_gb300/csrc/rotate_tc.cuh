// Bulk prefill on the 5th-generation tensor cores: rotate (y = x R), clip,
// INT2-quantise and pack a list of tokens into the mixed cache.
//
// "Technical Summary: OSCAR ...", section 2.2B: sink and recent tokens stay
// BF16, the middle history is stored in INT2 after the fixed rotation and
// clipping.  Same result, byte for byte, as the prefill mode of
// quantize_kernel (which keeps serving the one-token-per-sequence append).
//
// The rotation of a prompt is a dense (tokens x d) x (d x d) product per KV
// head and K/V; on FP32 FMAs it keeps the kernel ALU-bound far above its memory
// time.  Here it runs as tcgen05.mma (kind::f16: bf16 operands, fp32
// accumulation in tensor memory).  x is bf16 already, an exact operand.  R
// (fp32) is split into three bf16 pieces, each the bf16 rounding of what the
// earlier pieces leave (R = R1 + R2 + R3 to ~2^-24 relative); every product
// x * Ri is exact in fp32, so y = x R1 + x R2 + x R3 keeps the accuracy of an
// fp32 rotation.
//
// One CTA per SM (persistent), serving one (KV head, K or V) pair:
//   warp 0     TMA producer: 128-token x d tiles of x, 128-byte swizzled, into a
//              ring of 3 stages;
//   warp 1     allocates 2d TMEM columns (two fp32 accumulators of 128 lanes x
//              d) and, from one lane, issues 3 * d/16 MMAs (M = 128 tokens,
//              N = d, K = 16) per tile; tcgen05.commit frees the ring stage and
//              publishes the accumulator;
//   warps 2, 3 destinations, alternate tiles: each token's INT2 or BF16 slot
//              (sequence, length and page-table lookups) for tiles ahead, into
//              a shared ring (one warp alone needed most of a tile's time);
//   warps 4..  epilogue, d/32 warpgroups: a warp reads TMEM lanes 32*(w%4) ..
//              +31 (one token per thread) and one group of 32 columns, then in
//              the thread's own registers: clip, min/max, s16, z16, codes, and
//              the stores into the page format (each byte of the format holds
//              codes of one token, so no two threads ever write the same byte).
// The B operand (R^T in three pieces, K-major, 128-byte swizzled) is built once
// per CTA in shared memory.  Every wait is bounded; a CTA that gives up drains
// its copies and MMAs in flight before it frees tensor memory.
#pragma once

#include <cuda_bf16.h>

namespace oscar {

constexpr int kTcM = 128;          // tokens per tile (MMA M, TMEM lanes)
constexpr int kTcStages = 3;
constexpr int kTcMeta = 4;         // tiles of destinations resolved ahead

template <int D>
struct TcSmem {
  static constexpr int kPiece = D * D * 2;                  // one bf16 piece of R^T
  static constexpr int kStage = kTcM * D * 2;               // one A tile
  static constexpr int kAtomA = kTcM * 128;                 // 64-channel swizzle atom of A
  static constexpr int kAtomB = D * 128;                    // same for B (N = d rows)
  static constexpr int kB = 0;
  static constexpr int kA = 3 * kPiece;
  static constexpr int kMeta = kA + kTcStages * kStage;     // int [kTcMeta][2][128]: INT2, BF16 slot
  static constexpr int kBars = kMeta + kTcMeta * 2 * kTcM * 4;
  // u64: full[3] empty[3] acc_full[2] acc_empty[2] meta_full[4] meta_empty[4]
  static constexpr int kMisc = kBars + 24 * 8;              // u32 tmem base, int abort, int issued, int mma_done
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kEpiWarps = 4 * (D / 32);            // one warp per (lane quarter, group)
  static constexpr int kThreads = 32 * (4 + kEpiWarps);
  static constexpr int kAlloc = kBytes + 1024;              // the base is rounded up to 1024 bytes
  static constexpr int kCols = 2 * D;                       // TMEM columns: two accumulators
  static_assert(kA % 1024 == 0 && kStage % 1024 == 0 && kPiece % 1024 == 0,
                "swizzle atoms start on 1024-byte boundaries");
};

// ------------------------------------------------------------ PTX wrappers

// Shared-memory matrix descriptor of a K-major, 128-byte swizzled operand
// (tcgen05 format): start address >> 4 in bits 0-13, leading byte offset (unused
// for swizzled K-major operands) = 1 in bits 16-29, stride byte offset 1024 >> 4
// (8 rows of 128 bytes) in bits 32-45, version 1 in bits 46-47, layout 2
// (128-byte swizzle) in bits 61-63.
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and an
// fp32 accumulator: D format bits 4-5 = 1, A format bits 7-9 = 1, B format bits
// 10-12 = 1, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       int accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on bar once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::
                   "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tc_alloc(uint32_t* dst, int ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, int ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 consecutive fp32 columns of the warp's 32 TMEM lanes (one row per thread),
// waited for inside the same statement so the registers are complete on exit.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

// Byte offset of element (row, k) in a K-major operand of `rows` rows built
// from 64-element (128-byte) swizzle atoms: atom k/64 holds rows x 128 bytes,
// row r at r * 128, its 16-byte chunk c stored at chunk c ^ (r % 8).
__device__ __forceinline__ uint32_t tc_sw128_offset(int row, int k, int rows) {
  const int kin = k & 63;
  return static_cast<uint32_t>((k >> 6) * rows * 128 + row * 128 +
                               ((((kin >> 3) ^ (row & 7)) & 7) << 4) + ((kin & 7) << 1));
}

// ------------------------------------------------------------------ kernel

// Code of one value: rint(fl((y_c - z16) / s16)) clamped to [0, max_code], the
// division correctly rounded.  The product with the reciprocal differs from the
// quotient by ~1e-6 at most (relative), so it decides the code unless it lies
// within 4e-6 * (1 + |q|) of a half-integer; there the exact quotient is taken.
__device__ __forceinline__ int tc_code(float yc, float zf, float sf, float inv, int max_code) {
  const float a = __fsub_rn(yc, zf);
  float q = __fmul_rn(a, inv);
  float r = rintf(q);
  if (fabsf(fabsf(q - r) - 0.5f) < 4e-6f * (1.f + fabsf(q))) r = rintf(__fdiv_rn(a, sf));
  return min(max(static_cast<int>(r), 0), max_code);
}

template <int D, int P>
__global__ void __launch_bounds__(TcSmem<D>::kThreads, 1)
    rotate_tc_kernel(const QuantParams p, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v) {
  using S = TcSmem<D>;
  constexpr int NG = D / 32;
  constexpr int KS = D / 16;          // MMA k-steps per piece
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBars);
  uint64_t* full = bars;
  uint64_t* empty = bars + 3;
  uint64_t* acc_full = bars + 6;
  uint64_t* acc_empty = bars + 8;
  uint64_t* meta_full = bars + 10;
  uint64_t* meta_empty = bars + 14;
  int* meta = reinterpret_cast<int*>(smem + S::kMeta);     // [kTcMeta][2][128]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kMisc + 4);
  volatile int* n_issued = reinterpret_cast<volatile int*>(smem + S::kMisc + 8);
  volatile int* n_mma = reinterpret_cast<volatile int*>(smem + S::kMisc + 12);

  const int h = blockIdx.y, kv = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CUtensorMap* map = kv ? &map_v : &map_k;

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], S::kEpiWarps);
    }
    for (int i = 0; i < kTcMeta; ++i) {
      mbar_init(&meta_full[i], 1);
      mbar_init(&meta_empty[i], S::kEpiWarps);
    }
    *abort_flag = 0;
    *n_issued = 0;
    *n_mma = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc_alloc(tmem_slot, S::kCols);
  // programmatic stream serialisation: inputs are read only after the
  // predecessor grid has completed; then the next kernel may launch
  pdl_wait();
  pdl_trigger();

  // ---- B operand: R^T as three bf16 pieces, K-major (row n, column k = R[k][n])
  const float* rot = (kv ? p.r_v : p.r_k) + static_cast<size_t>(h) * D * D;
  for (int e = tid; e < D * D; e += S::kThreads) {
    const int k = e / D, n = e % D;
    const float r = rot[e];
    const __nv_bfloat16 r1 = __float2bfloat16_rn(r);
    const float e1 = r - __bfloat162float(r1);        // exact: the bits r1 left out
    const __nv_bfloat16 r2 = __float2bfloat16_rn(e1);
    const float e2 = e1 - __bfloat162float(r2);
    const __nv_bfloat16 r3 = __float2bfloat16_rn(e2);
    const uint32_t off = tc_sw128_offset(n, k, D);
    *reinterpret_cast<__nv_bfloat16*>(smem + S::kB + off) = r1;
    *reinterpret_cast<__nv_bfloat16*>(smem + S::kB + S::kPiece + off) = r2;
    *reinterpret_cast<__nv_bfloat16*>(smem + S::kB + 2 * S::kPiece + off) = r3;
  }
  fence_proxy_async();      // generic stores above, tensor-core reads below
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t n_tiles = (p.n_items + kTcM - 1) / kTcM;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int it = 0;
      for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
        const int s = it % kTcStages;
        const uint32_t ph = static_cast<uint32_t>(it / kTcStages) & 1u;
        if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, p.status)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], S::kStage);
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          tma_load_2d(smem + S::kA + s * S::kStage + a * S::kAtomA, map, h * D + 64 * a,
                      static_cast<int>(tile * kTcM), &full[s]);
        *n_issued = it + 1;
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc_bf16(kTcM, D);
      int it = 0;
      for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
        const int s = it % kTcStages;
        const uint32_t ph = static_cast<uint32_t>(it / kTcStages) & 1u;
        const int buf = it & 1;
        const uint32_t pb = static_cast<uint32_t>(it >> 1) & 1u;
        if (*abort_flag || !mbar_wait(&acc_empty[buf], pb ^ 1u, p.status) ||
            !mbar_wait(&full[s], ph, p.status)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * D);
        const uint32_t a0 = sb + S::kA + s * S::kStage;
#pragma unroll
        for (int pc = 0; pc < 3; ++pc) {
          const uint32_t b0 = sb + S::kB + pc * S::kPiece;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t ka = (kk >> 2) * S::kAtomA + (kk & 3) * 32;
            const uint32_t kb = (kk >> 2) * S::kAtomB + (kk & 3) * 32;
            tc_mma(d_tmem, tc_desc_sw128(a0 + ka), tc_desc_sw128(b0 + kb), idesc,
                   (pc | kk) != 0);
          }
        }
        tc_commit(&empty[s]);
        tc_commit(&acc_full[buf]);
        *n_mma = it + 1;
      }
    }
  } else if (warp == 2 || warp == 3) {
    // -------------------------------------------------------- destinations
    // per row: INT2 slot (page * 16 + slot) or -1, BF16 slot likewise
    int it = warp - 2;   // this warp's tiles: every second one of the CTA's
    for (int64_t tile = blockIdx.x + static_cast<int64_t>(warp - 2) * gridDim.x; tile < n_tiles;
         tile += 2 * static_cast<int64_t>(gridDim.x), it += 2) {
      const int s = it % kTcMeta;
      const uint32_t ph = static_cast<uint32_t>(it / kTcMeta) & 1u;
      const bool ok = !*abort_flag && mbar_wait(&meta_empty[s], ph ^ 1u, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      int* mi = meta + s * 2 * kTcM;
      // The four tokens of each lane are resolved level by level, so each level's
      // loads are in flight together: ids and positions, then the sequences'
      // lengths, then the page-table entries (three round trips per tile).
      constexpr int U = kTcM / 32;
      int seq[U], pos[U], L[U], pg[U];
      bool ok2[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t item = tile * kTcM + u * 32 + lane;
        const bool in = item < p.n_items;
        seq[u] = in ? p.seq_ids[item] : -1;
        pos[u] = in ? p.positions[item] : -1;
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        L[u] = (seq[u] >= 0 && seq[u] < p.num_seqs) ? p.seq_lens[seq[u]] : -1;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        ok2[u] = seq[u] >= 0 && seq[u] < p.num_seqs && pos[u] >= 0 && pos[u] < L[u] &&
                 pos[u] / kPage < p.max_pages;
        pg[u] = -1;
        if (ok2[u]) {
          const int64_t trow = static_cast<int64_t>(seq[u]) * p.max_pages + pos[u] / kPage;
          pg[u] = (pos[u] >= p.sink && pos[u] < L[u] - p.window) ? p.int2_pt[trow] : p.bf16_pt[trow];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int row = u * 32 + lane;
        const int64_t item = tile * kTcM + row;
        int i2 = -1, bf = -1;
        if (item < p.n_items) {
          if (!ok2[u]) {
            flag(p.status, OSCAR_DEVERR_SEQ_LEN);
          } else if (pos[u] >= p.sink && pos[u] < L[u] - p.window) {
            if (pg[u] < 0 || pg[u] >= p.n_int2_pages) flag(p.status, OSCAR_DEVERR_PAGE_ID);
            else i2 = pg[u] * kPage + pos[u] % kPage;
          } else {
            if (pg[u] < 0 || pg[u] >= p.n_bf16_pages) flag(p.status, OSCAR_DEVERR_PAGE_ID);
            else bf = pg[u] * kPage + pos[u] % kPage;
          }
        }
        mi[row] = i2;
        mi[kTcM + row] = bf;
      }
      __syncwarp();
      if (lane == 0) tc_arrive(&meta_full[s]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;             // TMEM lanes this warp may read
    const int grp = (warp - 4) >> 2;          // its group of 32 columns
    const int row = 32 * quarter + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const float clip = (kv ? p.clip_v : p.clip_k)[h];
    const uint16_t* src = kv ? p.v_src : p.k_src;
    int it = 0;
    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int buf = it & 1;
      const uint32_t pb = static_cast<uint32_t>(it >> 1) & 1u;
      const int ms = it % kTcMeta;
      const uint32_t mph = static_cast<uint32_t>(it / kTcMeta) & 1u;
      const bool okm = mbar_wait(&meta_full[ms], mph, p.status);
      if (!__all_sync(0xffffffffu, okm)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      const int i2 = meta[ms * 2 * kTcM + row];
      const int bf = meta[ms * 2 * kTcM + kTcM + row];
      __syncwarp();
      if (lane == 0) tc_arrive(&meta_empty[ms]);
      if (bf >= 0) {   // BF16 region: copy this group of the row as it is
        const int64_t item = tile * kTcM + row;
        const uint16_t* xr = src + (item * p.hkv + h) * D + 32 * grp;
        uint16_t* dst = p.bf16_pool + (static_cast<int64_t>(bf / kPage) * p.hkv + h) * (32 * D);
        const int slot = bf % kPage;
#pragma unroll
        for (int j0 = 0; j0 < 32; j0 += 8) {
          const uint4 v = *reinterpret_cast<const uint4*>(xr + j0);
          const uint16_t* ve = reinterpret_cast<const uint16_t*>(&v);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = 32 * grp + j0 + u;
            const int e = kv ? 16 * D + bf16_value_elem(slot, j) : bf16_key_elem(slot, j);
            dst[e] = ve[u];
          }
        }
      }
      const bool ok = mbar_wait(&acc_full[buf], pb, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      tc_fence_after();
      float y[32];
      tc_ld32(tmem + static_cast<uint32_t>(buf * D + 32 * grp) + lane_off, y);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) tc_arrive(&acc_empty[buf]);
      if (i2 < 0) continue;
      if (p.y_out) {   // diagnostic: the rotated values this row's decisions start from
        float4* yo = reinterpret_cast<float4*>(
            p.y_out + ((tile * kTcM + row) * p.hkv + h) * (2 * D) + kv * D + 32 * grp);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4)
          yo[j4] = make_float4(y[4 * j4], y[4 * j4 + 1], y[4 * j4 + 2], y[4 * j4 + 3]);
      }
      const int slot = i2 % kPage;
      using F = Fmt<D, P>;
      constexpr int kMaxCode = P == 2 ? 15 : 3;   // INT4 variant / INT2
      uint8_t* blk = p.int2_pool + (static_cast<int64_t>(i2 / kPage) * p.hkv + h) * F::kInt2Block;
      // Clipping is monotone, so the clipped group's minimum and maximum are
      // the clipped extremes of the raw values, and a value beyond the clip
      // threshold lands on code 0 or the top code either way: the values
      // themselves are never clipped on this path.
      // A NaN carries through min.NaN / max.NaN and an infinity ends up as an
      // extreme, so the group is finite exactly when both extremes are; a
      // non-finite group is stored as a zero group (s = z = 0: every code 0).
      float mn = y[0], mx = y[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) {
        mn = fmin_nan(mn, y[j]);
        mx = fmax_nan(mx, y[j]);
      }
      if (!(isfinite(mn) && isfinite(mx))) {
        flag(p.status, OSCAR_DEVERR_NONFINITE);
        mn = mx = 0.f;
      }
      mn = fminf(fmaxf(mn, -clip), clip);
      mx = fminf(fmaxf(mx, -clip), clip);
      const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), static_cast<float>(kMaxCode)));
      const __half z16 = __float2half_rn(mn);
      const float sf = __half2float(s16), zf = __half2float(z16);
      const bool live = sf != 0.f;            // a zero scale gives code 0 everywhere
      // approximate reciprocal (a few ulp), times 1/top: the quotient stays far
      // inside the near-tie margin below of the correctly rounded one
      const float inv_top = live ? __fdividef(1.0f, sf) * (1.0f / kMaxCode) : 0.f;
      const uint32_t sz = static_cast<uint32_t>(__half_as_ushort(s16)) |
                          (static_cast<uint32_t>(__half_as_ushort(z16)) << 16);
      uint32_t bytes[P][8];
#pragma unroll
      for (int pl = 0; pl < P; ++pl)
#pragma unroll
        for (int b8 = 0; b8 < 8; ++b8) bytes[pl][b8] = 0u;
      // code = round-half-even of the quotient clamped to [0, top] (the same as
      // clamping the rounded quotient).  The clamp is the saturation of
      // t = (y - z) / (s top) to [0, 1] (a free modifier of the multiply; it
      // also turns a NaN into 0); top * t + 1.5 * 2^23 in one fused
      // multiply-add rounds the quotient to an integer held in the low
      // mantissa bits, and a second one gives its distance from that integer.
      // A clamped quotient within 6.4e-5 of a half-integer flags the group for
      // the correctly rounded division; at the clamp bounds both roundings
      // give the same code.
      constexpr float kMagic = 12582912.0f;
      constexpr float kTop = static_cast<float>(kMaxCode);
      float dev = 0.f;
      if constexpr (P == 1) {
        // the codes as small integers in fp32 (r = rint(top t)); byte b holds
        // the codes of values b, b + 8, b + 16, b + 24 at bit positions 0, 4,
        // 2, 6, assembled as r0 + 16 r1 + 4 r2 + 64 r3 (exact) and turned into
        // bits by one more 1.5 * 2^23 addition (the low byte is the value)
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float t = __saturatef(__fmul_rn(__fsub_rn(y[j], zf), inv_top));
          r[j] = __fsub_rn(__fmaf_rn(t, kTop, kMagic), kMagic);
          dev = fmaxf(dev, fabsf(__fmaf_rn(t, kTop, -r[j])));
        }
#pragma unroll
        for (int b8 = 0; b8 < 8; ++b8) {
          const float v = __fmaf_rn(r[b8 + 24], 64.f,
                                    __fmaf_rn(r[b8 + 16], 4.f, __fmaf_rn(r[b8 + 8], 16.f, r[b8])));
          bytes[0][b8] = __float_as_uint(__fadd_rn(v, kMagic));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float t = __saturatef(__fmul_rn(__fsub_rn(y[j], zf), inv_top));
          const float m = __fmaf_rn(t, kTop, kMagic);
          dev = fmaxf(dev, fabsf(__fmaf_rn(t, kTop, -__fsub_rn(m, kMagic))));
          const uint32_t c = __float_as_uint(m);
          const int pos = 4 * ((j >> 3) & 1) + 2 * (j >> 4);
#pragma unroll
          for (int pl = 0; pl < P; ++pl) bytes[pl][j & 7] |= ((c >> (2 * (P - 1 - pl))) & 3u) << pos;
        }
      }
      if (live && dev > 0.5f - 6.4e-5f) {   // rare: the whole group again with the correctly rounded division
#pragma unroll
        for (int pl = 0; pl < P; ++pl)
#pragma unroll
          for (int b8 = 0; b8 < 8; ++b8) bytes[pl][b8] = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float yc = fminf(fmaxf(y[j], -clip), clip);
          const uint32_t c = static_cast<uint32_t>(
              min(max(static_cast<int>(rintf(__fdiv_rn(__fsub_rn(yc, zf), sf))), 0), kMaxCode));
          const int pos = 4 * ((j >> 3) & 1) + 2 * (j >> 4);
#pragma unroll
          for (int pl = 0; pl < P; ++pl) bytes[pl][j & 7] |= ((c >> (2 * (P - 1 - pl))) & 3u) << pos;
        }
      }
      if (kv == 0) {
#pragma unroll
        for (int b8 = 0; b8 < 8; ++b8)
#pragma unroll
          for (int pl = 0; pl < P; ++pl)
            blk[F::kKc + pl * F::kPlane + key_byte<D>(slot, b8 >> 1, grp, b8 & 1)] =
                static_cast<uint8_t>(bytes[pl][b8]);
        reinterpret_cast<uint32_t*>(blk + F::kKsz)[slot * NG + grp] = sz;
      } else {
#pragma unroll
        for (int b8 = 0; b8 < 8; ++b8)
#pragma unroll
          for (int pl = 0; pl < P; ++pl)
            blk[F::kVc + pl * F::kPlane + value_byte<D>(slot, b8, grp)] = static_cast<uint8_t>(bytes[pl][b8]);
        const int e = vsz_index<D>(slot, grp);
        reinterpret_cast<uint16_t*>(blk + F::kVs)[e] = static_cast<uint16_t>(sz & 0xffffu);
        reinterpret_cast<uint16_t*>(blk + F::kVz)[e] = static_cast<uint16_t>(sz >> 16);
      }
    }
  }

  // ---- teardown: after a give-up, let copies and MMAs in flight finish first
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) {
      for (int it = *n_mma; it < *n_issued; ++it)
        mbar_wait(&full[it % kTcStages], static_cast<uint32_t>(it / kTcStages) & 1u, p.status);
    } else if (tid == 32 && *n_mma > 0) {
      const int it = *n_mma - 1;
      mbar_wait(&acc_full[it & 1], static_cast<uint32_t>(it >> 1) & 1u, p.status);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tc_dealloc(tmem, S::kCols);
  }
}

// ------------------------------------------------------------------- host

// 2-D view [rows = tokens][cols = Hkv * d] of a bf16 token-major K or V array;
// boxes of 64 channels x 128 tokens, 128-byte swizzled, zero fill past the end.
inline bool make_token_map(CUtensorMap* m, const void* base, int64_t rows, int cols) {
  oscar_host::TensorMapEncodeTiled enc = oscar_host::tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTcM)};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch the tensor-core prefill; returns false (nothing launched) when the
// inputs do not meet the tensor maps' rules, so the caller can take the
// CUDA-core kernel instead.
template <int D, int P>
bool launch_rotate_tc_p(const QuantParams& p, cudaStream_t st, oscar_status* result) {
  using S = TcSmem<D>;
  if ((reinterpret_cast<uintptr_t>(p.k_src) | reinterpret_cast<uintptr_t>(p.v_src)) & 15)
    return false;
  if (p.n_items >= (int64_t(1) << 31)) return false;
  CUtensorMap mk, mv;
  if (!make_token_map(&mk, p.k_src, p.n_items, p.hkv * D) ||
      !make_token_map(&mv, p.v_src, p.n_items, p.hkv * D))
    return false;
  if (!oscar_host::allow_smem(reinterpret_cast<const void*>(rotate_tc_kernel<D, P>), S::kAlloc)) {
    *result = OSCAR_ERR_CUDA;
    return true;
  }
  const int64_t tiles = (p.n_items + kTcM - 1) / kTcM;
  const int sms = oscar_host::sm_count();
  const int64_t per_pair = std::max<int64_t>(1, sms / (2 * p.hkv));
  const dim3 grid(static_cast<unsigned>(std::min<int64_t>(tiles, per_pair)), p.hkv, 2);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(S::kThreads);
  cfg.dynamicSmemBytes = S::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  *result = cudaLaunchKernelEx(&cfg, rotate_tc_kernel<D, P>, p, mk, mv) == cudaSuccess
                ? OSCAR_OK
                : OSCAR_ERR_CUDA;
  return true;
}

template <int D>
bool launch_rotate_tc(const QuantParams& p, cudaStream_t st, oscar_status* result) {
  return p.planes == 2 ? launch_rotate_tc_p<D, 2>(p, st, result)
                       : launch_rotate_tc_p<D, 1>(p, st, result);
}

}  // namespace oscar
