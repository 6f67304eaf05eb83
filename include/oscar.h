/*
 * oscar.h -- C ABI of the OSCAR mixed-precision INT2 KV-cache library (sm_103a).
 *
 * The library implements the online serving path of OSCAR (Offline Spectral
 * Covariance-Aware Rotation for 2-bit KV cache quantisation) and the offline
 * rotation builder that feeds it.  Sources, cited by page and section:
 *   [Summary]  "Technical Summary: OSCAR - Offline Spectral Covariance-Aware
 *              Rotation for 2-bit KV Cache Quantization" (gist.science);
 *   [Abstract] the arXiv abstract on the page "OSCAR: Offline Spectral
 *              Covariance-Aware Rotation for 2-bit KV Cache Quantization".
 *
 * Conventions shared by every call
 *   - Activations are row vectors; a rotation acts on the right: y = x R.
 *   - Pointers documented "device" must be device memory of the current CUDA
 *     device; "host" pointers are ordinary host memory.  All memory is owned
 *     by the caller; the library never allocates device memory, never frees
 *     anything and never synchronises a stream.
 *   - Argument errors are detected on the host and returned before any kernel
 *     is launched.  A launch failure returns OSCAR_ERR_CUDA (cudaGetLastError).
 *     Faults found inside kernels (an out-of-range page id, a wait that ran out
 *     of time) are never trapped: the kernel skips the bad access and ORs a bit
 *     into the optional device word desc->status (see OSCAR_DEVERR_*).
 *   - `stream` is a cudaStream_t passed as void*; 0 means the legacy stream.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the kernel before it on the stream drains, and reads that
 *     kernel's results only after waiting for it.  The rotations desc->r_k and
 *     desc->r_v are constants of the layer and are read before that wait, so
 *     the kernel launched immediately before a call on its stream must not
 *     write them (any copy or other stream-ordered work in between suffices).
 *   - Calls are stateless and may be issued from several host threads.
 *
 * Cache format (one layer).  Page size 16 tokens, quantisation group 32
 * channels, head_dim d in {64, 128}, G = num_q_heads / num_kv_heads in
 * {1, 2, 4, 8, 16} (G = 16 is served as two halves of 8 query heads, each of
 * which reads the KV head's pages).  A sequence of length L (current token included) keeps tokens
 * t < sink and t >= L - window in BF16 pages, and tokens sink <= t < L - window
 * in INT2 pages [Summary 2.2B, "Mixed-Precision Layout"].  Logical page
 * p = t / 16 of sequence b maps to a physical page through two tables of int32
 * ids, int2_page_table[b * max_pages_per_seq + p] and bf16_page_table[...]
 * (-1 = none); equal ids in several rows share a page (prefix caching,
 * [Summary 2.2B "Kernel Integration"], [Summary 3.3]).
 *   INT2 pool: num_int2_pages * num_kv_heads blocks of 12*d bytes; block
 *     (page, head) at byte (page*num_kv_heads + head)*12*d holds, for the 16
 *     slots, key codes (4d B), key fp16 (scale, zero) pairs (2d B), value codes
 *     (4d B), value fp16 scales (d B) and zeros (d B), in the fragment order
 *     documented in int2_rotated_kv_gb300/csrc/layout.cuh.
 *   BF16 pool: num_bf16_pages * num_kv_heads blocks of 64*d bytes (keys then
 *     values, 16*d bf16 each, same fragment order).
 * Stored INT2 values are, per group of 32 rotated channels, code*s + z with
 * s = fp16((max-min)/3), z = fp16(min) of the clipped group and
 * code = round-half-even((y_clipped - z)/s) in [0, 3] (0 when s == 0).  A
 * group whose rotated values are not all finite (a NaN or an infinity in the
 * token's input makes every rotated value non-finite) is stored as a zero group,
 * s = z = 0 and codes 0, and OSCAR_DEVERR_NONFINITE is set.  BF16 tokens are
 * stored as given, NaN included.
 *
 * INT4 variant (desc->code_bits = 4; a format beside the pages' INT2, for the
 * comparison with INT4 caches in [Summary 4]): sixteen levels, s = fp16((max -
 * min)/15), codes in [0, 15].  A code c is stored as two 2-bit planes, c >> 2
 * in plane 0 and c & 3 in plane 1, each in the INT2 code order; the block of a
 * (page, head) is 20*d bytes: key planes (2 x 4d B), key (scale, zero) pairs
 * (2d B), value planes (2 x 4d B), value scales (d B) and zeros (d B).  Every
 * device call accepts either width; the BF16 pool is the same.
 */
#ifndef OSCAR_H_
#define OSCAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int oscar_status;
#define OSCAR_OK 0
#define OSCAR_ERR_INVALID_ARG (-1)   /* null pointer, negative size, bad combination   */
#define OSCAR_ERR_UNSUPPORTED (-2)   /* shape outside the supported set                 */
#define OSCAR_ERR_WORKSPACE (-3)     /* workspace too small                             */
#define OSCAR_ERR_CUDA (-4)          /* a CUDA runtime call or a launch failed          */
#define OSCAR_ERR_NOT_CONVERGED (-5) /* eigen-solver did not converge / degenerate gap  */

/* bits ORed into *desc->status by kernels (never trapped) */
#define OSCAR_DEVERR_PAGE_ID 1       /* a page id outside [0, num_pages) was skipped    */
#define OSCAR_DEVERR_TIMEOUT 2       /* an mbarrier wait ran out of time                */
#define OSCAR_DEVERR_SEQ_LEN 4       /* a length or position outside its valid range    */
#define OSCAR_DEVERR_NONFINITE 8     /* a group of rotated values held a NaN or an
                                        infinity; it was stored as a zero group
                                        (s = z = 0, codes 0)                            */

#define OSCAR_VARIANT_OSCAR 0        /* R = U H P_br                                    */
#define OSCAR_VARIANT_HADAMARD 1     /* R = H (data-oblivious baseline)                 */
#define OSCAR_VARIANT_IDENTITY 2     /* R = I (unrotated baseline)                      */

typedef struct oscar_cache_desc {
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t head_dim;                /* 64 or 128                                       */
  int32_t sink;                    /* BF16 tokens at the start (>= 0)                 */
  int32_t window;                  /* BF16 recent tokens (>= 1)                       */
  int32_t max_pages_per_seq;       /* row length of both page tables                  */
  int64_t num_int2_pages;          /* physical pages in the INT2 pool                 */
  int64_t num_bf16_pages;          /* physical pages in the BF16 pool                 */
  void* int2_pool;                 /* device, see format above                        */
  void* bf16_pool;                 /* device                                          */
  const int32_t* int2_page_table;  /* device [batch][max_pages_per_seq]               */
  const int32_t* bf16_page_table;  /* device [batch][max_pages_per_seq]               */
  const float* r_k;                /* device [num_kv_heads][d][d], y = x R_K, 16-B aligned */
  const float* r_v;                /* device [num_kv_heads][d][d], 16-byte aligned    */
  const float* clip_k;             /* device [num_kv_heads]                           */
  const float* clip_v;             /* device [num_kv_heads]                           */
  int32_t* status;                 /* optional device word (OSCAR_DEVERR_* bits)      */
  int32_t code_bits;               /* 2 (or 0): INT2 pages; 4: the INT4 variant       */
} oscar_cache_desc;

/* ---------------------------------------------------------------- host calls */

/* Query-aware key target C_Q = (1/N) sum_n q_n^T q_n [Summary 2.1, 2.2A.1].
 * q: host fp32 [n][g][d] calibration queries of the g query heads that read one
 * KV head (pooled: the sum runs over n and g, normaliser n*g).
 * c_out: host fp64 [d][d].  Synchronous, no CUDA. */
oscar_status oscar_query_covariance(int32_t d, int32_t g, int64_t n, const float* q,
                                    double* c_out);

/* Score-aware value target C_S = (1/N) V^T S^T S V [Summary 2.1, 2.2A.1], with S
 * the post-softmax causal attention probabilities (scale 1/sqrt(d)) of each of
 * the g query heads over one calibration sequence: C_S = (1/(n g)) sum_h
 * (S_h V)^T (S_h V).  q: host fp32 [n][g][d]; k, v: host fp32 [n][d].
 * d must be a multiple of 4.  num_threads <= 0 uses every hardware thread.
 * c_out: host fp64 [d][d]. */
oscar_status oscar_score_covariance(int32_t d, int32_t g, int64_t n, const float* q,
                                    const float* k, const float* v, int32_t num_threads,
                                    double* c_out);

/* Offline rotation and clip for one (layer, KV head, K or V) [Summary 2.2A.2-4]:
 * eigen-decompose C (Jacobi, fp64), order eigenvectors by descending eigenvalue,
 * make the largest-magnitude entry of each column positive (ties: lowest row),
 * form R = U H P_br (H the normalised Sylvester Hadamard, P_br[i][br(i)] = 1),
 * round R to fp32, and set clip = the `percentile` (linear interpolation between
 * order statistics) of |calib_x R32| over all n*d entries.
 * variant: OSCAR_VARIANT_* (HADAMARD and IDENTITY ignore c).
 * c: host fp64 [d][d] symmetric; calib_x: host fp32 [n][d]; n >= 1.
 * Outputs (host): r64_out [d][d] (nullable), r32_out [d][d], clip_out [1],
 * eigvals_out [d] (nullable).  d must be a power of two in [2, 256].
 * Returns OSCAR_ERR_NOT_CONVERGED if the sweep limit is hit or two eigenvalues
 * are closer than 1e-12 * ||C|| (the eigenbasis would not be unique). */
oscar_status oscar_build_rotation(int32_t d, const double* c, const float* calib_x, int64_t n,
                                  double percentile, int32_t variant, double* r64_out,
                                  float* r32_out, float* clip_out, double* eigvals_out);

/* ------------------------------------------------------------- device calls */

/* Bulk placement of prompt tokens [Summary 2.2B]: every token i of the list
 * (sequence seq_ids[i], position positions[i]) is written either to its BF16
 * slot (when it is a sink or recent token for the sequence's final length
 * seq_lens_final[seq]) or rotated by R_K / R_V, clipped, quantised and packed
 * into its INT2 slot.  k, v: device bf16 [total_tokens][num_kv_heads][d];
 * seq_ids, positions: device int32 [total_tokens]; seq_lens_final: device int32
 * [num_seqs], indexed by sequence id (ids must lie in [0, num_seqs) and index
 * rows of the page tables).  Tokens sharing a page are fine; two tokens with
 * the same (sequence, position) race.  Asynchronous on `stream`. */
oscar_status oscar_prefill_quantize(const oscar_cache_desc* desc, const void* k, const void* v,
                                    const int32_t* seq_ids, const int32_t* positions,
                                    const int32_t* seq_lens_final, int32_t num_seqs,
                                    int64_t total_tokens, void* stream);

/* One decode step of cache maintenance for `batch` sequences [Summary 2.2B]:
 * sequence b's new token (position L-1, L = seq_lens_after[b]) is written to its
 * BF16 slot, and when L > sink + window the token at position L-1-window, which
 * has just left the recent window, is read from its BF16 slot, rotated, clipped,
 * quantised and packed into its INT2 slot.  k_new, v_new: device bf16
 * [batch][num_kv_heads][d]; seq_lens_after: device int32 [batch].  The caller
 * allocates the pages beforehand.  Asynchronous. */
oscar_status oscar_quantize_append(const oscar_cache_desc* desc, const void* k_new,
                                   const void* v_new, const int32_t* seq_lens_after,
                                   int32_t batch, void* stream);

/* Diagnostic forms of the two placement calls: the same kernels, the same pool
 * bytes, and in addition the fp32 rotated values y = x R that each INT2
 * placement computed before clipping, so that a test can check the rotation
 * (against x R in higher precision) apart from the decisions that follow it
 * (clip, group range, s, z, codes: a function of y alone).  The pages describe
 * no such output.
 *   oscar_prefill_quantize_trace: y_out device fp32
 *     [total_tokens][num_kv_heads][2][d] (index 0 keys, 1 values); rows of
 *     tokens placed in BF16 slots are not written.
 *   oscar_quantize_append_trace: y_out device fp32 [batch][num_kv_heads][2][d],
 *     the values of the token that leaves the window (rows of sequences with
 *     no leaving token are not written).
 * y_out 16-byte aligned or null (null: the plain call).  Other arguments as
 * oscar_prefill_quantize / oscar_quantize_append. */
oscar_status oscar_prefill_quantize_trace(const oscar_cache_desc* desc, const void* k,
                                          const void* v, const int32_t* seq_ids,
                                          const int32_t* positions, const int32_t* seq_lens_final,
                                          int32_t num_seqs, int64_t total_tokens, float* y_out,
                                          void* stream);
oscar_status oscar_quantize_append_trace(const oscar_cache_desc* desc, const void* k_new,
                                         const void* v_new, const int32_t* seq_lens_after,
                                         int32_t batch, float* y_out, void* stream);

/* Bytes of device workspace oscar_decode_attention / _bf16 need for this batch
 * and maximum sequence length (depends on the device's SM count). */
size_t oscar_decode_workspace_size(const oscar_cache_desc* desc, int32_t batch,
                                   int32_t max_seq_len);

/* Decode attention over the mixed cache [Summary 2.2B "Kernel Integration"],
 * [Abstract]: out[b][hq] = softmax(q k~^T / sqrt(d)) v~ over the L = seq_lens[b]
 * tokens of sequence b, where query head hq reads KV head hq / G, BF16 tokens
 * are used as stored and INT2 tokens stand for k~ = y_hat_K R_K^T,
 * v~ = y_hat_V R_V^T.  The kernel never forms k~ or v~: it rotates the query
 * once (q R_K), attends in the rotated basis, and rotates the INT2 part of the
 * output back once (o R_V^T); split-K partials are merged with log-sum-exp.
 * q, out: device bf16 [batch][num_q_heads][d]; seq_lens: device int32 [batch]
 * (each in [1, max_seq_len], max_seq_len <= 16 * max_pages_per_seq);
 * workspace: device, >= oscar_decode_workspace_size bytes, 16-byte aligned,
 * no initial contents required.  Asynchronous. */
oscar_status oscar_decode_attention(const oscar_cache_desc* desc, const void* q,
                                    const int32_t* seq_lens, int32_t batch, int32_t max_seq_len,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Same-design BF16 baseline [Summary 4, the BF16 comparison]: every token of
 * every sequence is read from the BF16 pool through bf16_page_table; the INT2
 * fields of desc are ignored.  Arguments as oscar_decode_attention. */
oscar_status oscar_decode_attention_bf16(const oscar_cache_desc* desc, const void* q,
                                         const int32_t* seq_lens, int32_t batch,
                                         int32_t max_seq_len, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* Attention for several query rows per sequence over the mixed cache: a chunk
 * of new tokens (chunked prefill after a prefix-cache hit) or tokens to verify
 * ("Technical Summary: OSCAR ...", section 2.2B: compatibility with paged KV
 * serving and prefix caching).  The cache holds seq_lens[b] tokens of sequence
 * b, the rows' own tokens included (placed beforehand with
 * oscar_prefill_quantize or oscar_quantize_append), in the form a sequence of
 * that length stores them; row m of sequence b attends to the stored tokens at
 * positions 0 .. q_pos[b * m_rows + m] (causal).
 *   q, out:  bf16 [batch][m_rows][Hq][d], device.
 *   q_pos:   int32 [batch][m_rows], device.  A position outside
 *            [0, seq_lens[b]) gives a zero output row and sets
 *            OSCAR_DEVERR_SEQ_LEN in desc->status.
 *   workspace: oscar_multiquery_workspace_size(desc, batch, m_rows,
 *            max_seq_len) bytes, no initial contents required.
 * Rows of one sequence share page reads: a CTA serves 8 / G consecutive rows
 * of a sequence (G = num_q_heads / num_kv_heads, at most 8 per CTA), so the
 * tensor-core tile's eight query columns carry G heads of each of those rows;
 * G >= 8 reads the pages once per row.  Asynchronous. */
oscar_status oscar_multiquery_attention(const oscar_cache_desc* desc, const void* q,
                                        const int32_t* seq_lens, const int32_t* q_pos,
                                        int32_t batch, int32_t m_rows, int32_t max_seq_len,
                                        void* out, void* workspace, size_t workspace_bytes,
                                        void* stream);

/* One decode step over the mixed cache: oscar_quantize_append (the new token
 * into its BF16 slot, the token leaving the recent window rotated, clipped,
 * quantised and packed into its INT2 slot) followed by oscar_decode_attention
 * at the new lengths, as one fused pipeline ("Technical Summary: OSCAR ...",
 * section 2.2B: compatibility with fused kernel pipelines).  The append kernel
 * also computes the step's rotated query q' = q R_K, so no separate rotation
 * kernel runs; the attention kernels copy the pages the append writes only
 * after it has completed.  Arguments: q, out as oscar_decode_attention;
 * k_new, v_new, seq_lens_after as oscar_quantize_append (seq_lens_after is the
 * length including the new token); workspace as oscar_decode_attention (the
 * same size).  Result equals the two calls in sequence. */
oscar_status oscar_decode_step(const oscar_cache_desc* desc, const void* q, const void* k_new,
                               const void* v_new, const int32_t* seq_lens_after, int32_t batch,
                               int32_t max_seq_len, void* out, void* workspace,
                               size_t workspace_bytes, void* stream);

/* oscar_decode_step with the rotary position embedding of the serving model
 * applied to the step's new query and key first (the fused pipeline of a
 * decode layer, [Abstract] "fused kernel pipelines"): for the new token at
 * position m = seq_lens_after[b] - 1, every head vector x of q and k_new is
 * rotated pairwise, (x_i, x_{i+d/2}) -> (x_i cos a - x_{i+d/2} sin a,
 * x_{i+d/2} cos a + x_i sin a), a = m * rope_base^(-2i/d), i < d/2 (the
 * rotate-half arrangement over the whole head, as in Qwen3), and rounded to
 * bf16; the rotated key enters the cache, the rotated query attends.  Angles
 * are formed and reduced modulo 2 pi in fp64, cos/sin and the rotation in fp32.
 * v_new is not rotated.  Tokens already in the cache are used as stored (they
 * were rotated when they entered).  rope_base > 1 and finite
 * (else OSCAR_ERR_INVALID_ARG); the workspace is oscar_decode_workspace_size
 * bytes, as for oscar_decode_step. */
oscar_status oscar_decode_step_rope(const oscar_cache_desc* desc, const void* q, const void* k_new,
                                    const void* v_new, const int32_t* seq_lens_after,
                                    int32_t batch, int32_t max_seq_len, double rope_base,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Bytes of device staging that oscar_decode_step_host needs for `batch`
 * sequences: the step's inputs (see below), then, from the next multiple of
 * 256 bytes, the device copy of the output.  0 for an invalid descriptor or
 * batch < 1. */
size_t oscar_decode_step_host_staging_size(const oscar_cache_desc* desc, int32_t batch);

/* The fused decode step (oscar_decode_step, or oscar_decode_step_rope when
 * rope_base > 0) for a caller whose step tensors live in host memory, as in a
 * serving loop that receives the new token's projections from the host.
 *   in_host: host, contiguous bf16, in this order: q [batch][Hq][d], k_new
 *     [batch][Hkv][d], v_new [batch][Hkv][d]
 *     (oscar_decode_step_host_staging_size's input part, batch*(Hq+2Hkv)*d*2 bytes).
 *   out_host: host, bf16 [batch][Hq][d], written when the stream reaches the end
 *     of the call.
 *   staging: device, 16-byte aligned, staging_bytes >=
 *     oscar_decode_step_host_staging_size(desc, batch).
 *   seq_lens_after, workspace, max_seq_len: as oscar_decode_step (device).
 * When both host buffers are page-locked memory mapped into the device's
 * address space (cudaHostAlloc memory under unified addressing, or
 * cudaHostRegister'ed with mapping; each range's first and last bytes are
 * checked with cudaPointerGetAttributes), the step's kernels read q, k_new and
 * v_new from in_host and write the output to out_host in place, over the
 * CPU-GPU link.  Otherwise one host-to-device copy of in_host into staging
 * precedes the kernels and one device-to-host copy of the output follows them
 * (asynchronous only for page-locked memory).  Everything is queued on
 * `stream`; the call returns once the work is queued: synchronise the stream
 * before reading out_host or reusing in_host.  Every argument is checked
 * before anything is queued: OSCAR_ERR_INVALID_ARG for a null or misaligned
 * buffer or a rope_base that is neither 0 (no rotary embedding) nor finite and
 * > 1, OSCAR_ERR_WORKSPACE for staging or workspace that is
 * too small, then oscar_decode_step's errors; OSCAR_ERR_CUDA when a copy cannot
 * be queued.  Result: the bytes oscar_decode_step writes to its `out` and the
 * cache, with the same inputs. */
oscar_status oscar_decode_step_host(const oscar_cache_desc* desc, const void* in_host,
                                    const int32_t* seq_lens_after, int32_t batch,
                                    int32_t max_seq_len, double rope_base, void* out_host,
                                    void* staging, size_t staging_bytes, void* workspace,
                                    size_t workspace_bytes, void* stream);

/* oscar_decode_attention for callers that cannot allocate device memory.
 * The pages describe no counterpart; it exists because some callers have no
 * allocator at hand when they run attention: a plug-in inside a runtime that
 * owns every device allocation, or a latency-bound loop that must never enter
 * the allocator (which may synchronise or fail under memory pressure).  Instead
 * of a workspace argument the call uses one 16 MiB scratch buffer compiled into
 * the library; every GPU that loads the library reserves it until the process
 * exits.  Shapes whose workspace (oscar_decode_workspace_size) exceeds it return
 * OSCAR_ERR_WORKSPACE before any launch.  The call allocates nothing (no
 * cudaMalloc, no cudaFree, no allocating library routine); the buffer needs no
 * initial contents, since every call writes each byte it later reads.  All
 * calls share the one buffer: calls whose kernels overlap on the GPU (streams
 * without ordering between them, or several host threads) race and give wrong
 * results -- serialise them.  The first call on a device looks up the buffer's
 * device address (cudaGetSymbolAddress) with that device current; make that
 * first call before any stream capture.  Other arguments as
 * oscar_decode_attention. */
oscar_status oscar_decode_attention_static(const oscar_cache_desc* desc, const void* q,
                                           const int32_t* seq_lens, int32_t batch,
                                           int32_t max_seq_len, void* out, void* stream);

/* ------------------------------------------------- calibration on the device
 *
 * The three statistics the offline step gathers per layer [Summary 2.1],
 * [Summary 2.2A.1, 2.2A.4], computed on the GPU for long calibration sets and
 * many layers; the eigendecomposition stays on the host (oscar_build_rotation
 * takes the fp64 C these calls write).  Calibration tokens are one causal
 * sequence of n tokens in the prefill's token-major layout:
 *   q: device bf16 [n][num_q_heads][d]; k, v, x: device bf16 [n][num_kv_heads][d].
 * Shapes: d in {64, 128}, G = num_q_heads / num_kv_heads in {1, 2, 4, 8, 16},
 * 1 <= n <= 2^24 (else OSCAR_ERR_UNSUPPORTED / INVALID_ARG).  Pointers 16-byte
 * aligned.  The calls are asynchronous on `stream`, allocate nothing and use
 * the caller's workspace of at least oscar_calibration_workspace_size() bytes
 * (one size serves all three calls; calls sharing a workspace must not overlap
 * on the GPU).  Precision: bf16 inputs, products exact in fp32, fp32
 * accumulation over at most 128 rows before a compensated (two-float) running
 * sum; the result is rounded to fp64 (covariances) or fp32 (clip) at the end. */

/* Workspace bytes for the calibration calls of one layer; 0 for an unsupported
 * shape.  Depends on the current device's SM count. */
size_t oscar_calibration_workspace_size(int32_t num_kv_heads, int32_t num_q_heads, int32_t d,
                                        int64_t n);

/* C_Q for every KV head [Summary 2.1 keys, 2.2A.1]: c_out[h] = (1/(n G))
 * sum_t sum_{g<G} q[t][hG+g]^T q[t][hG+g] (the G query heads that read KV head
 * h pooled).  c_out: device fp64 [num_kv_heads][d][d]. */
oscar_status oscar_query_covariance_device(int32_t num_kv_heads, int32_t num_q_heads, int32_t d,
                                           int64_t n, const void* q, double* c_out,
                                           void* workspace, size_t workspace_bytes, void* stream);

/* C_S for every KV head [Summary 2.1 values, 2.2A.1]: for each query head
 * hq = hG+g, O = S V with S the causal softmax(q_hq k_h^T / sqrt(d))
 * probabilities over the calibration sequence; c_out[h] = (1/(n G)) sum_g O^T O.
 * O is formed in fp32 with the probabilities carried as a bf16 (hi, lo) pair
 * and kept in the workspace as a bf16 (hi, lo) pair.  c_out: device fp64
 * [num_kv_heads][d][d]. */
oscar_status oscar_score_covariance_device(int32_t num_kv_heads, int32_t num_q_heads, int32_t d,
                                           int64_t n, const void* q, const void* k, const void* v,
                                           double* c_out, void* workspace, size_t workspace_bytes,
                                           void* stream);

/* Clip per KV head [Summary 2.2A.4]: clip_out[h] = the `percentile` (0..100,
 * linear interpolation between order statistics, as oscar_build_rotation) of
 * |x[:, h, :] R_h| over all n*d entries, with y = x R_h formed in fp32
 * (sequential FMA over the input channel) and the order statistics selected
 * exactly among those fp32 values.  r: device fp32 [num_kv_heads][d][d] (the
 * cache's r_k or r_v); clip_out: device fp32 [num_kv_heads]. */
oscar_status oscar_clip_threshold_device(int32_t num_kv_heads, int32_t d, int64_t n, const void* x,
                                         const float* r, double percentile, float* clip_out,
                                         void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace oscar_multiquery_attention needs for `batch`
 * sequences of m_rows query rows each (depends on the device's SM count);
 * 0 for invalid arguments. */
size_t oscar_multiquery_workspace_size(const oscar_cache_desc* desc, int32_t batch, int32_t m_rows,
                                       int32_t max_seq_len);

/* Number of SMs the split heuristics assume for the current device (>= 1). */
int32_t oscar_device_sm_count(void);

/* Static text for a status code. */
const char* oscar_status_string(oscar_status s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t oscar_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H_ */
