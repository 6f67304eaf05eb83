/* A plain C11 caller of the library's device calls, with the CUDA runtime API
 * and no Python in between: one sequence's prompt is placed in a mixed cache
 * (oscar_prefill_quantize) and attended by one decode query
 * (oscar_decode_attention).  Both page tables map logical page p to physical
 * page p.
 *
 * Usage: decode_from_c IN OUT
 *   IN : int32 d, hkv, hq, sink, window, L; then bf16 (as uint16) k[L][hkv][d],
 *        v[L][hkv][d], q[hq][d]; fp32 r_k[hkv][d][d], r_v[hkv][d][d],
 *        clip_k[hkv], clip_v[hkv]
 *   OUT: int32 statuses: prefill, decode, the CUDA status after synchronising,
 *        the device status word; then bf16 (as uint16) out[hq][d]
 * Exit status 0 when everything succeeded, 1 on an I/O or allocation error,
 * 2 when a call failed (the statuses are still written). */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "oscar.h"

static int rd(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n; }

static void* dev_copy(const void* host, size_t bytes) {
  void* d = NULL;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
  if (host && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  if (!host && cudaMemset(d, 0, bytes) != cudaSuccess) return NULL;
  return d;
}

int main(int argc, char** argv) {
  if (argc != 3) return 1;
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 1;
  int32_t hdr[6];
  if (!rd(in, hdr, sizeof hdr)) return 1;
  const int32_t d = hdr[0], hkv = hdr[1], hq = hdr[2], sink = hdr[3], window = hdr[4], L = hdr[5];
  if (d != 64 && d != 128) return 1;
  if (hkv < 1 || hq < hkv || L < 1 || L > (1 << 20)) return 1;
  const size_t kv_n = (size_t)L * hkv * d, q_n = (size_t)hq * d, r_n = (size_t)hkv * d * d;
  uint16_t* k = malloc(kv_n * 2);
  uint16_t* v = malloc(kv_n * 2);
  uint16_t* q = malloc(q_n * 2);
  float* rk = malloc(r_n * 4);
  float* rv = malloc(r_n * 4);
  float* ck = malloc((size_t)hkv * 4);
  float* cv = malloc((size_t)hkv * 4);
  if (!k || !v || !q || !rk || !rv || !ck || !cv) return 1;
  if (!rd(in, k, kv_n * 2) || !rd(in, v, kv_n * 2) || !rd(in, q, q_n * 2) || !rd(in, rk, r_n * 4) ||
      !rd(in, rv, r_n * 4) || !rd(in, ck, (size_t)hkv * 4) || !rd(in, cv, (size_t)hkv * 4))
    return 1;
  fclose(in);

  const int32_t pages = (L + 15) / 16, max_pages = pages + 1;
  int32_t* table = malloc((size_t)max_pages * 4);
  int32_t* seq_ids = malloc((size_t)L * 4);
  int32_t* positions = malloc((size_t)L * 4);
  if (!table || !seq_ids || !positions) return 1;
  for (int32_t p = 0; p < max_pages; ++p) table[p] = p < pages ? p : -1;
  for (int32_t t = 0; t < L; ++t) {
    seq_ids[t] = 0;
    positions[t] = t;
  }

  oscar_cache_desc c;
  memset(&c, 0, sizeof c);
  c.num_kv_heads = hkv;
  c.num_q_heads = hq;
  c.head_dim = d;
  c.sink = sink;
  c.window = window;
  c.max_pages_per_seq = max_pages;
  c.num_int2_pages = max_pages;
  c.num_bf16_pages = max_pages;
  c.code_bits = 2;
  c.int2_pool = dev_copy(NULL, (size_t)max_pages * hkv * 12 * d);
  c.bf16_pool = dev_copy(NULL, (size_t)max_pages * hkv * 64 * d);
  c.int2_page_table = dev_copy(table, (size_t)max_pages * 4);
  c.bf16_page_table = dev_copy(table, (size_t)max_pages * 4);
  c.r_k = dev_copy(rk, r_n * 4);
  c.r_v = dev_copy(rv, r_n * 4);
  c.clip_k = dev_copy(ck, (size_t)hkv * 4);
  c.clip_v = dev_copy(cv, (size_t)hkv * 4);
  c.status = dev_copy(NULL, 4);
  void* dk = dev_copy(k, kv_n * 2);
  void* dv = dev_copy(v, kv_n * 2);
  void* dq = dev_copy(q, q_n * 2);
  void* dout = dev_copy(NULL, q_n * 2);
  void* dids = dev_copy(seq_ids, (size_t)L * 4);
  void* dpos = dev_copy(positions, (size_t)L * 4);
  const int32_t len = L;
  void* dlen = dev_copy(&len, 4);
  const size_t ws_bytes = oscar_decode_workspace_size(&c, 1, L);
  void* ws = ws_bytes ? dev_copy(NULL, ws_bytes) : NULL;
  if (!c.int2_pool || !c.bf16_pool || !c.int2_page_table || !c.bf16_page_table || !c.r_k ||
      !c.r_v || !c.clip_k || !c.clip_v || !c.status || !dk || !dv || !dq || !dout || !dids ||
      !dpos || !dlen || !ws)
    return 1;

  int32_t st[4];
  st[0] = oscar_prefill_quantize(&c, dk, dv, dids, dpos, dlen, 1, L, NULL);
  st[1] = oscar_decode_attention(&c, dq, dlen, 1, L, dout, ws, ws_bytes, NULL);
  st[2] = (int32_t)cudaDeviceSynchronize();
  st[3] = -1;
  uint16_t* out = malloc(q_n * 2);
  if (!out) return 1;
  memset(out, 0, q_n * 2);
  if (st[2] == 0) {
    cudaMemcpy(&st[3], c.status, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(out, dout, q_n * 2, cudaMemcpyDeviceToHost);
  }
  FILE* f = fopen(argv[2], "wb");
  if (!f) return 1;
  const int ok = fwrite(st, 4, 4, f) == 4 && fwrite(out, 2, q_n, f) == q_n;
  fclose(f);
  if (!ok) return 1;
  return (st[0] || st[1] || st[2] || st[3]) ? 2 : 0;
}
