/* A plain C99 caller of the library's host calls, built against include/oscar.h
 * and linked to liboscar.so, with no Python in between.
 *
 * Usage: host_calls IN OUT
 *   IN : int32 d, int32 g, int64 n, then float32 q[n][g][d], float32 x[n][d]
 *   OUT: int32 status of each call (3 of them), int32 version, then
 *        double C[d][d] (query covariance of q), float R32[d][d] and
 *        double eigenvalues[d] (rotation built from C), float clip (99.9th
 *        percentile of |x R32|), then the text of oscar_status_string(-3) and
 *        a NUL.
 * Exit status 0 when every call returned OSCAR_OK, 1 on an I/O error, 2 when
 * a call failed (its status is still written). */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "oscar.h"

static int read_all(FILE* f, void* p, size_t bytes) { return fread(p, 1, bytes, f) == bytes; }
static int write_all(FILE* f, const void* p, size_t bytes) { return fwrite(p, 1, bytes, f) == bytes; }

int main(int argc, char** argv) {
  if (argc != 3) return 1;
  FILE* in = fopen(argv[1], "rb");
  if (!in) return 1;
  int32_t d = 0, g = 0;
  int64_t n = 0;
  if (!read_all(in, &d, 4) || !read_all(in, &g, 4) || !read_all(in, &n, 8) || d < 2 || d > 256 ||
      g < 1 || n < 1) {
    fclose(in);
    return 1;
  }
  const size_t nq = (size_t)n * (size_t)g * (size_t)d, nx = (size_t)n * (size_t)d;
  const size_t dd = (size_t)d * (size_t)d;
  float* q = malloc(nq * sizeof(float));
  float* x = malloc(nx * sizeof(float));
  double* c = malloc(dd * sizeof(double));
  float* r32 = malloc(dd * sizeof(float));
  double* ev = malloc((size_t)d * sizeof(double));
  if (!q || !x || !c || !r32 || !ev || !read_all(in, q, nq * sizeof(float)) ||
      !read_all(in, x, nx * sizeof(float))) {
    fclose(in);
    return 1;
  }
  fclose(in);
  float clip = 0.f;
  int32_t st[3];
  st[0] = oscar_query_covariance(d, g, n, q, c);
  st[1] = oscar_build_rotation(d, c, x, n, 99.9, OSCAR_VARIANT_OSCAR, NULL, r32, &clip, ev);
  /* a missing C must be refused (reported as OSCAR_OK here when it is) */
  {
    float r_unused[4], clip_unused;
    st[2] = oscar_build_rotation(2, NULL, x, n, 99.9, OSCAR_VARIANT_OSCAR, NULL, r_unused,
                                 &clip_unused, NULL) == OSCAR_ERR_INVALID_ARG ? OSCAR_OK : -100;
  }
  const int32_t version = oscar_version();
  const char* text = oscar_status_string(OSCAR_ERR_WORKSPACE);
  FILE* out = fopen(argv[2], "wb");
  if (!out) return 1;
  int ok = write_all(out, st, sizeof st) && write_all(out, &version, 4) &&
           write_all(out, c, dd * sizeof(double)) && write_all(out, r32, dd * sizeof(float)) &&
           write_all(out, ev, (size_t)d * sizeof(double)) && write_all(out, &clip, 4) &&
           write_all(out, text, strlen(text) + 1);
  fclose(out);
  free(q); free(x); free(c); free(r32); free(ev);
  if (!ok) return 1;
  for (int i = 0; i < 3; ++i)
    if (st[i] != OSCAR_OK) return 2;
  return 0;
}
