// Offline OSCAR calibration on the host (fp64): covariance targets, eigenbasis,
// composite rotation R = U H P_br and clipping threshold.
//
// "Technical Summary: OSCAR - Offline Spectral Covariance-Aware Rotation for
// 2-bit KV Cache Quantization", section 2.1 (the targets Q^T Q and V^T S^T S V)
// and section 2.2, phase A, steps 1-4 (covariance estimation, eigen-
// decomposition, composite rotation, clipping thresholds).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <thread>
#include <vector>

#include "oscar.h"

namespace {

// Cyclic Jacobi eigen-solver for a symmetric matrix (row-major, fp64).  On
// return a holds the eigenvalues on its diagonal and v the eigenvectors as
// columns.  Classic two-sided rotation method (Golub & Van Loan, "Matrix
// Computations", section 8.5): each rotation zeroes one off-diagonal pair.
bool jacobi_eigen(int n, std::vector<double>& a, std::vector<double>& v) {
  v.assign(static_cast<size_t>(n) * n, 0.0);
  for (int i = 0; i < n; ++i) v[i * n + i] = 1.0;
  double fro = 0.0;
  for (double x : a) fro += x * x;
  fro = std::sqrt(fro);
  if (fro == 0.0) return true;
  for (int sweep = 0; sweep < 100; ++sweep) {
    double off = 0.0;
    for (int p = 0; p < n; ++p)
      for (int q = p + 1; q < n; ++q) off += a[p * n + q] * a[p * n + q];
    if (std::sqrt(2.0 * off) <= 1e-15 * fro) return true;
    for (int p = 0; p < n - 1; ++p) {
      for (int q = p + 1; q < n; ++q) {
        const double apq = a[p * n + q];
        if (std::fabs(apq) <= 1e-300) continue;
        const double app = a[p * n + p], aqq = a[q * n + q];
        const double theta = (aqq - app) / (2.0 * apq);
        const double t = (theta >= 0 ? 1.0 : -1.0) /
                         (std::fabs(theta) + std::sqrt(theta * theta + 1.0));
        const double c = 1.0 / std::sqrt(t * t + 1.0);
        const double s = t * c;
        for (int k = 0; k < n; ++k) {        // columns p, q of A
          const double akp = a[k * n + p], akq = a[k * n + q];
          a[k * n + p] = c * akp - s * akq;
          a[k * n + q] = s * akp + c * akq;
        }
        for (int k = 0; k < n; ++k) {        // rows p, q of A
          const double apk = a[p * n + k], aqk = a[q * n + k];
          a[p * n + k] = c * apk - s * aqk;
          a[q * n + k] = s * apk + c * aqk;
        }
        a[p * n + q] = a[q * n + p] = 0.0;
        for (int k = 0; k < n; ++k) {        // accumulate V = V J
          const double vkp = v[k * n + p], vkq = v[k * n + q];
          v[k * n + p] = c * vkp - s * vkq;
          v[k * n + q] = s * vkp + c * vkq;
        }
      }
    }
  }
  return false;
}

int popcount_u32(unsigned x) {
  int c = 0;
  while (x) { c += x & 1u; x >>= 1; }
  return c;
}

int bit_reverse(int i, int bits) {
  int r = 0;
  for (int b = 0; b < bits; ++b)
    if ((i >> b) & 1) r |= 1 << (bits - 1 - b);
  return r;
}

// Linear-interpolation percentile (Hyndman-Fan type 7) of vals, p in [0, 100].
double percentile_linear(std::vector<double>& vals, double p) {
  const size_t n = vals.size();
  const double h = (static_cast<double>(n) - 1.0) * p / 100.0;
  size_t lo = static_cast<size_t>(std::floor(h));
  if (lo >= n - 1) {
    return *std::max_element(vals.begin(), vals.end());
  }
  std::nth_element(vals.begin(), vals.begin() + lo, vals.end());
  const double xlo = vals[lo];
  const double xhi = *std::min_element(vals.begin() + lo + 1, vals.end());
  return xlo + (h - static_cast<double>(lo)) * (xhi - xlo);
}

}  // namespace

extern "C" {

oscar_status oscar_query_covariance(int32_t d, int32_t g, int64_t n, const float* q,
                                    double* c_out) {
  if (d <= 0 || g <= 0 || n <= 0 || !q || !c_out) return OSCAR_ERR_INVALID_ARG;
  std::vector<double> acc(static_cast<size_t>(d) * d, 0.0), row(d);
  const int64_t rows = n * g;
  for (int64_t r = 0; r < rows; ++r) {
    const float* x = q + r * d;
    for (int i = 0; i < d; ++i) row[i] = x[i];
    for (int i = 0; i < d; ++i) {
      const double xi = row[i];
      double* out = acc.data() + static_cast<size_t>(i) * d;
      for (int j = 0; j < d; ++j) out[j] += xi * row[j];
    }
  }
  const double inv = 1.0 / static_cast<double>(rows);
  for (size_t i = 0; i < acc.size(); ++i) c_out[i] = acc[i] * inv;
  return OSCAR_OK;
}

oscar_status oscar_score_covariance(int32_t d, int32_t g, int64_t n, const float* q,
                                    const float* k, const float* v, int32_t num_threads,
                                    double* c_out) {
  if (d <= 0 || (d % 4) || g <= 0 || n <= 0 || !q || !k || !v || !c_out)
    return OSCAR_ERR_INVALID_ARG;
  int nt = num_threads > 0 ? num_threads : static_cast<int>(std::thread::hardware_concurrency());
  nt = std::max(1, std::min<int>(nt, 256));
  std::vector<double> kd(static_cast<size_t>(n) * d), vd(static_cast<size_t>(n) * d);
  for (size_t i = 0; i < kd.size(); ++i) { kd[i] = k[i]; vd[i] = v[i]; }
  const double scale = 1.0 / std::sqrt(static_cast<double>(d));
  const int64_t work = n * g;   // one unit = one (query row, head)
  std::vector<std::vector<double>> part(nt, std::vector<double>(static_cast<size_t>(d) * d, 0.0));
  auto body = [&](int tid) {
    std::vector<double> logit(n), o(d), qq(d);
    double* acc = part[tid].data();
    // interleaved rows so long causal rows are spread over threads
    for (int64_t u = tid; u < work; u += nt) {
      const int64_t i = u / g;
      const int h = static_cast<int>(u % g);
      const float* qr = q + (i * g + h) * d;
      for (int c = 0; c < d; ++c) qq[c] = qr[c];
      double mx = -INFINITY;
      for (int64_t m = 0; m <= i; ++m) {
        const double* km = kd.data() + m * d;
        // four partial sums keep the FMA pipes busy (d is a multiple of 4)
        double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
        for (int c = 0; c < d; c += 4) {
          s0 += qq[c] * km[c];
          s1 += qq[c + 1] * km[c + 1];
          s2 += qq[c + 2] * km[c + 2];
          s3 += qq[c + 3] * km[c + 3];
        }
        const double s = ((s0 + s1) + (s2 + s3)) * scale;
        logit[m] = s;
        mx = std::max(mx, s);
      }
      double tot = 0.0;
      std::fill(o.begin(), o.end(), 0.0);
      for (int64_t m = 0; m <= i; ++m) {
        const double p = std::exp(logit[m] - mx);
        tot += p;
        const double* vm = vd.data() + m * d;
        for (int c = 0; c < d; ++c) o[c] += p * vm[c];
      }
      const double inv = 1.0 / tot;
      for (int c = 0; c < d; ++c) o[c] *= inv;
      for (int a = 0; a < d; ++a) {
        const double oa = o[a];
        double* out = acc + static_cast<size_t>(a) * d;
        for (int b = 0; b < d; ++b) out[b] += oa * o[b];
      }
    }
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nt; ++t) pool.emplace_back(body, t);
  body(0);
  for (auto& th : pool) th.join();
  const double inv = 1.0 / static_cast<double>(work);
  for (size_t i = 0; i < static_cast<size_t>(d) * d; ++i) {
    double s = 0.0;
    for (int t = 0; t < nt; ++t) s += part[t][i];
    c_out[i] = s * inv;
  }
  return OSCAR_OK;
}

oscar_status oscar_build_rotation(int32_t d, const double* c, const float* calib_x, int64_t n,
                                  double percentile, int32_t variant, double* r64_out,
                                  float* r32_out, float* clip_out, double* eigvals_out) {
  if (d < 2 || d > 256 || (d & (d - 1)) || !calib_x || n < 1 || !r32_out || !clip_out)
    return OSCAR_ERR_INVALID_ARG;
  if (!(percentile >= 0.0 && percentile <= 100.0)) return OSCAR_ERR_INVALID_ARG;
  if (variant != OSCAR_VARIANT_OSCAR && variant != OSCAR_VARIANT_HADAMARD &&
      variant != OSCAR_VARIANT_IDENTITY)
    return OSCAR_ERR_INVALID_ARG;
  if (variant == OSCAR_VARIANT_OSCAR && !c) return OSCAR_ERR_INVALID_ARG;
  const size_t dd = static_cast<size_t>(d) * d;
  int bits = 0;
  while ((1 << bits) < d) ++bits;
  std::vector<double> h(dd);
  const double inv_sqrt = 1.0 / std::sqrt(static_cast<double>(d));
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j)
      h[i * d + j] = (popcount_u32(static_cast<unsigned>(i & j)) & 1) ? -inv_sqrt : inv_sqrt;
  std::vector<double> r(dd, 0.0);
  std::vector<double> evals(d, 0.0);
  if (variant == OSCAR_VARIANT_IDENTITY) {
    for (int i = 0; i < d; ++i) r[i * d + i] = 1.0;
  } else if (variant == OSCAR_VARIANT_HADAMARD) {
    r = h;
  } else {
    std::vector<double> a(c, c + dd), vecs;
    for (int i = 0; i < d; ++i)          // symmetrise
      for (int j = i + 1; j < d; ++j) {
        const double m = 0.5 * (a[i * d + j] + a[j * d + i]);
        a[i * d + j] = a[j * d + i] = m;
      }
    double fro = 0.0;
    for (double x : a) fro += x * x;
    fro = std::sqrt(fro);
    if (!jacobi_eigen(d, a, vecs)) return OSCAR_ERR_NOT_CONVERGED;
    std::vector<int> order(d);
    for (int i = 0; i < d; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](int x, int y) { return a[x * d + x] > a[y * d + y]; });
    std::vector<double> u(dd);
    for (int col = 0; col < d; ++col) {
      const int src = order[col];
      evals[col] = a[src * d + src];
      int arg = 0;
      double best = -1.0;
      for (int i = 0; i < d; ++i) {
        const double m = std::fabs(vecs[i * d + src]);
        if (m > best) { best = m; arg = i; }
      }
      const double sgn = vecs[arg * d + src] < 0 ? -1.0 : 1.0;
      for (int i = 0; i < d; ++i) u[i * d + col] = sgn * vecs[i * d + src];
    }
    for (int i = 0; i + 1 < d; ++i)
      if (evals[i] - evals[i + 1] < 1e-12 * fro) return OSCAR_ERR_NOT_CONVERGED;
    // R = U H P_br: column j of H P_br is column br(j) of H
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) {
        const int hj = bit_reverse(j, bits);
        double s = 0.0;
        for (int k = 0; k < d; ++k) s += u[i * d + k] * h[k * d + hj];
        r[i * d + j] = s;
      }
  }
  for (size_t i = 0; i < dd; ++i) r32_out[i] = static_cast<float>(r[i]);
  if (r64_out) std::memcpy(r64_out, r.data(), dd * sizeof(double));
  if (eigvals_out) std::memcpy(eigvals_out, evals.data(), d * sizeof(double));
  // clip from the fp32 rotation actually stored
  std::vector<double> y(static_cast<size_t>(n) * d);
  std::vector<double> r32d(dd);
  for (size_t i = 0; i < dd; ++i) r32d[i] = r32_out[i];
  for (int64_t t = 0; t < n; ++t) {
    const float* x = calib_x + t * d;
    double* yt = y.data() + t * d;
    for (int j = 0; j < d; ++j) yt[j] = 0.0;
    for (int i = 0; i < d; ++i) {
      const double xi = x[i];
      const double* rr = r32d.data() + static_cast<size_t>(i) * d;
      for (int j = 0; j < d; ++j) yt[j] += xi * rr[j];
    }
    for (int j = 0; j < d; ++j) yt[j] = std::fabs(yt[j]);
  }
  *clip_out = static_cast<float>(percentile_linear(y, percentile));
  return OSCAR_OK;
}

const char* oscar_status_string(oscar_status s) {
  switch (s) {
    case OSCAR_OK: return "ok";
    case OSCAR_ERR_INVALID_ARG: return "invalid argument";
    case OSCAR_ERR_UNSUPPORTED: return "unsupported shape";
    case OSCAR_ERR_WORKSPACE: return "workspace too small";
    case OSCAR_ERR_CUDA: return "CUDA error";
    case OSCAR_ERR_NOT_CONVERGED: return "eigen-solver did not converge or spectrum degenerate";
    default: return "unknown status";
  }
}

int32_t oscar_version(void) { return 100; }

}  // extern "C"
