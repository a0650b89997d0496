// Host float64 construction of the fixed OSCAR rotation R = U . H_Had . P_br
// and of the per-layer clip threshold.
//
// gist.science, "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit
// KV Cache Quantization", Technical summary 2.1 (C_Q = Q^T Q for keys,
// C_S = V^T S^T S V for values) and 2.2 A (eigendecomposition -> U, Hadamard,
// bit-reversal permutation, R = U H P; thresholds from rotated calibration
// activations).  myzaker.com OSCAR article, part "OSCAR 把旋转对准 attention".
//
// The eigensolver is cyclic Jacobi (Golub & Van Loan, "Matrix Computations",
// section 8.5): symmetric 2x2 rotations annihilate each off-diagonal entry in
// turn until the off-diagonal mass is below 1e-15 of the Frobenius norm.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "oscar.h"
#include "trace.h"

namespace {

bool is_pow2(int d) { return d > 0 && (d & (d - 1)) == 0; }

int bit_reverse(int i, int bits) {
  int r = 0;
  for (int b = 0; b < bits; ++b) {
    r = (r << 1) | (i & 1);
    i >>= 1;
  }
  return r;
}

// Eigen-decomposition of the symmetric a[d][d] (destroyed).  On return the
// columns of v are eigenvectors and w the eigenvalues (unsorted).
bool jacobi_eigen(std::vector<double>& a, int d, std::vector<double>& v, std::vector<double>& w) {
  v.assign(size_t(d) * d, 0.0);
  for (int i = 0; i < d; ++i) v[size_t(i) * d + i] = 1.0;
  double fro = 0.0;
  for (double x : a) fro += x * x;
  fro = std::sqrt(fro);
  const int kMaxSweeps = 100;
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    double off = 0.0;
    for (int p = 0; p < d; ++p)
      for (int q = p + 1; q < d; ++q) off += 2.0 * a[size_t(p) * d + q] * a[size_t(p) * d + q];
    if (std::sqrt(off) <= 1e-15 * fro || fro == 0.0) {
      w.resize(d);
      for (int i = 0; i < d; ++i) w[i] = a[size_t(i) * d + i];
      return true;
    }
    for (int p = 0; p < d - 1; ++p) {
      for (int q = p + 1; q < d; ++q) {
        const double apq = a[size_t(p) * d + q];
        if (apq == 0.0) continue;
        const double app = a[size_t(p) * d + p], aqq = a[size_t(q) * d + q];
        // choose t = tan(theta) of the smaller rotation that zeroes a[p][q]
        const double theta = (aqq - app) / (2.0 * apq);
        const double t = (theta >= 0 ? 1.0 : -1.0) / (std::fabs(theta) + std::sqrt(theta * theta + 1.0));
        const double c = 1.0 / std::sqrt(t * t + 1.0), s = t * c;
        // A <- J^T A J with J the rotation in the (p, q) plane
        for (int k = 0; k < d; ++k) {
          const double akp = a[size_t(k) * d + p], akq = a[size_t(k) * d + q];
          a[size_t(k) * d + p] = c * akp - s * akq;
          a[size_t(k) * d + q] = s * akp + c * akq;
        }
        for (int k = 0; k < d; ++k) {
          const double apk = a[size_t(p) * d + k], aqk = a[size_t(q) * d + k];
          a[size_t(p) * d + k] = c * apk - s * aqk;
          a[size_t(q) * d + k] = s * apk + c * aqk;
        }
        a[size_t(p) * d + q] = a[size_t(q) * d + p] = 0.0;
        for (int k = 0; k < d; ++k) {
          const double vkp = v[size_t(k) * d + p], vkq = v[size_t(k) * d + q];
          v[size_t(k) * d + p] = c * vkp - s * vkq;
          v[size_t(k) * d + q] = s * vkp + c * vkq;
        }
      }
    }
  }
  return false;
}

}  // namespace

namespace {

// R = U . H . P from a symmetric covariance c[d][d] (destroyed).
oscar_status rotation_from_cov(std::vector<double>& c, int d, double* r_out, double* eigvals_out) {
  std::vector<double> v, w;
  if (!jacobi_eigen(c, d, v, w)) return OSCAR_ERR_NO_CONVERGENCE;
  // order by descending eigenvalue; sign: largest-|entry| positive
  std::vector<int> order(d);
  for (int i = 0; i < d; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return w[a] > w[b]; });
  std::vector<double> u(size_t(d) * d);
  for (int col = 0; col < d; ++col) {
    const int src = order[col];
    int arg = 0;
    double best = -1.0;
    for (int i = 0; i < d; ++i) {
      const double m = std::fabs(v[size_t(i) * d + src]);
      if (m > best) {
        best = m;
        arg = i;
      }
    }
    const double sgn = v[size_t(arg) * d + src] < 0 ? -1.0 : 1.0;
    for (int i = 0; i < d; ++i) u[size_t(i) * d + col] = sgn * v[size_t(i) * d + src];
    if (eigvals_out) eigvals_out[col] = w[src];
  }
  // R = U . H . P: (U H)[i][k] = sum_m U[i][m] (-1)^popcount(m & k) / sqrt(d),
  // then column j of R is column br(j) of U H.
  int bits = 0;
  while ((1 << bits) < d) ++bits;
  const double inv = 1.0 / std::sqrt(double(d));
  std::vector<double> uh(size_t(d) * d, 0.0);
  for (int i = 0; i < d; ++i)
    for (int k = 0; k < d; ++k) {
      double s = 0.0;
      for (int m = 0; m < d; ++m) s += (__builtin_popcount(unsigned(m & k)) & 1) ? -u[size_t(i) * d + m] : u[size_t(i) * d + m];
      uh[size_t(i) * d + k] = s * inv;
    }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) r_out[size_t(i) * d + j] = uh[size_t(i) * d + bit_reverse(j, bits)];
  return OSCAR_OK;
}

}  // namespace

extern "C" oscar_status oscar_build_rotation(const double* x, int64_t n, int32_t d, double* r_out,
                                             double* eigvals_out) {
  OSCAR_TRACE_CALL();
  if (!x || !r_out || n < 1 || d < 2 || d > 1024 || !is_pow2(d)) return OSCAR_ERR_INVALID_ARG;
  // C = x^T x / n (uncentred)
  std::vector<double> c(size_t(d) * d, 0.0);
  for (int64_t r = 0; r < n; ++r) {
    const double* row = x + r * d;
    for (int i = 0; i < d; ++i) {
      const double xi = row[i];
      double* ci = c.data() + size_t(i) * d;
      for (int j = i; j < d; ++j) ci[j] += xi * row[j];
    }
  }
  for (int i = 0; i < d; ++i)
    for (int j = i; j < d; ++j) {
      c[size_t(i) * d + j] /= double(n);
      c[size_t(j) * d + i] = c[size_t(i) * d + j];
    }
  return rotation_from_cov(c, d, r_out, eigvals_out);
}

// R from a covariance computed elsewhere (e.g. oscar_covariance on the
// device): the symmetric part (c + c^T) / 2 is decomposed.
extern "C" oscar_status oscar_build_rotation_from_covariance(const double* c, int32_t d, double* r_out,
                                                             double* eigvals_out) {
  OSCAR_TRACE_CALL();
  if (!c || !r_out || d < 2 || d > 1024 || !is_pow2(d)) return OSCAR_ERR_INVALID_ARG;
  std::vector<double> a(size_t(d) * d);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      const double v = 0.5 * (c[size_t(i) * d + j] + c[size_t(j) * d + i]);
      if (!std::isfinite(v)) return OSCAR_ERR_INVALID_ARG;
      a[size_t(i) * d + j] = v;
    }
  return rotation_from_cov(a, d, r_out, eigvals_out);
}

extern "C" oscar_status oscar_score_weighted_rows(const double* q, int64_t n_q, const double* k,
                                                  const double* v, int64_t n_k, int32_t d,
                                                  double scale, double* out) {
  OSCAR_TRACE_CALL();
  if (!q || !k || !v || !out || n_q < 1 || n_k < 1 || d < 1) return OSCAR_ERR_INVALID_ARG;
  std::vector<double> s(static_cast<size_t>(n_k));
  for (int64_t r = 0; r < n_q; ++r) {
    const double* qr = q + r * d;
    double mx = -INFINITY;
    for (int64_t t = 0; t < n_k; ++t) {
      const double* kt = k + t * d;
      double acc = 0.0;
      for (int c = 0; c < d; ++c) acc += qr[c] * kt[c];
      s[t] = acc * scale;
      mx = std::max(mx, s[t]);
    }
    double sum = 0.0;
    for (int64_t t = 0; t < n_k; ++t) {
      s[t] = std::exp(s[t] - mx);
      sum += s[t];
    }
    double* o = out + r * d;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int64_t t = 0; t < n_k; ++t) {
      const double wgt = s[t] / sum;
      const double* vt = v + t * d;
      for (int c = 0; c < d; ++c) o[c] += wgt * vt[c];
    }
  }
  return OSCAR_OK;
}

extern "C" oscar_status oscar_clip_threshold(const double* acts, int64_t rows, int32_t n_heads,
                                             int32_t d, const double* r, double quantile,
                                             double* tau_out) {
  OSCAR_TRACE_CALL();
  if (!acts || !r || !tau_out || rows < 1 || n_heads < 1 || d < 1 || !(quantile > 0.0) ||
      quantile > 1.0)
    return OSCAR_ERR_INVALID_ARG;
  std::vector<double> mags;
  mags.reserve(size_t(rows) * n_heads * d);
  for (int h = 0; h < n_heads; ++h) {
    const double* rh = r + size_t(h) * d * d;
    for (int64_t row = 0; row < rows; ++row) {
      const double* x = acts + (size_t(h) * rows + row) * d;
      for (int j = 0; j < d; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d; ++i) acc += x[i] * rh[size_t(i) * d + j];
        mags.push_back(std::fabs(acc));
      }
    }
  }
  // nearest rank: the ceil(q N)-th smallest magnitude
  int64_t rank = int64_t(std::ceil(quantile * double(mags.size())));
  rank = std::max<int64_t>(1, std::min<int64_t>(rank, int64_t(mags.size())));
  std::nth_element(mags.begin(), mags.begin() + (rank - 1), mags.end());
  *tau_out = mags[size_t(rank - 1)];
  return OSCAR_OK;
}

// OScaR variant ([CSDN] section 四.2): channels split into groups of `block`,
// each rotated by the orthonormal Sylvester Hadamard of that size.
extern "C" oscar_status oscar_build_canalized_rotation(int32_t d, int32_t block, double* r_out) {
  OSCAR_TRACE_CALL();
  if (!r_out || d < 1 || d > 1024 || !is_pow2(d) || block < 1 || block > d || !is_pow2(block))
    return OSCAR_ERR_INVALID_ARG;
  const double inv = 1.0 / std::sqrt(double(block));
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) {
      double v = 0.0;
      if (i / block == j / block) {
        const int a = i % block, b = j % block;
        v = (__builtin_popcount(unsigned(a & b)) & 1) ? -inv : inv;
      }
      r_out[size_t(i) * d + j] = v;
    }
  return OSCAR_OK;
}
