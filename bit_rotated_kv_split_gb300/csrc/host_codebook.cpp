// Host fit of the Lloyd-Max codebook of one layer's K or V.
//
// myzaker.com OSCAR article, part "OSCAR 把旋转对准 attention" (closing part):
// the code repo combines the attention-aware rotation with a Lloyd-Max
// codebook.  The pages give no procedure; this library fits four levels in
// the codec's normalised domain u = (x~ - zero) / scale (the uniform codec's
// per-row fp16 scale and zero point) by Lloyd's iteration (S. P. Lloyd,
// "Least squares quantization in PCM"; J. Max, "Quantizing for minimum
// distortion", 1960): thresholds at the midpoints of adjacent levels, each
// level the mean of the values in its cell.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "oscar.h"
#include "trace.h"

namespace {

// Nearest fp16 value of x (ties to even), as a double: 11 significant bits
// for normal magnitudes (exponent >= -14), a fixed quantum of 2^-24 below,
// infinity above the largest finite fp16 (65504) after rounding.
double round_fp16(double x) {
  if (!std::isfinite(x) || x == 0.0) return x;
  const double a = std::fabs(x);
  int e = 0;
  std::frexp(a, &e);                       // a = m 2^e, m in [0.5, 1)
  const int q = std::max(e - 11, -24);     // quantum exponent
  const double r = std::nearbyint(std::ldexp(a, -q));   // round half to even
  double y = std::ldexp(r, q);
  if (y > 65504.0) y = INFINITY;
  return std::copysign(y, x);
}

}  // namespace

extern "C" oscar_status oscar_fit_codebook(const double* x, int64_t n, int32_t d, const double* r, double tau,
                                           int32_t iters, float* levels_out) {
  OSCAR_TRACE_CALL();
  if (!x || !r || !levels_out || n < 1 || d != OSCAR_HEAD_DIM || !(tau > 0.0) || !std::isfinite(tau) || iters < 1)
    return OSCAR_ERR_INVALID_ARG;
  std::vector<double> u;
  u.reserve(size_t(n) * d);
  std::vector<double> row(d);
  for (int64_t i = 0; i < n; ++i) {
    const double* xi = x + i * d;
    for (int j = 0; j < d; ++j) {
      double acc = 0.0;
      for (int k = 0; k < d; ++k) acc += xi[k] * r[size_t(k) * d + j];
      row[j] = std::min(std::max(acc, -tau), tau);
    }
    const double mn = *std::min_element(row.begin(), row.end());
    const double mx = *std::max_element(row.begin(), row.end());
    const double s = round_fp16((mx - mn) / 3.0), z = round_fp16(mn);
    if (!(s > 0.0) || !std::isfinite(s)) continue;
    for (int j = 0; j < d; ++j) u.push_back((row[j] - z) / s);
  }
  if (u.empty()) return OSCAR_ERR_INVALID_ARG;
  std::sort(u.begin(), u.end());
  double lv[4] = {0.0, 1.0, 2.0, 3.0};
  for (int it = 0; it < iters; ++it) {
    const double t[3] = {(lv[0] + lv[1]) / 2, (lv[1] + lv[2]) / 2, (lv[2] + lv[3]) / 2};
    // cells of the sorted values: [b_k, b_(k+1)) holds u with exactly k
    // thresholds strictly below it
    size_t b[5];
    b[0] = 0;
    for (int k = 0; k < 3; ++k) b[k + 1] = size_t(std::upper_bound(u.begin(), u.end(), t[k]) - u.begin());
    b[4] = u.size();
    double nl[4];
    for (int k = 0; k < 4; ++k) {
      nl[k] = lv[k];
      if (b[k + 1] > b[k]) {
        double sum = 0.0;
        for (size_t i = b[k]; i < b[k + 1]; ++i) sum += u[i];
        nl[k] = sum / double(b[k + 1] - b[k]);
      }
    }
    const bool same = nl[0] == lv[0] && nl[1] == lv[1] && nl[2] == lv[2] && nl[3] == lv[3];
    for (int k = 0; k < 4; ++k) lv[k] = nl[k];
    if (same) break;
  }
  // levels clamped to [0, 3] (the fp16 scale and zero can put u a rounding
  // step outside it), then rounded to fp16
  // (built locally: levels_out is written only once all four are strictly
  // increasing, so a rejected fit leaves it untouched)
  float h[4];
  for (int k = 0; k < 4; ++k) {
    h[k] = float(round_fp16(std::min(std::max(lv[k], 0.0), 3.0)));
    if (k > 0 && !(h[k] > h[k - 1])) return OSCAR_ERR_INVALID_ARG;
  }
  for (int k = 0; k < 4; ++k) levels_out[k] = h[k];
  return OSCAR_OK;
}
