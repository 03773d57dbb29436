// Coefficient tables on the host: the default table, the Polar Express
// construction (dmuon_polar_express_coefficients), and the fp16 range check
// of the Gram-space backend (dmuon_gram_check_coefficients).  No device code.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "../../include/dmuon.h"
#include "coeffs.cuh"

namespace dmuon {

const float kYouCoefficients[5][3] = {
    {4.0848f, -6.8946f, 2.927f},
    {3.9505f, -6.3029f, 2.6377f},
    {3.7418f, -5.5913f, 2.3037f},
    {2.8769f, -3.1427f, 1.2046f},
    {2.8366f, -3.0525f, 1.2012f},
};

std::vector<std::pair<int, int>> restart_windows(int ns_steps, const std::vector<int>& restarts) {
  std::vector<int> cuts;
  for (int k : restarts)
    if (k > 0 && k < ns_steps) cuts.push_back(k);
  std::sort(cuts.begin(), cuts.end());
  cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());
  std::vector<std::pair<int, int>> w;
  int start = 0;
  auto add = [&](int k0, int k1) {
    // A window of len > kMaxGramWindow steps becomes ceil(len / kMaxGramWindow)
    // windows as even as possible, the longer ones first.
    const int len = k1 - k0, parts = (len + kMaxGramWindow - 1) / kMaxGramWindow;
    int a = k0;
    for (int i = 0; i < parts; ++i) {
      const int l = len / parts + (i < len % parts ? 1 : 0);
      w.push_back({a, a + l});
      a += l;
    }
  };
  for (int k : cuts) { add(start, k); start = k; }
  if (ns_steps > start) add(start, ns_steps);
  return w;
}

namespace {

// Positive real roots of al y^2 + be y + ga = 0, ascending; returns how many.
int positive_roots(double al, double be, double ga, double y[2]) {
  double r[2];
  int n = 0;
  if (al == 0.0) {
    if (be != 0.0) r[n++] = -ga / be;
  } else {
    const double disc = be * be - 4.0 * al * ga;
    if (disc >= 0.0) {
      const double q = -0.5 * (be + std::copysign(std::sqrt(disc), be));
      if (q != 0.0) {
        r[n++] = q / al;
        r[n++] = ga / q;
      } else {
        r[n++] = 0.0;  // be = 0 and disc = 0: a double root at 0
      }
    }
  }
  int m = 0;
  for (int i = 0; i < n; ++i)
    if (r[i] > 0.0 && std::isfinite(r[i])) y[m++] = r[i];
  if (m == 2 && y[0] > y[1]) std::swap(y[0], y[1]);
  return m;
}

// p(x) = a x + b x^3 + c x^5.
double quintic(const double* q, double x) {
  const double x2 = x * x;
  return x * (q[0] + x2 * (q[1] + q[2] * x2));
}

// max |p(x)| over x in [0, hi]: p(0) = 0, the end point, and the points
// where p'(x) = a + 3 b x^2 + 5 c x^4 vanishes.
double max_abs_quintic(const double* q, double hi) {
  double best = std::fabs(quintic(q, hi));
  double y[2];
  const int n = positive_roots(5.0 * q[2], 3.0 * q[1], q[0], y);
  for (int i = 0; i < n; ++i) {
    const double x = std::sqrt(y[i]);
    if (x < hi) best = std::max(best, std::fabs(quintic(q, x)));
  }
  return best;
}

// max |Z(l)| over l in [0, L], Z(l) = a + b l + c l^2 (the factor of one step
// on a Gram eigenvalue l).
double max_abs_factor(const double* q, double L) {
  auto z = [&](double l) { return q[0] + l * (q[1] + q[2] * l); };
  double best = std::max(std::fabs(z(0.0)), std::fabs(z(L)));
  if (q[2] != 0.0) {
    const double v = -q[1] / (2.0 * q[2]);
    if (v > 0.0 && v < L) best = std::max(best, std::fabs(z(v)));
  }
  return best;
}

// max |l Z(l)| over l in [0, L] (an eigenvalue of R Z).
double max_abs_gram_factor(const double* q, double L) {
  auto f = [&](double l) { return l * (q[0] + l * (q[1] + q[2] * l)); };
  double best = std::fabs(f(L));
  double y[2];
  const int n = positive_roots(3.0 * q[2], 2.0 * q[1], q[0], y);
  for (int i = 0; i < n; ++i)
    if (y[i] < L) best = std::max(best, std::fabs(f(y[i])));
  return best;
}

// Gaussian elimination with partial pivoting on a 4 x 4 system (augmented).
bool solve4(double M[4][5], double out[4]) {
  for (int c = 0; c < 4; ++c) {
    int p = c;
    for (int r = c + 1; r < 4; ++r)
      if (std::fabs(M[r][c]) > std::fabs(M[p][c])) p = r;
    if (M[p][c] == 0.0) return false;
    if (p != c)
      for (int k = 0; k < 5; ++k) std::swap(M[p][k], M[c][k]);
    for (int r = c + 1; r < 4; ++r) {
      const double f = M[r][c] / M[c][c];
      for (int k = c; k < 5; ++k) M[r][k] -= f * M[c][k];
    }
  }
  for (int r = 3; r >= 0; --r) {
    double s = M[r][4];
    for (int k = r + 1; k < 4; ++k) s -= M[r][k] * out[k];
    out[r] = s / M[r][r];
  }
  return true;
}

// The odd quintic q minimising max |1 - p(x)| over [lo, hi], and that error
// E (> 0, with 1 - p(lo) = +E): Remez exchange on four reference points,
// which for this three-term family alternate at lo, the two interior
// extrema of 1 - p (roots of p', a quadratic in x^2) and hi.
bool minimax_quintic(double lo, double hi, double q[3], double* err) {
  const double pi = 3.14159265358979323846;
  double x[4];
  for (int k = 0; k < 4; ++k) x[k] = 0.5 * (lo + hi) - 0.5 * (hi - lo) * std::cos(pi * k / 3.0);
  x[0] = lo;
  x[3] = hi;
  double E = 0.0, prev = 0.0;
  for (int it = 0; it < 200; ++it) {
    double M[4][5];
    for (int i = 0; i < 4; ++i) {
      const double xi = x[i], x3 = xi * xi * xi;
      M[i][0] = xi;
      M[i][1] = x3;
      M[i][2] = x3 * xi * xi;
      M[i][3] = (i & 1) ? -1.0 : 1.0;
      M[i][4] = 1.0;
    }
    double s[4];
    if (!solve4(M, s)) return false;
    q[0] = s[0];
    q[1] = s[1];
    q[2] = s[2];
    E = s[3];
    double y[2];
    if (positive_roots(5.0 * q[2], 3.0 * q[1], q[0], y) != 2) return false;
    const double x1 = std::sqrt(y[0]), x2 = std::sqrt(y[1]);
    if (!(lo < x1 && x1 < x2 && x2 < hi)) return false;
    x[1] = x1;
    x[2] = x2;
    if (it > 0 && std::fabs(E - prev) <= 1e-15 * std::fabs(E)) break;
    prev = E;
  }
  if (!(E > 0.0) || !std::isfinite(E)) return false;
  *err = E;
  return true;
}

void set_why(char* why, size_t len, const char* fmt, int k, double v) {
  if (why && len) std::snprintf(why, len, fmt, k, v);
}

}  // namespace

// Every stored buffer is fp16 (largest finite value 65504).  Following the
// largest singular value the iterate can reach -- 1 for the normalised
// input, then u' = max over [0, u] of |p_k| after step k -- bounds every
// buffer over all inputs: with Gram eigenvalues in [0, u^2], the step's
// factor Z = a I + b R + c R^2 has |Z| <= max |Z(l)|, kappa R and
// kappa R Z have at most kappa u^2 and kappa max |l Z(l)| (kappa <= 1024),
// and a window's factor Q at most the product of its steps' max |Z|.
// Limits: 32768 (half the fp16 maximum, for rounding) for kappa R, kappa R Z
// and Z; 8192 for a window's Q.  The iterate itself, stored as beta X with
// beta <= 1024, stays below 1024 u <= 32768 wherever kappa u^2 does.  Below:
// Z is stored without a scale, so each row needs a >= 1/64 (kMinLinear): the
// identity part a I keeps Z's significant entries in fp16's normal range,
// where without it the entries of c A A (about s^4 for the singular values s
// of a normalised m x n input, s^2 ~ 1/m) fall into the subnormals for m of
// a few hundred.  Every Newton-Schulz step has a = p'(0) > 0 (the factor by
// which it lifts small singular values); a < 1/64 is no such step.
constexpr double kMinLinear = 1.0 / 64.0;
bool direct_table_fits(int ns_steps, const float* coeffs, char* why, size_t why_len) {
  constexpr double kKappa = 1024.0, kLimit = 32768.0;
  double u = 1.0;
  for (int k = 0; k < ns_steps; ++k) {
    const float* r = coefficient_row(coeffs, k);
    const double q[3] = {r[0], r[1], r[2]};
    if (!(q[0] >= kMinLinear)) {
      set_why(why, why_len, "step %d: a = %.4g, below 1/64: Z = a I + b A + c A A is stored in fp16 without a "
              "scale and needs its identity part (every Newton-Schulz step has a = p'(0) > 0)", k, q[0]);
      return false;
    }
    if (kKappa * u * u > kLimit) {
      set_why(why, why_len, "step %d: singular values may reach %.4g, past the fp16 range of kappa X X^T", k, u);
      return false;
    }
    const double zmax = max_abs_factor(q, u * u);
    if (zmax > kLimit) {
      set_why(why, why_len, "step %d: the step factor Z may reach %.4g, past fp16", k, zmax);
      return false;
    }
    u = max_abs_quintic(q, u);
  }
  return true;
}

bool gram_table_fits(int ns_steps, const float* coeffs, const std::vector<int>& restarts, char* why,
                     size_t why_len) {
  constexpr double kKappa = 1024.0, kLimit = 32768.0, kWindowGain = 8192.0;
  double u = 1.0;
  for (const auto& w : restart_windows(ns_steps, restarts)) {
    double gain = 1.0;
    for (int k = w.first; k < w.second; ++k) {
      const float* r = coefficient_row(coeffs, k);
      const double q[3] = {r[0], r[1], r[2]};
      if (!(q[0] >= kMinLinear)) {
        set_why(why, why_len, "step %d: a = %.4g, below 1/64: the fp16 step factor Z = a I + b R + c R R needs "
                "its identity part (every Newton-Schulz step has a = p'(0) > 0)", k, q[0]);
        return false;
      }
      const double L = u * u;
      if (kKappa * L > kLimit) {
        set_why(why, why_len, "step %d: singular values may reach %.4g, past the fp16 range of kappa R", k,
                u);
        return false;
      }
      const double zmax = max_abs_factor(q, L), gmax = max_abs_gram_factor(q, L);
      if (zmax > kLimit) {
        set_why(why, why_len, "step %d: the step factor Z may reach %.4g, past fp16", k, zmax);
        return false;
      }
      if (kKappa * gmax > kLimit) {
        set_why(why, why_len, "step %d: kappa R Z may reach 1024 x %.4g, past fp16", k, gmax);
        return false;
      }
      gain *= std::max(1.0, zmax);
      u = max_abs_quintic(q, u);
    }
    if (gain > kWindowGain) {
      set_why(why, why_len, "window ending at step %d: its factor's gain %.4g exceeds 8192; add restarts",
              w.second, gain);
      return false;
    }
  }
  if (kKappa * u * u > kLimit) {
    set_why(why, why_len, "after %d steps: singular values may reach %.4g, past the fp16 range of kappa R",
            ns_steps, u);
    return false;
  }
  return true;
}

}  // namespace dmuon

using namespace dmuon;

extern "C" {

int dmuon_polar_express_coefficients(int steps, double lower, double upper, double safety, float* out) {
  if (!out || steps < 1 || steps > DMUON_MAX_NS_STEPS || !(lower > 0.0) || !(upper > lower) || !(safety > 0.0) ||
      !std::isfinite(upper) || !std::isfinite(safety))
    return DMUON_ERR_ARG;
  // Once the interval lies within 1e-7 of the point 1 the exchange has
  // nothing left to resolve in double precision: such rows take the
  // construction's limit, the quintic with p(1) = 1, p'(1) = p''(1) = 0.
  constexpr double kTiny = 1e-7;
  double lo = lower, hi = upper;
  const double s = safety, s3 = s * s * s, s5 = s3 * s * s;
  for (int k = 0; k < steps; ++k) {
    double q[3], E;
    if (lo >= 1.0 - kTiny && hi <= 1.0 + kTiny) {
      q[0] = 15.0 / 8.0;
      q[1] = -10.0 / 8.0;
      q[2] = 3.0 / 8.0;
      E = std::max(std::fabs(1.0 - quintic(q, lo)), std::fabs(1.0 - quintic(q, hi)));
    } else if (!minimax_quintic(lo, hi, q, &E)) {
      return DMUON_ERR_ARG;
    }
    out[3 * k + 0] = (float)(q[0] / s);
    out[3 * k + 1] = (float)(q[1] / s3);
    out[3 * k + 2] = (float)(q[2] / s5);
    lo = 1.0 - E;
    hi = 1.0 + E;
    if (!(lo > 0.0)) return DMUON_ERR_ARG;  // the next interval would reach 0
  }
  return DMUON_OK;
}

int dmuon_gram_check_coefficients(int ns_steps, const float* coeffs, const int* restarts, int n_restarts,
                                  char* why, size_t why_len) {
  if (why && why_len) why[0] = 0;
  if (ns_steps < 0 || ns_steps > DMUON_MAX_NS_STEPS || n_restarts < 0 || n_restarts > DMUON_MAX_NS_STEPS ||
      (n_restarts > 0 && !restarts))
    return DMUON_ERR_ARG;
  if (coeffs)
    for (int i = 0; i < 3 * ns_steps; ++i)
      if (!std::isfinite(coeffs[i])) return DMUON_ERR_ARG;
  std::vector<int> r;
  if (restarts) r.assign(restarts, restarts + n_restarts);
  else r.push_back(2);
  std::vector<float> pe;
  if (!coeffs && ns_steps > 0) {  // the backend's default: the Polar Express table
    pe.resize(3 * (size_t)ns_steps);
    if (dmuon_polar_express_coefficients(ns_steps, 1e-3, 1.0, 1.05, pe.data()) != DMUON_OK) return DMUON_ERR_ARG;
    coeffs = pe.data();
  }
  return gram_table_fits(ns_steps, coeffs, r, why, why_len) ? DMUON_OK : DMUON_ERR_ARG;
}

}  // extern "C"
