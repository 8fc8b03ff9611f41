// Latency-table calibration: host code (no kernel).
//
// BASTION ("Bastion: Budget-Aware Speculative Decoding with Tree-structured
// Block Diffusion Drafting"), Methodik §3: the online controller grows the
// tree while S(N) = A_hat(T_N) * L_AR / C(N) does not fall, with C(N) the cost
// of a step that verifies N tree tokens; the pages model the verification
// latency from memory bandwidth and compute, calibrated on the device's
// observed runtimes.  The caller times the verification pass (this library's
// tree attention) at several N; this file fits
//     T_verify(N) = a + b N + c max(0, N - knee)
// by least squares for every integer knee of a range, keeps the knee with the
// smallest squared error, and turns the model into the stage-2 table
// C[n] = t_draft + T_verify(n) and L_AR = T_verify(1).
//
// Each fit is a least-squares problem with at most three columns (1, N and the
// hinge), solved by Householder QR in float64 (no normal equations, whose
// condition number grows as N^2).  A knee at or past every N leaves the hinge
// column zero, and a knee below every N (or at the only N below it) makes the
// hinge a combination of 1 and N; such a fit is the straight line, c = 0.
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/bastion.h"

namespace bst {

// min ||A x - t|| over x for the m x p matrix A given by columns (p <= 3).
// Returns j >= 0 when column j lies (to 1e-9 of its norm) in the span of the
// columns before it -- nothing is solved then -- and -1 on success with
// x[0..p-1] and *sse = residual^2.
static int lsq_qr(int m, int p, std::vector<double> cols[3], const double *t, double *x, double *sse) {
  std::vector<double> y(t, t + m);
  double R[3][3] = {{0.0}};
  for (int j = 0; j < p; ++j) {
    std::vector<double> &v = cols[j];
    double full2 = 0.0, norm2 = 0.0;
    for (int i = 0; i < m; ++i) full2 += v[i] * v[i];   // rows < j hold its projection on the earlier columns
    for (int i = j; i < m; ++i) norm2 += v[i] * v[i];   // its part orthogonal to them
    if (!(norm2 > 1e-18 * full2)) return j;
    const double norm = std::sqrt(norm2);
    const double alpha = v[j] > 0.0 ? -norm : norm;   // R[j][j], sign chosen against cancellation
    // Householder vector u = v[j..] - alpha e_j, applied as H = I - 2 u u^T / (u^T u)
    const double u0 = v[j] - alpha;
    const double utu = norm2 - v[j] * v[j] + u0 * u0;
    v[j] = u0;
    if (utu > 0.0) {
      for (int k = j + 1; k < p; ++k) {
        double dot = 0.0;
        for (int i = j; i < m; ++i) dot += v[i] * cols[k][i];
        const double f = 2.0 * dot / utu;
        for (int i = j; i < m; ++i) cols[k][i] -= f * v[i];
      }
      double dot = 0.0;
      for (int i = j; i < m; ++i) dot += v[i] * y[i];
      const double f = 2.0 * dot / utu;
      for (int i = j; i < m; ++i) y[i] -= f * v[i];
    }
    R[j][j] = alpha;
    for (int k = j + 1; k < p; ++k) R[j][k] = cols[k][j];
  }
  for (int j = p - 1; j >= 0; --j) {
    double s = y[j];
    for (int k = j + 1; k < p; ++k) s -= R[j][k] * x[k];
    x[j] = s / R[j][j];
  }
  double r2 = 0.0;
  for (int i = p; i < m; ++i) r2 += y[i] * y[i];
  *sse = r2;
  return -1;
}

}  // namespace bst

extern "C" {

bastion_status bastion_fit_verify_latency(const int32_t *N, const double *t, int m, int knee_lo, int knee_hi,
                                          double *abc, int32_t *knee_out, double *sse_out) {
  if (!N || !t || !abc || !knee_out || !sse_out) return BASTION_ERR_INVALID_ARG;
  if (m < 3 || m > 65536 || knee_lo > knee_hi || static_cast<int64_t>(knee_hi) - knee_lo > 1000000)
    return BASTION_ERR_INVALID_ARG;
  double energy = 0.0;
  for (int i = 0; i < m; ++i) {
    if (!std::isfinite(t[i])) return BASTION_ERR_INVALID_ARG;
    energy += t[i] * t[i];
  }
  struct Fit {
    double sse, a, b, c;
    int knee;
  };
  std::vector<Fit> fits;
  fits.reserve(static_cast<size_t>(knee_hi - knee_lo + 1));
  std::vector<double> cols[3];
  for (int knee = knee_lo; knee <= knee_hi; ++knee) {
    cols[0].assign(m, 1.0);
    cols[1].resize(m);
    cols[2].resize(m);
    bool hinge = false;
    for (int i = 0; i < m; ++i) {
      cols[1][i] = static_cast<double>(N[i]);
      cols[2][i] = N[i] > knee ? static_cast<double>(N[i] - knee) : 0.0;
      hinge = hinge || cols[2][i] > 0.0;
    }
    double x[3] = {0.0, 0.0, 0.0}, sse = 0.0;
    int dep = bst::lsq_qr(m, hinge ? 3 : 2, cols, t, x, &sse);
    if (dep == 2) {
      // the hinge lies in the span of 1 and N at this knee (every N on one
      // side of it, or a single N at the knee): the fit is the straight line
      cols[0].assign(m, 1.0);
      for (int i = 0; i < m; ++i) cols[1][i] = static_cast<double>(N[i]);
      x[2] = 0.0;
      dep = bst::lsq_qr(m, 2, cols, t, x, &sse);
    }
    if (dep >= 0) return BASTION_ERR_INVALID_ARG;   // fewer than two distinct N
    fits.push_back(Fit{sse, x[0], x[1], hinge ? x[2] : 0.0, knee});
  }
  double best = fits[0].sse;
  for (const Fit &f : fits) best = f.sse < best ? f.sse : best;
  // ties: within 1e-9 of the minimum, relative, or 1e-12 of sum t^2
  const double tol = best * 1e-9 + 1e-12 * energy;
  for (const Fit &f : fits) {
    if (f.sse <= best + tol) {
      abc[0] = f.a;
      abc[1] = f.b;
      abc[2] = f.c;
      *knee_out = f.knee;
      *sse_out = f.sse;
      return BASTION_OK;
    }
  }
  return BASTION_ERR_INVALID_ARG;
}

bastion_status bastion_latency_table(const double *abc, int32_t knee, double t_draft, int n_max, float *C,
                                     float *L_AR) {
  if (!abc || !C || !L_AR || n_max < 1 || n_max > BASTION_MAX_NODES) return BASTION_ERR_INVALID_ARG;
  const double a = abc[0], b = abc[1], c = abc[2];
  for (int n = 0; n <= n_max; ++n) {
    const double hinge = n > knee ? static_cast<double>(n - knee) : 0.0;
    C[n] = static_cast<float>(t_draft + a + b * n + c * hinge);
  }
  *L_AR = static_cast<float>(a + b + c * (1 > knee ? static_cast<double>(1 - knee) : 0.0));
  return BASTION_OK;
}

}  // extern "C"
