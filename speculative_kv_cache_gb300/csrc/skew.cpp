// Offline skew and partial-column choice (InfiniGen paper-graph summary, section 3.4,
// "Skewed Partial Weights" and "Prefill Stage", Steps 2-3).  Host code, float64 throughout.
//
// Per head h: Q_h = X_s W_Q,h (rotated by RoPE at positions 0..Ns-1 for RoPE models); the
// right singular vectors of Q_h (one-sided Jacobi, Hestenes' method: plane rotations applied
// to the columns of Q_h until every pair is orthogonal, the same rotations accumulated into V)
// sorted by descending singular value form A_h; W~ = W A is rounded once to fp16; the column
// score is the column sum of |W~_Q,h| plus the column sum of |K~_h| over the prompt keys; the
// k best columns (ties to the lower index) are returned in ascending order.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <thread>
#include <vector>

#include "../../include/ig.h"

namespace ig {
ig_status fail(ig_status st, const char* fmt, ...);
}

namespace {

constexpr int kMaxSweeps = 80;

// Host-side fault injection for tests: IG_FAULT=svd_noconverge gives the Jacobi iteration no
// sweeps at all, so it ends unconverged exactly as data that needed more than kMaxSweeps would.
int max_sweeps() {
  const char* f = getenv("IG_FAULT");
  return (f && strstr(f, "svd_noconverge")) ? 0 : kMaxSweeps;
}

double half_to_double(uint16_t h) {
  const int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 1024), e - 25);
  return s ? -v : v;
}

// float64 -> fp16, round to nearest even, in one step (no intermediate float32 rounding).
uint16_t double_to_half(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return sign | 0x7e00;
  double a = fabs(x);
  if (a >= 65520.0) return sign | 0x7c00;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);  // a = f * 2^e, f in [0.5, 1): the leading bit has weight 2^(e-1)
  int E = e - 1;
  if (E >= -14) {
    double r = nearbyint(ldexp(a, 10 - E));  // in [1024, 2048]
    if (r >= 2048.0) {
      r = 1024.0;
      ++E;
    }
    if (E > 15) return sign | 0x7c00;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
  }
  double r = nearbyint(ldexp(a, 24));  // subnormal units of 2^-24 (1024 becomes the smallest normal)
  return sign | (uint16_t)r;
}

struct SkewJob {
  int D, H, d, Ns, Nk, k;
  double theta;
  const double* X;     // [Ns][D]
  const uint16_t* Wq;  // [D][H*d]
  const uint16_t* Wk;
  const uint16_t* Kp;  // [Nk][H][d] or null
  float* A;
  uint16_t* Wq_skew;
  uint16_t* Wk_skew;
  uint16_t* Kp_skew;
  int32_t* cols;
  float* sigma = nullptr;      // [H][d] singular values, descending (optional)
  bool spectrum_only = false;  // stop after the SVD
  std::atomic<int> failed{0};
};

void skew_head(SkewJob& J, int h) {
  const int D = J.D, d = J.d, Ns = J.Ns, Hd = J.H * J.d;
  // W_Q,h as float64 [D][d]
  std::vector<double> Wh((size_t)D * d);
  for (int r = 0; r < D; ++r)
    for (int j = 0; j < d; ++j) Wh[(size_t)r * d + j] = half_to_double(J.Wq[(size_t)r * Hd + h * d + j]);
  // Q_h transposed: column j of Q_h is Qt[j][0..Ns)
  std::vector<double> Qt((size_t)d * Ns);
  std::vector<double> row(d);
  for (int n = 0; n < Ns; ++n) {
    std::fill(row.begin(), row.end(), 0.0);
    const double* x = J.X + (size_t)n * D;
    for (int r = 0; r < D; ++r) {
      const double xv = x[r];
      const double* w = &Wh[(size_t)r * d];
      for (int j = 0; j < d; ++j) row[j] += xv * w[j];
    }
    if (J.theta > 0) {
      const int half = d / 2;
      for (int j = 0; j < half; ++j) {
        const double ang = (double)n * pow(J.theta, -2.0 * j / d);
        const double c = cos(ang), s = sin(ang);
        const double lo = row[j], hi = row[j + half];
        row[j] = lo * c - hi * s;
        row[j + half] = lo * s + hi * c;
      }
    }
    for (int j = 0; j < d; ++j) Qt[(size_t)j * Ns + n] = row[j];
  }
  // one-sided Jacobi
  std::vector<double> V((size_t)d * d, 0.0);  // column j of V at V[j*d ..]
  for (int j = 0; j < d; ++j) V[(size_t)j * d + j] = 1.0;
  std::vector<double> nrm(d);
  for (int j = 0; j < d; ++j) {
    double s = 0;
    for (int n = 0; n < Ns; ++n) s += Qt[(size_t)j * Ns + n] * Qt[(size_t)j * Ns + n];
    nrm[j] = s;
  }
  const double tol = 1e-15;
  bool converged = false;
  const int sweeps = max_sweeps();
  for (int sweep = 0; sweep < sweeps && !converged; ++sweep) {
    converged = true;
    for (int p = 0; p < d - 1; ++p) {
      for (int q = p + 1; q < d; ++q) {
        double* cp = &Qt[(size_t)p * Ns];
        double* cq = &Qt[(size_t)q * Ns];
        double g = 0;
        for (int n = 0; n < Ns; ++n) g += cp[n] * cq[n];
        const double a = nrm[p], b = nrm[q];
        if (fabs(g) <= tol * sqrt(a * b) || g == 0.0) continue;
        converged = false;
        const double zeta = (b - a) / (2.0 * g);
        const double t = (zeta >= 0 ? 1.0 : -1.0) / (fabs(zeta) + sqrt(1.0 + zeta * zeta));
        const double c = 1.0 / sqrt(1.0 + t * t), s = c * t;
        for (int n = 0; n < Ns; ++n) {
          const double xp = cp[n], xq = cq[n];
          cp[n] = c * xp - s * xq;
          cq[n] = s * xp + c * xq;
        }
        double* vp = &V[(size_t)p * d];
        double* vq = &V[(size_t)q * d];
        for (int i = 0; i < d; ++i) {
          const double xp = vp[i], xq = vq[i];
          vp[i] = c * xp - s * xq;
          vq[i] = s * xp + c * xq;
        }
        // recompute the two norms exactly (the update formula drifts)
        double na = 0, nb = 0;
        for (int n = 0; n < Ns; ++n) {
          na += cp[n] * cp[n];
          nb += cq[n] * cq[n];
        }
        nrm[p] = na;
        nrm[q] = nb;
      }
    }
  }
  if (!converged) {
    J.failed = 1;
    return;
  }
  // order by descending singular value, canonical signs
  std::vector<int> ord(d);
  for (int j = 0; j < d; ++j) ord[j] = j;
  std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) { return nrm[x] > nrm[y]; });
  if (J.sigma)
    for (int j = 0; j < d; ++j) J.sigma[(size_t)h * d + j] = (float)sqrt(nrm[ord[j]]);
  if (J.spectrum_only) return;
  std::vector<double> Ah((size_t)d * d);  // row-major A_h[i][j]
  for (int j = 0; j < d; ++j) {
    const double* v = &V[(size_t)ord[j] * d];
    int r = 0;
    for (int i = 1; i < d; ++i)
      if (fabs(v[i]) > fabs(v[r])) r = i;
    const double sg = v[r] < 0 ? -1.0 : 1.0;
    for (int i = 0; i < d; ++i) Ah[(size_t)i * d + j] = sg * v[i];
  }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) J.A[((size_t)h * d + i) * d + j] = (float)Ah[(size_t)i * d + j];
  // W~ = W A (rounded once); column sums of |W~_Q|
  std::vector<double> score(d, 0.0);
  std::vector<double> out(d);
  for (int pass = 0; pass < 2; ++pass) {
    const uint16_t* W = pass == 0 ? J.Wq : J.Wk;
    uint16_t* Wout = pass == 0 ? J.Wq_skew : J.Wk_skew;
    if (pass == 1 && !Wout) break;
    for (int r = 0; r < D; ++r) {
      std::fill(out.begin(), out.end(), 0.0);
      for (int i = 0; i < d; ++i) {
        const double w = pass == 0 ? Wh[(size_t)r * d + i] : half_to_double(W[(size_t)r * Hd + h * d + i]);
        const double* arow = &Ah[(size_t)i * d];
        for (int j = 0; j < d; ++j) out[j] += w * arow[j];
      }
      for (int j = 0; j < d; ++j) {
        const uint16_t hv = double_to_half(out[j]);
        if (Wout) Wout[(size_t)r * Hd + h * d + j] = hv;
        if (pass == 0) score[j] += fabs(half_to_double(hv));
      }
    }
  }
  // skewed prompt keys and their column sums
  if (J.Kp) {
    std::vector<double> kr(d);
    for (int t = 0; t < J.Nk; ++t) {
      const uint16_t* krow = J.Kp + ((size_t)t * J.H + h) * d;
      for (int i = 0; i < d; ++i) kr[i] = half_to_double(krow[i]);
      std::fill(out.begin(), out.end(), 0.0);
      for (int i = 0; i < d; ++i) {
        const double* arow = &Ah[(size_t)i * d];
        for (int j = 0; j < d; ++j) out[j] += kr[i] * arow[j];
      }
      for (int j = 0; j < d; ++j) {
        const uint16_t hv = double_to_half(out[j]);
        if (J.Kp_skew) J.Kp_skew[((size_t)t * J.H + h) * d + j] = hv;
        score[j] += fabs(half_to_double(hv));
      }
    }
  }
  std::vector<int> cidx(d);
  for (int j = 0; j < d; ++j) cidx[j] = j;
  std::stable_sort(cidx.begin(), cidx.end(), [&](int x, int y) {
    if (score[x] != score[y]) return score[x] > score[y];
    return x < y;
  });
  std::vector<int> chosen(cidx.begin(), cidx.begin() + J.k);
  std::sort(chosen.begin(), chosen.end());
  for (int c = 0; c < J.k; ++c) J.cols[(size_t)h * J.k + c] = chosen[c];
}

}  // namespace

extern "C" ig_status ig_skew_weights(int D, int H, int d, float ratio, float rope_theta,
                                     const uint16_t* Xs, int Ns, const uint16_t* Wq,
                                     const uint16_t* Wk, const uint16_t* Kp, int Nk, float* A,
                                     uint16_t* Wq_skew, uint16_t* Wk_skew, uint16_t* Kp_skew,
                                     int32_t* cols, int* k_out, int threads) {
  if (D <= 0 || H <= 0 || d <= 0 || Ns <= 0) return ig::fail(IG_ERR_INVALID, "sizes must be positive");
  if (!(ratio > 0.f && ratio <= 1.f)) return ig::fail(IG_ERR_INVALID, "ratio must be in (0, 1]");
  if (!Xs || !Wq || !A || !cols || !k_out) return ig::fail(IG_ERR_INVALID, "null required pointer");
  if (Wk_skew && !Wk) return ig::fail(IG_ERR_INVALID, "Wk_skew needs Wk");
  if (rope_theta < 0.f || (rope_theta > 0.f && d % 2)) return ig::fail(IG_ERR_INVALID, "RoPE needs even d and theta > 0");
  if (Kp && Nk <= 0) return ig::fail(IG_ERR_INVALID, "Nk must be positive when Kp is given");
  const int k = (int)floor((double)ratio * d + 0.5);
  if (k < 1 || k > d) return ig::fail(IG_ERR_INVALID, "ratio gives k = %d", k);
  std::vector<double> X((size_t)Ns * D);
  for (size_t i = 0; i < X.size(); ++i) X[i] = half_to_double(Xs[i]);
  SkewJob J;
  J.D = D; J.H = H; J.d = d; J.Ns = Ns; J.Nk = Kp ? Nk : 0; J.k = k;
  J.theta = rope_theta;
  J.X = X.data(); J.Wq = Wq; J.Wk = Wk; J.Kp = Kp;
  J.A = A; J.Wq_skew = Wq_skew; J.Wk_skew = Wk_skew; J.Kp_skew = Kp ? Kp_skew : nullptr;
  J.cols = cols;
  int nt = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (nt < 1) nt = 1;
  if (nt > H) nt = H;
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (int h = next++; h < H; h = next++) skew_head(J, h);
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& t : pool) t.join();
  if (J.failed) return ig::fail(IG_ERR_NUMERIC, "Jacobi SVD did not converge");
  *k_out = k;
  return IG_OK;
}

extern "C" ig_status ig_skew_spectrum(int D, int H, int d, float rope_theta, const uint16_t* Xs, int Ns,
                                      const uint16_t* Wq, float* sigma, int threads) {
  if (D <= 0 || H <= 0 || d <= 0 || Ns <= 0) return ig::fail(IG_ERR_INVALID, "sizes must be positive");
  if (!Xs || !Wq || !sigma) return ig::fail(IG_ERR_INVALID, "null required pointer");
  if (rope_theta < 0.f || (rope_theta > 0.f && d % 2)) return ig::fail(IG_ERR_INVALID, "RoPE needs even d and theta > 0");
  std::vector<double> X((size_t)Ns * D);
  for (size_t i = 0; i < X.size(); ++i) X[i] = half_to_double(Xs[i]);
  SkewJob J;
  J.D = D; J.H = H; J.d = d; J.Ns = Ns; J.Nk = 0; J.k = 1;
  J.theta = rope_theta;
  J.X = X.data(); J.Wq = Wq; J.Wk = nullptr; J.Kp = nullptr;
  std::vector<float> A((size_t)H * d * d);
  J.A = A.data(); J.Wq_skew = nullptr; J.Wk_skew = nullptr; J.Kp_skew = nullptr;
  std::vector<int32_t> cols(H);
  J.cols = cols.data();
  J.sigma = sigma;
  J.spectrum_only = true;
  int nt = threads > 0 ? threads : (int)std::thread::hardware_concurrency();
  if (nt < 1) nt = 1;
  if (nt > H) nt = H;
  std::atomic<int> next{0};
  auto worker = [&]() {
    for (int h = next++; h < H; h = next++) skew_head(J, h);
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nt; ++i) pool.emplace_back(worker);
  worker();
  for (auto& t : pool) t.join();
  if (J.failed) return ig::fail(IG_ERR_NUMERIC, "Jacobi SVD did not converge");
  return IG_OK;
}

extern "C" ig_status ig_ratio_from_spectrum(int H, int d, const float* sigma, float energy, int* k_out) {
  if (H <= 0 || d <= 0 || !sigma || !k_out) return ig::fail(IG_ERR_INVALID, "bad argument");
  if (!(energy > 0.f && energy <= 1.f)) return ig::fail(IG_ERR_INVALID, "energy must be in (0, 1]");
  std::vector<double> mean(d, 0.0);
  for (int h = 0; h < H; ++h) {
    double tot = 0;
    for (int j = 0; j < d; ++j) tot += (double)sigma[(size_t)h * d + j] * sigma[(size_t)h * d + j];
    double run = 0;
    for (int j = 0; j < d; ++j) {
      run += (double)sigma[(size_t)h * d + j] * sigma[(size_t)h * d + j];
      mean[j] += tot > 0 ? run / tot : 1.0;
    }
  }
  int k = d;
  for (int j = 0; j < d; ++j)
    if (mean[j] / H >= (double)energy) {
      k = j + 1;
      break;
    }
  *k_out = k;
  return IG_OK;
}
