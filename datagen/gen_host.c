/*
 * gen_host.c - host side of the seeded synthetic-mixture generator.
 *
 * Builds the planted mixture tables for each workload (weights, centres,
 * spreads), the initial parameters theta_0 that both the CUDA path and the
 * fp64 oracle start from, and any range of points (OpenMP over points).
 * Every point is drawn by gen_point() in mixture_gen.h, the same code the
 * device generator runs, so a point's bits do not depend on where it was made.
 *
 * Compile with -ffp-contract=off (no fused multiply-add): bit agreement with
 * the device build depends on it.
 */
#include "mixture_gen.h"

#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- helpers */

/* Standard normal number i of purpose `purpose` in the parameter stream. */
static double param_normal(uint64_t seed, uint32_t purpose, uint64_t i) {
  double z0, z1;
  gen_normal_pair(seed, GEN_STREAM_PARAMS, ((uint64_t)purpose << 40) | (i >> 1), 0, &z0, &z1);
  return (i & 1) ? z1 : z0;
}

static double param_uniform(uint64_t seed, uint32_t purpose, uint64_t i) {
  double u0, u1;
  gen_uniform_pair(seed, GEN_STREAM_PARAMS, ((uint64_t)purpose << 40) | (i >> 1), 1, &u0, &u1);
  return (i & 1) ? u1 : u0;
}

/* exp(x) for moderate x: x = k ln2 + r with |r| <= ln2/2, Taylor series of
 * exp(r) to r^20, then scaling by 2^k through the exponent field. */
static double own_exp(double x) {
  const double LN2 = 0.6931471805599453;
  double kd = x / LN2;
  long k = (long)(kd < 0 ? kd - 0.5 : kd + 0.5);
  double r = x - (double)k * LN2;
  double term = 1.0, sum = 1.0;
  for (int i = 1; i <= 20; ++i) { term = term * r / (double)i; sum = sum + term; }
  if (k > 1000) k = 1000;
  if (k < -1000) k = -1000;
  return sum * gen_bitsd((uint64_t)(1023 + k) << 52);
}

/* Gamma(alpha, 1) draw number i (Marsaglia and Tsang, ACM TOMS 26(3), 2000;
 * alpha < 1 through Gamma(alpha + 1) * U^(1/alpha)). */
static double gamma_draw(uint64_t seed, uint32_t purpose, uint64_t i, double alpha) {
  double boost = 1.0;
  if (alpha < 1.0) {
    double u = param_uniform(seed, purpose + 1, i);
    if (u <= 0.0) u = 1e-300;
    boost = own_exp(gen_ln(u) / alpha);
    alpha = alpha + 1.0;
  }
  double d = alpha - 1.0 / 3.0;
  double c = 1.0 / sqrt(9.0 * d);
  for (uint64_t t = 0;; ++t) {
    uint64_t j = (i << 16) | (t & 0xFFFF);
    double z = param_normal(seed, purpose + 2, j);
    double v = 1.0 + c * z;
    if (v <= 0.0) continue;
    v = v * v * v;
    double u = param_uniform(seed, purpose + 3, j);
    if (u <= 0.0) continue;
    if (gen_ln(u) < 0.5 * z * z + d - d * v + d * gen_ln(v)) return d * v * boost;
  }
}

static void weights_to_cdf(int K, const double* w, double* cdf) {
  double acc = 0.0;
  for (int k = 0; k < K; ++k) { acc = acc + w[k]; cdf[k] = acc; }
}

/* Dirichlet(alpha) weights (symmetric); alpha <= 0 means uniform 1/K. */
static void dirichlet(uint64_t seed, int K, double alpha, double* w) {
  double s = 0.0;
  for (int k = 0; k < K; ++k) {
    w[k] = alpha > 0 ? gamma_draw(seed, 100, (uint64_t)k, alpha) : 1.0;
    s = s + w[k];
  }
  for (int k = 0; k < K; ++k) w[k] = w[k] / s;
}

/* ---------------------------------------------------- planted mixtures */

/* Diagonal mixture.  Means N(0, mean_sd^2) per dimension.  Spread:
 *   sd_mode 0: per-dimension variance U[lo, hi]  (sd = sqrt(var))
 *   sd_mode 1: per-component standard deviation U[lo, hi], same in every dimension.
 * Weights Dirichlet(alpha) (alpha <= 0: uniform).  Outputs w[K], cdf[K],
 * mu[K*D], sd[K*D]. */
int gen_planted_diag(uint64_t seed, int D, int K, double mean_sd, int sd_mode, double lo,
                     double hi, double alpha, double* w, double* cdf, double* mu, double* sd) {
  if (D <= 0 || K <= 0 || (D & 1)) return 1;
  for (int k = 0; k < K; ++k)
    for (int d = 0; d < D; ++d)
      mu[(size_t)k * D + d] = mean_sd * param_normal(seed, 10, (uint64_t)k * D + d);
  for (int k = 0; k < K; ++k) {
    double comp = lo + (hi - lo) * param_uniform(seed, 20, (uint64_t)k);
    for (int d = 0; d < D; ++d) {
      if (sd_mode == 0) {
        double var = lo + (hi - lo) * param_uniform(seed, 21, (uint64_t)k * D + d);
        sd[(size_t)k * D + d] = sqrt(var);
      } else {
        sd[(size_t)k * D + d] = comp;
      }
    }
  }
  dirichlet(seed, K, alpha, w);
  weights_to_cdf(K, w, cdf);
  return 0;
}

/* Full-covariance mixture: mu ~ N(0, mean_sd^2 I), Sigma = A A^T / D + ridge I,
 * A_ij ~ N(0,1); outputs sigma[K*D*D], chol[K*D*D] (lower, row-major). */
int gen_planted_full(uint64_t seed, int D, int K, double mean_sd, double ridge, double alpha,
                     double* w, double* cdf, double* mu, double* sigma, double* chol) {
  if (D <= 0 || K <= 0 || (D & 1)) return 1;
  double* A = (double*)malloc(sizeof(double) * (size_t)D * D);
  if (!A) return 2;
  for (int k = 0; k < K; ++k) {
    for (int d = 0; d < D; ++d) mu[(size_t)k * D + d] = mean_sd * param_normal(seed, 30, (uint64_t)k * D + d);
    for (int i = 0; i < D * D; ++i) A[i] = param_normal(seed, 31, (uint64_t)k * D * D + i);
    double* S = sigma + (size_t)k * D * D;
    for (int i = 0; i < D; ++i)
      for (int j = 0; j < D; ++j) {
        double acc = 0.0;
        for (int t = 0; t < D; ++t) acc = acc + A[i * D + t] * A[j * D + t];
        S[i * D + j] = acc / (double)D + (i == j ? ridge : 0.0);
      }
    /* Cholesky factor used only to draw correlated noise. */
    double* L = chol + (size_t)k * D * D;
    for (int i = 0; i < D * D; ++i) L[i] = 0.0;
    for (int j = 0; j < D; ++j) {
      double s = S[j * D + j];
      for (int t = 0; t < j; ++t) s = s - L[j * D + t] * L[j * D + t];
      if (s <= 0.0) { free(A); return 3; }
      double ljj = sqrt(s);
      L[j * D + j] = ljj;
      for (int i = j + 1; i < D; ++i) {
        double v = S[i * D + j];
        for (int t = 0; t < j; ++t) v = v - L[i * D + t] * L[j * D + t];
        L[i * D + j] = v / ljj;
      }
    }
  }
  free(A);
  dirichlet(seed, K, alpha, w);
  weights_to_cdf(K, w, cdf);
  return 0;
}

/* Unit-norm centres g/|g|, g ~ N(0, I), uniform weights. */
int gen_planted_sphere(uint64_t seed, int D, int K, double* w, double* cdf, double* mu) {
  if (D <= 0 || K <= 0 || (D & 1)) return 1;
  for (int k = 0; k < K; ++k) {
    double ss = 0.0;
    for (int d = 0; d < D; ++d) {
      double g = param_normal(seed, 40, (uint64_t)k * D + d);
      mu[(size_t)k * D + d] = g;
      ss = ss + g * g;
    }
    double inv = 1.0 / sqrt(ss);
    for (int d = 0; d < D; ++d) mu[(size_t)k * D + d] = mu[(size_t)k * D + d] * inv;
  }
  dirichlet(seed, K, 0.0, w);
  weights_to_cdf(K, w, cdf);
  return 0;
}

/* ---------------------------------------------------------------- points */

/* Points [start, start+count) of mixture m, written row-major into out
 * (dtype GEN_*).  OpenMP over points. */
int gen_points(const gen_mixture* m, uint64_t start, uint64_t count, int dtype, void* out) {
  if (m->D <= 0 || (m->D & 1) || m->D > 1024) return 1;
  size_t esz = dtype == GEN_F32 ? 4 : 2;
  long long n = (long long)count;
#pragma omp parallel
  {
    double scratch[1024];
#pragma omp for schedule(static)
    for (long long i = 0; i < n; ++i)
      gen_point(m, start + (uint64_t)i, dtype, (char*)out + (size_t)i * m->D * esz, scratch);
  }
  return 0;
}

/* Points with the given indices (any order), row i of out = point idx[i]. */
int gen_points_at(const gen_mixture* m, const int64_t* idx, int64_t count, int dtype, void* out) {
  if (m->D <= 0 || (m->D & 1) || m->D > 1024) return 1;
  size_t esz = dtype == GEN_F32 ? 4 : 2;
  long long n = (long long)count;
#pragma omp parallel
  {
    double scratch[1024];
#pragma omp for schedule(static)
    for (long long i = 0; i < n; ++i)
      gen_point(m, (uint64_t)idx[i], dtype, (char*)out + (size_t)i * m->D * esz, scratch);
  }
  return 0;
}

/* ------------------------------------------------------- initial params */

/* K distinct point indices in [0, N) (uniform, first-come rejection of
 * repeats, in draw order). */
int gen_init_indices(uint64_t seed, int64_t N, int K, int64_t* idx) {
  if (K <= 0 || N < K) return 1;
  int got = 0;
  for (uint64_t t = 0; got < K; ++t) {
    double u0, u1;
    gen_uniform_pair(seed, GEN_STREAM_INIT, t, 0, &u0, &u1);
    double us[2] = {u0, u1};
    for (int h = 0; h < 2 && got < K; ++h) {
      int64_t c = (int64_t)(us[h] * (double)N);
      if (c >= N) c = N - 1;
      int dup = 0;
      for (int i = 0; i < got; ++i) if (idx[i] == c) { dup = 1; break; }
      if (!dup) idx[got++] = c;
    }
  }
  return 0;
}

/* Decode one stored coordinate to double. */
static double stored_to_double(const void* row, int dtype, int d) {
  if (dtype == GEN_F32) return (double)((const float*)row)[d];
  uint16_t h = ((const uint16_t*)row)[d];
  if (dtype == GEN_BF16) {
    uint32_t f = (uint32_t)h << 16;
    float v;
    memcpy(&v, &f, 4);
    return (double)v;
  }
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = (double)m * (1.0 / 16777216.0);               /* m * 2^-24 */
  else if (e == 31) v = m ? (0.0 / 0.0) : (1.0 / 0.0);
  else v = (1.0 + (double)m / 1024.0) * gen_bitsd((uint64_t)(1023 + e - 15) << 52);
  return s ? -v : v;
}

/* Per-dimension mean and variance (biased, two-pass, index order) of the
 * stored rows X[0..n) - the "global variance" of the initialisation.
 * If cov != NULL the full D x D covariance is written too. */
int gen_global_moments(const void* X, int dtype, int64_t n, int D, double* mean, double* var,
                       double* cov) {
  if (n <= 0 || D <= 0) return 1;
  size_t esz = dtype == GEN_F32 ? 4 : 2;
  for (int d = 0; d < D; ++d) mean[d] = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const char* row = (const char*)X + (size_t)i * D * esz;
    for (int d = 0; d < D; ++d) mean[d] = mean[d] + stored_to_double(row, dtype, d);
  }
  for (int d = 0; d < D; ++d) mean[d] = mean[d] / (double)n;
  for (int d = 0; d < D; ++d) var[d] = 0.0;
  if (cov) for (int i = 0; i < D * D; ++i) cov[i] = 0.0;
  double* c = (double*)malloc(sizeof(double) * (size_t)D);
  if (!c) return 2;
  for (int64_t i = 0; i < n; ++i) {
    const char* row = (const char*)X + (size_t)i * D * esz;
    for (int d = 0; d < D; ++d) c[d] = stored_to_double(row, dtype, d) - mean[d];
    for (int d = 0; d < D; ++d) var[d] = var[d] + c[d] * c[d];
    if (cov)
      for (int a = 0; a < D; ++a)
        for (int b = 0; b < D; ++b) cov[a * D + b] = cov[a * D + b] + c[a] * c[b];
  }
  free(c);
  for (int d = 0; d < D; ++d) var[d] = var[d] / (double)n;
  if (cov) for (int i = 0; i < D * D; ++i) cov[i] = cov[i] / (double)n;
  return 0;
}

/* Stored rows widened to double (for initial means). */
int gen_rows_to_double(const void* X, int dtype, int64_t n, int D, double* out) {
  size_t esz = dtype == GEN_F32 ? 4 : 2;
  for (int64_t i = 0; i < n; ++i)
    for (int d = 0; d < D; ++d)
      out[(size_t)i * D + d] = stored_to_double((const char*)X + (size_t)i * D * esz, dtype, d);
  return 0;
}

/* Philox block exposed for known-answer tests. */
void gen_philox_block(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  for (int i = 0; i < 4; ++i) out[i] = ctr[i];
  gen_philox4x32_10(out, key[0], key[1]);
}

/* Bulk normals / ln / rounding for the generator's own tests. */
void gen_normals(uint64_t seed, uint32_t stream, uint64_t idx, uint32_t npairs, double* out) {
  for (uint32_t j = 0; j < npairs; ++j) gen_normal_pair(seed, stream, idx, j, &out[2 * j], &out[2 * j + 1]);
}
double gen_ln_host(double s) { return gen_ln(s); }
uint16_t gen_to_f16_host(double x) { return gen_to_f16(x); }
uint16_t gen_to_bf16_host(double x) { return gen_to_bf16(x); }
