/*
 * gmm_oracle.c - plain fp64 CPU oracle for one EM iteration of a Gaussian
 * mixture model, and for top-m soft assignment.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code with
 * the CUDA path (its own stored-value decoding, its own Cholesky, its own
 * reductions) and is never tuned: it writes the textbook definitions out
 * step by step in double precision, with OpenMP over points.
 *
 * What it follows (page titles as given in the source pages):
 *  - "low-precision GMM operator" design notes (hotelren.com news 5857197):
 *      sec. 1.1  posterior p(z=k|x) = pi_k N(x|mu_k,S_k) / sum_j pi_j N(x|mu_j,S_j)
 *      sec. 1.2  N(x|mu,S) = (2 pi)^(-D/2) |S|^(-1/2) exp(-(x-mu)^T S^-1 (x-mu)/2),
 *                evaluated by the Cholesky route: S = L L^T, z = L^-1 (x-mu),
 *                d^2 = z^T z, log|S| = 2 sum log L_ii
 *      sec. 4.2  log-space posterior with the max subtracted before exp
 *      sec. 3.3 / 4.1  positive-definiteness check, ridge S + eps I with
 *                eps = 1e-3 tr(S)/D
 *  - "Flash-GMM" summary (ai-feeds.com paper 2606.10896), Method:
 *      s0_k = sum_n g_nk, s1_k = sum_n g_nk x_n, s2_k = sum_n g_nk x_n x_n^T,
 *      then the parameters are updated from these statistics (the page prints
 *      no update formula; the maximum-likelihood update is used:
 *      pi' = s0/N, mu' = s1/s0, S' = sum g (x-mu')(x-mu')^T / s0, the
 *      second moment taken about mu' in a second pass so no cancellation
 *      enters the reference).
 *
 * Readings where the pages are silent (each also used by the CUDA path):
 *  - ridge: opts[0] * tr(S)/D is always added (default 0); if the Cholesky
 *    factorisation (diagonal: a variance) is still not positive, 1e-3*tr(S)/D
 *    is added on top and it is retried once (flag bit 1); if that fails the
 *    component is not positive definite (flag bit 2, status 3).
 *  - variance floor: diagonal/isotropic variances, and the diagonal of a
 *    full covariance, are raised to opts[1] after the update (flag bit 4).
 *  - empty component: if s0_k < opts[2], pi'_k = s0_k/N and mu_k, S_k are
 *    kept from the input (flag bit 8).
 *  - isotropic variance: the mean over dimensions of the diagonal update.
 *  - a weight pi_k = 0 gives log pi_k = -inf: the component takes no
 *    responsibility; the max for the log-sum-exp is taken over finite terms.
 *  - log-likelihood returned: sum_n log sum_k pi_k N(x_n|...) at the INPUT
 *    parameters.
 *  - top-m: components sorted by descending log joint density, ties to the
 *    lower index; the reported responsibility is the full-K posterior.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { O_F32 = 0, O_F16 = 1, O_BF16 = 2 };
enum { O_FULL = 0, O_DIAG = 1, O_ISO = 2 };
enum { O_OK = 0, O_INVALID = 1, O_NOT_PD = 3, O_NONFINITE = 4, O_NOMEM = 8 };
enum { FLAG_RIDGE = 1, FLAG_NOT_PD = 2, FLAG_FLOOR = 4, FLAG_EMPTY = 8 };

static const double LOG_2PI = 1.8378770664093454835606594728112;

/* ------------------------------------------------------ stored values */

static double half_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x400), e - 25);
  return s ? -v : v;
}

static double bf16_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 7) & 0xff, m = h & 0x7f;
  double v;
  if (e == 0) v = ldexp((double)m, -133);
  else if (e == 255) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x80), e - 134);
  return s ? -v : v;
}

static void load_x(const void* X, int dtype, int64_t n, int D, double* x) {
  if (dtype == O_F32) {
    const float* r = (const float*)X + (size_t)n * D;
    for (int d = 0; d < D; ++d) x[d] = (double)r[d];
  } else if (dtype == O_F16) {
    const uint16_t* r = (const uint16_t*)X + (size_t)n * D;
    for (int d = 0; d < D; ++d) x[d] = half_to_double(r[d]);
  } else {
    const uint16_t* r = (const uint16_t*)X + (size_t)n * D;
    for (int d = 0; d < D; ++d) x[d] = bf16_to_double(r[d]);
  }
}

/* ------------------------------------------------ component set-up */

/* Per-component quantities the density needs. */
typedef struct {
  int D, K, cov;
  const double* mu;    /* K*D */
  double* logpi;       /* K */
  double* logdet;      /* K   log|S_k| */
  double* L;           /* full: K*D*D lower Cholesky factors */
  double* var;         /* diag: K*D variances; iso: K */
} comps_t;

/* Cholesky S = L L^T (lower, row-major).  Returns 0, or 1 if a pivot is not
 * positive. */
static int cholesky(int D, const double* S, double add, double* L) {
  for (int i = 0; i < D * D; ++i) L[i] = 0.0;
  for (int j = 0; j < D; ++j) {
    double s = S[j * D + j] + add;
    for (int t = 0; t < j; ++t) s -= L[j * D + t] * L[j * D + t];
    if (!(s > 0.0) || !isfinite(s)) return 1;
    double ljj = sqrt(s);
    L[j * D + j] = ljj;
    for (int i = j + 1; i < D; ++i) {
      double v = S[i * D + j];
      for (int t = 0; t < j; ++t) v -= L[i * D + t] * L[j * D + t];
      L[i * D + j] = v / ljj;
    }
  }
  return 0;
}

static void comps_free(comps_t* c) {
  free(c->logpi); free(c->logdet); free(c->L); free(c->var);
  memset(c, 0, sizeof(*c));
}

/* Builds the per-component factors.  flags[k] gets FLAG_RIDGE / FLAG_NOT_PD.
 * Returns O_OK, O_NOT_PD or O_NOMEM. */
static int comps_setup(int D, int K, int cov, const double* pi, const double* mu,
                       const double* covv, double ridge_rel, int* flags, comps_t* c) {
  memset(c, 0, sizeof(*c));
  c->D = D; c->K = K; c->cov = cov; c->mu = mu;
  c->logpi = (double*)malloc(sizeof(double) * K);
  c->logdet = (double*)malloc(sizeof(double) * K);
  if (cov == O_FULL) c->L = (double*)malloc(sizeof(double) * (size_t)K * D * D);
  else c->var = (double*)malloc(sizeof(double) * (size_t)K * (cov == O_DIAG ? D : 1));
  if (!c->logpi || !c->logdet || (cov == O_FULL ? !c->L : !c->var)) { comps_free(c); return O_NOMEM; }
  int status = O_OK;
  for (int k = 0; k < K; ++k) {
    flags[k] = 0;
    c->logpi[k] = pi[k] > 0.0 ? log(pi[k]) : -INFINITY;
    if (cov == O_FULL) {
      const double* S = covv + (size_t)k * D * D;
      double tr = 0.0;
      for (int d = 0; d < D; ++d) tr += S[d * D + d];
      double* L = c->L + (size_t)k * D * D;
      double add = ridge_rel * tr / D;
      if (cholesky(D, S, add, L)) {
        flags[k] |= FLAG_RIDGE;
        if (!(tr > 0.0) || cholesky(D, S, add + 1e-3 * tr / D, L)) {
          flags[k] |= FLAG_NOT_PD;
          status = O_NOT_PD;
          continue;
        }
      }
      double ld = 0.0;
      for (int d = 0; d < D; ++d) ld += log(L[d * D + d]);
      c->logdet[k] = 2.0 * ld;
    } else {
      int nv = cov == O_DIAG ? D : 1;
      const double* v = covv + (size_t)k * nv;
      double* w = c->var + (size_t)k * nv;
      double tr = 0.0;
      for (int d = 0; d < nv; ++d) tr += v[d];
      double add = ridge_rel * tr / nv;
      int ok = 1;
      for (int d = 0; d < nv; ++d) { w[d] = v[d] + add; if (!(w[d] > 0.0) || !isfinite(w[d])) ok = 0; }
      if (!ok) {
        flags[k] |= FLAG_RIDGE;
        ok = tr > 0.0;
        for (int d = 0; d < nv; ++d) { w[d] = v[d] + add + 1e-3 * tr / nv; if (!(w[d] > 0.0) || !isfinite(w[d])) ok = 0; }
        if (!ok) { flags[k] |= FLAG_NOT_PD; status = O_NOT_PD; continue; }
      }
      double ld = 0.0;
      for (int d = 0; d < nv; ++d) ld += log(w[d]);
      c->logdet[k] = cov == O_DIAG ? ld : D * ld;
    }
  }
  return status;
}

/* log pi_k + log N(x | mu_k, S_k).  work: D doubles. */
static double log_joint(const comps_t* c, int k, const double* x, double* work) {
  const int D = c->D;
  const double* mu = c->mu + (size_t)k * D;
  double d2 = 0.0;
  if (c->cov == O_FULL) {
    /* forward substitution L z = x - mu */
    const double* L = c->L + (size_t)k * D * D;
    for (int i = 0; i < D; ++i) {
      double v = x[i] - mu[i];
      for (int j = 0; j < i; ++j) v -= L[i * D + j] * work[j];
      work[i] = v / L[i * D + i];
      d2 += work[i] * work[i];
    }
  } else if (c->cov == O_DIAG) {
    const double* v = c->var + (size_t)k * D;
    for (int d = 0; d < D; ++d) { double t = x[d] - mu[d]; d2 += t * t / v[d]; }
  } else {
    double v = c->var[k];
    for (int d = 0; d < D; ++d) { double t = x[d] - mu[d]; d2 += t * t / v; }
  }
  return c->logpi[k] - 0.5 * d2 - 0.5 * c->logdet[k] - 0.5 * D * LOG_2PI;
}

/* Log-sum-exp over the K log joint densities l[], max subtracted first;
 * returns -inf if no term is finite. */
static double log_sum_exp(int K, const double* l) {
  double m = -INFINITY;
  for (int k = 0; k < K; ++k) if (l[k] > m) m = l[k];
  if (!isfinite(m)) return m;
  double s = 0.0;
  for (int k = 0; k < K; ++k) s += exp(l[k] - m);
  return m + log(s);
}

static int check_args(const void* X, int dtype, int64_t N, int D, int K, int cov) {
  if (!X || N < 0 || D <= 0 || K <= 0) return 0;
  if (dtype < O_F32 || dtype > O_BF16 || cov < O_FULL || cov > O_ISO) return 0;
  return 1;
}

/* ------------------------------------------------------- public API */

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Log joint density l[n*K + k] = log pi_k + log N(x_n | mu_k, S_k). */
int oracle_log_joint(const void* X, int dtype, int64_t N, int D, int K, const double* pi,
                     const double* mu, const double* cov, int cov_type, double ridge_rel,
                     double* out, int* flags) {
  if (!check_args(X, dtype, N, D, K, cov_type) || !out || !flags) return O_INVALID;
  comps_t c;
  int st = comps_setup(D, K, cov_type, pi, mu, cov, ridge_rel, flags, &c);
  if (st != O_OK) { comps_free(&c); return st; }
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * 2 * D);
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      load_x(X, dtype, n, D, x);
      for (int k = 0; k < K; ++k) out[(size_t)n * K + k] = log_joint(&c, k, x, x + D);
    }
    free(x);
  }
  comps_free(&c);
  return O_OK;
}

/* One EM iteration.  opts = {ridge_rel, var_floor, min_s0}.
 * Outputs the updated parameters, the log-likelihood at the input
 * parameters, optionally LSE_n (lse, N) and the raw statistics
 * s0 (K), s1 (K*D) and the centred second moments s2c (K*D*D full, lower
 * triangle filled; K*D otherwise, iso reports the per-dimension values). */
int oracle_em_step(const void* X, int dtype, int64_t N, int D, int K, const double* pi,
                   const double* mu, const double* cov, int cov_type, const double* opts,
                   double* pi_out, double* mu_out, double* cov_out, double* ll_out,
                   double* lse_out, double* s0_out, double* s1_out, double* s2c_out,
                   int* flags) {
  if (!check_args(X, dtype, N, D, K, cov_type) || N < 1 || !opts || !pi_out || !mu_out ||
      !cov_out || !ll_out || !flags)
    return O_INVALID;
  const double ridge_rel = opts[0], var_floor = opts[1], min_s0 = opts[2];
  comps_t c;
  int st = comps_setup(D, K, cov_type, pi, mu, cov, ridge_rel, flags, &c);
  if (st != O_OK) { comps_free(&c); return st; }
  const int full = cov_type == O_FULL;
  const size_t s2w = full ? (size_t)D * D : (size_t)D; /* second-moment entries per component */
  int nthr = 1;
#ifdef _OPENMP
  nthr = omp_get_max_threads();
#endif
  double* s0 = (double*)calloc((size_t)nthr * K, sizeof(double));
  double* s1 = (double*)calloc((size_t)nthr * K * D, sizeof(double));
  double* s2 = (double*)calloc((size_t)nthr * K * s2w, sizeof(double));
  double* llp = (double*)calloc((size_t)nthr, sizeof(double));
  double* mun = (double*)malloc(sizeof(double) * (size_t)K * D);
  int* bad = (int*)calloc((size_t)nthr, sizeof(int));
  if (!s0 || !s1 || !s2 || !llp || !mun || !bad) {
    free(s0); free(s1); free(s2); free(llp); free(mun); free(bad); comps_free(&c);
    return O_NOMEM;
  }

  /* Pass 1: responsibilities, s0, s1, log-likelihood. */
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    double* x = (double*)malloc(sizeof(double) * 2 * D);
    double* l = (double*)malloc(sizeof(double) * K);
    double* my0 = s0 + (size_t)t * K;
    double* my1 = s1 + (size_t)t * K * D;
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      load_x(X, dtype, n, D, x);
      for (int k = 0; k < K; ++k) l[k] = log_joint(&c, k, x, x + D);
      double lse = log_sum_exp(K, l);
      if (lse_out) lse_out[n] = lse;
      if (!isfinite(lse)) { bad[t] = 1; continue; }
      llp[t] += lse;
      for (int k = 0; k < K; ++k) {
        double g = exp(l[k] - lse);
        my0[k] += g;
        for (int d = 0; d < D; ++d) my1[(size_t)k * D + d] += g * x[d];
      }
    }
    free(x); free(l);
  }
  /* Merge thread partials in thread order. */
  for (int t = 1; t < nthr; ++t) {
    for (int k = 0; k < K; ++k) s0[k] += s0[(size_t)t * K + k];
    for (size_t i = 0; i < (size_t)K * D; ++i) s1[i] += s1[(size_t)t * K * D + i];
    llp[0] += llp[t];
    bad[0] |= bad[t];
  }
  for (int k = 0; k < K; ++k)
    for (int d = 0; d < D; ++d)
      mun[(size_t)k * D + d] = s0[k] > 0.0 ? s1[(size_t)k * D + d] / s0[k] : mu[(size_t)k * D + d];

  /* Pass 2: second moments about the new means. */
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    double* x = (double*)malloc(sizeof(double) * 3 * D);
    double* l = (double*)malloc(sizeof(double) * K);
    double* my2 = s2 + (size_t)t * K * s2w;
    double* y = x + 2 * D;
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      load_x(X, dtype, n, D, x);
      for (int k = 0; k < K; ++k) l[k] = log_joint(&c, k, x, x + D);
      double lse = log_sum_exp(K, l);
      if (!isfinite(lse)) continue;
      for (int k = 0; k < K; ++k) {
        double g = exp(l[k] - lse);
        for (int d = 0; d < D; ++d) y[d] = x[d] - mun[(size_t)k * D + d];
        double* o = my2 + (size_t)k * s2w;
        if (full) {
          for (int a = 0; a < D; ++a)
            for (int b = 0; b <= a; ++b) o[(size_t)a * D + b] += g * y[a] * y[b];
        } else {
          for (int d = 0; d < D; ++d) o[d] += g * y[d] * y[d];
        }
      }
    }
    free(x); free(l);
  }
  for (int t = 1; t < nthr; ++t)
    for (size_t i = 0; i < (size_t)K * s2w; ++i) s2[i] += s2[(size_t)t * K * s2w + i];

  /* M-step (maximum-likelihood update from the statistics). */
  for (int k = 0; k < K; ++k) {
    pi_out[k] = s0[k] / (double)N;
    const double* mk = mu + (size_t)k * D;
    if (!(s0[k] >= min_s0) || s0[k] <= 0.0) {
      flags[k] |= FLAG_EMPTY;
      for (int d = 0; d < D; ++d) mu_out[(size_t)k * D + d] = mk[d];
      size_t nc = full ? (size_t)D * D : (cov_type == O_DIAG ? (size_t)D : 1);
      for (size_t i = 0; i < nc; ++i) cov_out[(size_t)k * nc + i] = cov[(size_t)k * nc + i];
      continue;
    }
    for (int d = 0; d < D; ++d) mu_out[(size_t)k * D + d] = mun[(size_t)k * D + d];
    const double* o = s2 + (size_t)k * s2w;
    if (full) {
      double* Sk = cov_out + (size_t)k * D * D;
      for (int a = 0; a < D; ++a)
        for (int b = 0; b <= a; ++b) Sk[a * D + b] = Sk[b * D + a] = o[(size_t)a * D + b] / s0[k];
      for (int a = 0; a < D; ++a)
        if (Sk[a * D + a] < var_floor) { Sk[a * D + a] = var_floor; flags[k] |= FLAG_FLOOR; }
    } else if (cov_type == O_DIAG) {
      for (int d = 0; d < D; ++d) {
        double v = o[d] / s0[k];
        if (v < var_floor) { v = var_floor; flags[k] |= FLAG_FLOOR; }
        cov_out[(size_t)k * D + d] = v;
      }
    } else {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += o[d];
      double v = acc / ((double)D * s0[k]);
      if (v < var_floor) { v = var_floor; flags[k] |= FLAG_FLOOR; }
      cov_out[k] = v;
    }
  }
  *ll_out = bad[0] ? NAN : llp[0];
  if (s0_out) memcpy(s0_out, s0, sizeof(double) * K);
  if (s1_out) memcpy(s1_out, s1, sizeof(double) * (size_t)K * D);
  if (s2c_out) memcpy(s2c_out, s2, sizeof(double) * (size_t)K * s2w);
  st = bad[0] ? O_NONFINITE : O_OK;
  free(s0); free(s1); free(s2); free(llp); free(mun); free(bad);
  comps_free(&c);
  return st;
}

/* Top-m components per point: ids[n*m + j] by descending log joint density
 * (ties to the lower index), gamma = full-K posterior of that component,
 * lse[n] = log sum_k pi_k N(x_n|...). */
int oracle_topm(const void* X, int dtype, int64_t N, int D, int K, const double* pi,
                const double* mu, const double* cov, int cov_type, double ridge_rel, int m,
                int32_t* ids, double* gamma, double* lse) {
  if (!check_args(X, dtype, N, D, K, cov_type) || m < 1 || m > K || !ids || !gamma) return O_INVALID;
  int* flags = (int*)malloc(sizeof(int) * K);
  if (!flags) return O_NOMEM;
  comps_t c;
  int st = comps_setup(D, K, cov_type, pi, mu, cov, ridge_rel, flags, &c);
  free(flags);
  if (st != O_OK) { comps_free(&c); return st; }
  int bad = 0;
#pragma omp parallel reduction(| : bad)
  {
    double* x = (double*)malloc(sizeof(double) * 2 * D);
    double* l = (double*)malloc(sizeof(double) * K);
    int* used = (int*)malloc(sizeof(int) * K);
#pragma omp for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
      load_x(X, dtype, n, D, x);
      for (int k = 0; k < K; ++k) l[k] = log_joint(&c, k, x, x + D);
      double s = log_sum_exp(K, l);
      if (lse) lse[n] = s;
      if (!isfinite(s)) bad = 1;
      /* selection by repeated maximum: a full ordering of the first m */
      for (int k = 0; k < K; ++k) used[k] = 0;
      for (int j = 0; j < m; ++j) {
        int best = -1;
        for (int k = 0; k < K; ++k) {
          if (used[k]) continue;
          if (best < 0 || l[k] > l[best]) best = k;
        }
        used[best] = 1;
        ids[(size_t)n * m + j] = best;
        gamma[(size_t)n * m + j] = exp(l[best] - s);
      }
    }
    free(x); free(l); free(used);
  }
  comps_free(&c);
  return bad ? O_NONFINITE : O_OK;
}
