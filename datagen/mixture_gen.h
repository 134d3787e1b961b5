/*
 * mixture_gen.h - seeded, counter-based synthetic mixture data.
 *
 * This module only makes inputs.  It holds none of the Gaussian-mixture EM
 * arithmetic (no densities, responsibilities or statistics): it draws points
 * from a planted mixture whose parameters are given as tables.  The same
 * source is compiled for the host (gcc, -ffp-contract=off) and for the GPU
 * (nvcc, -fmad=false), and every step is integer work or a correctly rounded
 * IEEE double operation (+, -, *, /, sqrt) done in one fixed order, so the
 * host and the device produce the same bits for every point.  That lets a
 * host-side checker regenerate any point of a device-resident data set by
 * its index.
 *
 * Random numbers: Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11), keyed by (seed, stream) and
 * addressed by (point index, pair index, attempt).
 * Normal variates: Marsaglia and Bray's polar method (1964), with a natural
 * logarithm written here (exponent split plus the atanh series
 * ln m = 2 atanh((m-1)/(m+1))), so no platform libm enters the bits.
 * Quantisation: round-to-nearest-even from double straight to fp16 / bf16 /
 * fp32 (no double rounding through fp32).
 */
#ifndef MIXTURE_GEN_H
#define MIXTURE_GEN_H

#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define GEN_HD static __host__ __device__ __forceinline__
#else
#define GEN_HD static inline
#include <math.h>
#endif

enum { GEN_F32 = 0, GEN_F16 = 1, GEN_BF16 = 2 };
enum { GEN_MIX_DIAG = 0, GEN_MIX_FULL = 1, GEN_MIX_SPHERE = 2, GEN_MIX_IVF = 3 };
enum { GEN_STREAM_PARAMS = 1, GEN_STREAM_POINT_NORMAL = 2, GEN_STREAM_POINT_UNIFORM = 3,
       GEN_STREAM_INIT = 4 };

/* Tables describing one planted mixture.  All pointers address the memory
 * space of the side that runs gen_point (host arrays on the host, device
 * arrays on the GPU). */
typedef struct {
  int kind;            /* GEN_MIX_* */
  int D, K;
  uint64_t seed;
  double noise;        /* SPHERE: noise standard deviation before normalising */
  double mid_frac;     /* IVF: fraction of points drawn as midpoints of two centres */
  const double* cdf;   /* [K] running sum of the weights (last entry = total) */
  const double* mu;    /* [K*D] centres */
  const double* sd;    /* [K*D] per-dimension standard deviations (DIAG, IVF) */
  const double* chol;  /* [K*D*D] row-major lower Cholesky factors (FULL) */
} gen_mixture;

GEN_HD uint64_t gen_dbits(double x) { uint64_t b; memcpy(&b, &x, 8); return b; }
GEN_HD double gen_bitsd(uint64_t b) { double x; memcpy(&x, &b, 8); return x; }

/* Philox4x32-10 block: ten rounds of the published round function, the key
 * bumped by the Weyl constants between rounds. */
GEN_HD void gen_philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
  for (int r = 0; r < 10; ++r) {
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k0;
    uint32_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
}

/* Block for (seed, stream) at counter (idx, j, attempt). */
GEN_HD void gen_block(uint64_t seed, uint32_t stream, uint64_t idx, uint32_t j, uint32_t attempt,
                      uint32_t out[4]) {
  out[0] = (uint32_t)idx;
  out[1] = (uint32_t)(idx >> 32);
  out[2] = j;
  out[3] = attempt;
  gen_philox4x32_10(out, (uint32_t)seed ^ (uint32_t)(seed >> 32), stream);
}

/* 53-bit uniform on [0, 1) from two words. */
GEN_HD double gen_u53(uint32_t a, uint32_t b) {
  uint64_t m = ((uint64_t)(a >> 5) << 26) | (uint64_t)(b >> 6);
  return (double)m * (1.0 / 9007199254740992.0);
}

/* Natural log of a positive, finite, normal double.  s = m * 2^e with
 * m in [sqrt(1/2), sqrt(2)); ln m = 2 atanh(t), t = (m-1)/(m+1), |t| < 0.1716,
 * summed to t^23 (the next term is below 2^-60 relative). */
GEN_HD double gen_ln(double s) {
  uint64_t b = gen_dbits(s);
  int e = (int)((b >> 52) & 0x7ff) - 1023;
  double m = gen_bitsd((b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull);
  if (m > 1.4142135623730951) { m = m * 0.5; e += 1; }
  double t = (m - 1.0) / (m + 1.0);
  double t2 = t * t;
  double p = 1.0 / 23.0;
  p = p * t2 + 1.0 / 21.0;
  p = p * t2 + 1.0 / 19.0;
  p = p * t2 + 1.0 / 17.0;
  p = p * t2 + 1.0 / 15.0;
  p = p * t2 + 1.0 / 13.0;
  p = p * t2 + 1.0 / 11.0;
  p = p * t2 + 1.0 / 9.0;
  p = p * t2 + 1.0 / 7.0;
  p = p * t2 + 1.0 / 5.0;
  p = p * t2 + 1.0 / 3.0;
  p = p * t2 + 1.0;
  double lnm = 2.0 * t * p;
  /* ln 2 split so that e * LN2_HI is exact for |e| < 2^11 (the two-part
   * constant of Sun Microsystems' freely distributed fdlibm, e_log.c). */
  const double LN2_HI = 6.93147180369123816490e-01;
  const double LN2_LO = 1.90821492927058770002e-10;
  double ed = (double)e;
  return ed * LN2_HI + (ed * LN2_LO + lnm);
}

/* Two independent standard normals for (seed, stream, idx, pair j). */
GEN_HD void gen_normal_pair(uint64_t seed, uint32_t stream, uint64_t idx, uint32_t j,
                            double* z0, double* z1) {
  for (uint32_t attempt = 0;; ++attempt) {
    uint32_t w[4];
    gen_block(seed, stream, idx, j, attempt, w);
    double u = 2.0 * gen_u53(w[0], w[1]) - 1.0;
    double v = 2.0 * gen_u53(w[2], w[3]) - 1.0;
    double s = u * u + v * v;
    if (s > 0.0 && s < 1.0) {
      double f = sqrt((-2.0 * gen_ln(s)) / s);
      *z0 = u * f;
      *z1 = v * f;
      return;
    }
  }
}

/* One uniform pair for (seed, stream, idx, j). */
GEN_HD void gen_uniform_pair(uint64_t seed, uint32_t stream, uint64_t idx, uint32_t j,
                             double* u0, double* u1) {
  uint32_t w[4];
  gen_block(seed, stream, idx, j, 0, w);
  *u0 = gen_u53(w[0], w[1]);
  *u1 = gen_u53(w[2], w[3]);
}

/* Round a double to the nearest binary16 / bfloat16 value (ties to even).
 * sig is the 53-bit significand; the kept part is sig >> shift. */
GEN_HD uint16_t gen_round_small(double x, int man_bits, int emin, int bias, uint16_t inf_bits) {
  uint64_t b = gen_dbits(x);
  uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  int ef = (int)((b >> 52) & 0x7ff);
  uint64_t man = b & 0x000FFFFFFFFFFFFFull;
  if (ef == 0x7ff) return (uint16_t)(sign | inf_bits | (man ? 1u : 0u));
  if (ef == 0) return sign; /* zero or a double subnormal: far below both ranges */
  int E = ef - 1023;
  uint64_t sig = man | (1ull << 52);
  int sub = (E < emin) ? (emin - E) : 0;
  int shift = 52 - man_bits + sub;
  if (shift >= 63) return sign;
  uint64_t r = sig >> shift;
  uint64_t rem = sig & ((1ull << shift) - 1);
  uint64_t half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (r & 1))) r += 1;
  if (sub) return (uint16_t)(sign | (uint16_t)r); /* a carry into 1<<man_bits is the smallest normal */
  if (r == (2ull << man_bits)) { r >>= 1; E += 1; }
  int field = E + bias;
  if (field >= (int)(inf_bits >> man_bits)) return (uint16_t)(sign | inf_bits);
  return (uint16_t)(sign | ((uint16_t)field << man_bits) | (uint16_t)(r - (1ull << man_bits)));
}
GEN_HD uint16_t gen_to_f16(double x) { return gen_round_small(x, 10, -14, 15, 0x7C00u); }
GEN_HD uint16_t gen_to_bf16(double x) { return gen_round_small(x, 7, -126, 127, 0x7F80u); }

GEN_HD void gen_store(void* row, int dtype, int d, double v) {
  if (dtype == GEN_F32) ((float*)row)[d] = (float)v;
  else if (dtype == GEN_F16) ((uint16_t*)row)[d] = gen_to_f16(v);
  else ((uint16_t*)row)[d] = gen_to_bf16(v);
}

/* Index of the component for uniform u in [0, 1): the first k with
 * u * total < cdf[k] (binary search; comparisons only). */
GEN_HD int gen_pick(const double* cdf, int K, double u) {
  double target = u * cdf[K - 1];
  int lo = 0, hi = K - 1;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (target < cdf[mid]) hi = mid; else lo = mid + 1;
  }
  return lo;
}

/* Draw point idx of mixture m and store its D coordinates in `row`
 * (dtype GEN_*).  `scratch` must hold D doubles (used by FULL only). */
GEN_HD void gen_point(const gen_mixture* m, uint64_t idx, int dtype, void* row, double* scratch) {
  const int D = m->D;
  double ua, ub;
  gen_uniform_pair(m->seed, GEN_STREAM_POINT_UNIFORM, idx, 0, &ua, &ub);
  if (m->kind == GEN_MIX_IVF && ub < m->mid_frac) {
    /* Midpoint of two distinct centres a != b, with centre a's noise. */
    double uc, ud;
    gen_uniform_pair(m->seed, GEN_STREAM_POINT_UNIFORM, idx, 1, &uc, &ud);
    int a = (int)(uc * (double)m->K);
    int bsel = (int)(ud * (double)(m->K - 1));
    int bb = bsel + (bsel >= a ? 1 : 0);
    for (int j = 0; j < D / 2; ++j) {
      double z0, z1;
      gen_normal_pair(m->seed, GEN_STREAM_POINT_NORMAL, idx, (uint32_t)j, &z0, &z1);
      int d0 = 2 * j, d1 = 2 * j + 1;
      double c0 = (m->mu[(size_t)a * D + d0] + m->mu[(size_t)bb * D + d0]) * 0.5;
      double c1 = (m->mu[(size_t)a * D + d1] + m->mu[(size_t)bb * D + d1]) * 0.5;
      gen_store(row, dtype, d0, c0 + m->sd[(size_t)a * D + d0] * z0);
      gen_store(row, dtype, d1, c1 + m->sd[(size_t)a * D + d1] * z1);
    }
    return;
  }
  int k = gen_pick(m->cdf, m->K, ua);
  const double* mu = m->mu + (size_t)k * D;
  if (m->kind == GEN_MIX_DIAG || m->kind == GEN_MIX_IVF) {
    const double* sd = m->sd + (size_t)k * D;
    for (int j = 0; j < D / 2; ++j) {
      double z0, z1;
      gen_normal_pair(m->seed, GEN_STREAM_POINT_NORMAL, idx, (uint32_t)j, &z0, &z1);
      gen_store(row, dtype, 2 * j, mu[2 * j] + sd[2 * j] * z0);
      gen_store(row, dtype, 2 * j + 1, mu[2 * j + 1] + sd[2 * j + 1] * z1);
    }
  } else if (m->kind == GEN_MIX_SPHERE) {
    /* y = centre + noise * eps, then y / |y| (norm summed in index order). */
    double ss = 0.0;
    for (int j = 0; j < D / 2; ++j) {
      double z0, z1;
      gen_normal_pair(m->seed, GEN_STREAM_POINT_NORMAL, idx, (uint32_t)j, &z0, &z1);
      double y0 = mu[2 * j] + m->noise * z0;
      double y1 = mu[2 * j + 1] + m->noise * z1;
      ss = ss + y0 * y0;
      ss = ss + y1 * y1;
    }
    double inv = 1.0 / sqrt(ss);
    for (int j = 0; j < D / 2; ++j) {
      double z0, z1;
      gen_normal_pair(m->seed, GEN_STREAM_POINT_NORMAL, idx, (uint32_t)j, &z0, &z1);
      double y0 = mu[2 * j] + m->noise * z0;
      double y1 = mu[2 * j + 1] + m->noise * z1;
      gen_store(row, dtype, 2 * j, y0 * inv);
      gen_store(row, dtype, 2 * j + 1, y1 * inv);
    }
  } else { /* GEN_MIX_FULL: x = mu + L eps, row sums in index order */
    const double* L = m->chol + (size_t)k * D * D;
    for (int j = 0; j < D / 2; ++j) {
      double z0, z1;
      gen_normal_pair(m->seed, GEN_STREAM_POINT_NORMAL, idx, (uint32_t)j, &z0, &z1);
      scratch[2 * j] = z0;
      scratch[2 * j + 1] = z1;
    }
    for (int i = 0; i < D; ++i) {
      double acc = 0.0;
      for (int j = 0; j <= i; ++j) acc = acc + L[(size_t)i * D + j] * scratch[j];
      gen_store(row, dtype, i, mu[i] + acc);
    }
  }
}

#endif /* MIXTURE_GEN_H */
