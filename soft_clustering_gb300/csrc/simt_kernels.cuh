// simt_kernels.cuh - fp32 CUDA-core path of the fused EM step (all covariance
// types).  It is the general path (any K, all three covariance types, small
// problems where a tensor-core tile would be mostly padding) and the exact
// yardstick the tensor-core kernels are tested beside.
//
// Two passes over X, no N x K buffer:
//   lse_kernel:   one thread per point; l_nk for every component in the
//                 centred form (x - mu) with an online max/sum over k
//                 ("low-precision GMM operator" notes, sec. 3.2 fused
//                 distance + posterior, sec. 4.2 log-sum-exp); writes LSE_n,
//                 a per-block log-likelihood partial and, for assignment,
//                 the top-m components.
//   stats_kernel: grid (component chunk, point partition); recomputes l_nk
//                 for its chunk, g = exp(l - LSE_n), and accumulates
//                 [s0, sum g (x-mu), sum g (x-mu)^2 or (x-mu)(x-mu)^T]
//                 (Flash-GMM summary, Method: online sufficient statistics)
//                 about the input mean, fp32 per 64-point tile, fp64 across
//                 tiles, into a per-block partial.
#pragma once
#include <math.h>

#include <type_traits>

#include "gmm_internal.cuh"

namespace gmm {

namespace simt {

constexpr int kLseThreads = 128;
constexpr int kStatThreads = 256;
constexpr int kStatTile = 64;

// Components per chunk of the statistics kernel, chosen so that a thread
// owns at most ~9 (diag) accumulators.
template <int D, int COV>
struct StatShape {
  static constexpr int F = COV == GMM_COV_FULL ? 1 + D + D * (D + 1) / 2 : 1 + 2 * D;
  static constexpr int KC = COV == GMM_COV_FULL ? (D >= 64 ? 1 : (D == 32 ? 4 : 16))
                                                 : (D == 128 ? 8 : (D == 64 ? 16 : (D == 32 ? 32 : 64)));
  static constexpr int SLOTS = (KC * F + kStatThreads - 1) / kStatThreads;
};

// Components per shared-memory chunk of the LSE kernel.
template <int D, int COV>
struct LseShape {
  static constexpr int P = COV == GMM_COV_FULL ? D * D : (COV == GMM_COV_DIAG ? D : 1);
  static constexpr int KC = COV == GMM_COV_FULL ? (D == 128 ? 1 : (D == 64 ? 2 : 8)) : 16;
};

template <int XT, int D>
__device__ __forceinline__ void load_row(const void* X, int64_t n, float* x) {
#pragma unroll
  for (int d = 0; d < D; ++d) x[d] = load_x<XT>(X, (size_t)n * D + d);
}

// Sum of w_d (x_d - mu_d)^2 over d for diag / iso.  For D >= 64 the order
// is the one the tensor-core path's warp-cooperative refinement uses: 32
// partial sums over D/32 consecutive dimensions each (sequential fma), then
// the xor-butterfly tree of a warp reduction, so every kernel produces the
// same bits for the same (point, component).  Smaller D: 4 interleaved partial
// sums combined pairwise.
template <int D, int COV, typename XF, typename MF, typename WF>
__device__ __forceinline__ float dist2_diag(XF xf, MF mf, WF wf) {
  if constexpr (D >= 64) {
    constexpr int DPL = D / 32;
    float p[32];
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const int d = l * DPL + i;
        const float t = xf(d) - mf(d);
        part = fmaf(t * t, wf(d), part);
      }
      p[l] = part;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < o; ++i) p[i] = p[i] + p[i + o];
    return p[0];
  } else {
    float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int d = 0; d < D; ++d) {
      const float t = xf(d) - mf(d);
      p[d & 3] = fmaf(t * t, wf(d), p[d & 3]);
    }
    return (p[0] + p[2]) + (p[1] + p[3]);
  }
}

// log joint of one component for a point held in registers (diag / iso).
template <int D, int COV>
__device__ __forceinline__ float logj_diag(const float* x, const float* mu, const float* prec,
                                           float c) {
  const float s = dist2_diag<D, COV>([&](int d) { return x[d]; }, [&](int d) { return mu[d]; },
                                     [&](int d) { return COV == GMM_COV_DIAG ? prec[d] : prec[0]; });
  return c - 0.5f * s;
}

// Full: z = W (x - mu), d^2 = z.z, with W lower triangular.  Each z_i is
// summed in 4 interleaved partial sums; d^2 is accumulated with Neumaier's
// compensated summation.
template <int D>
__device__ __forceinline__ float logj_full(const float* y, const float* W, float c) {
  float s = 0.f, comp = 0.f;
  // fully unrolled up to D = 64 so y[] stays in registers
#pragma unroll(D <= 64 ? D : 4)
  for (int i = 0; i < D; ++i) {
    float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
    const float* Wi = W + i * D;
    int j = 0;
#pragma unroll(D <= 64 ? D / 4 : 1)
    for (; j + 3 <= i; j += 4) {
      z0 = fmaf(Wi[j], y[j], z0);
      z1 = fmaf(Wi[j + 1], y[j + 1], z1);
      z2 = fmaf(Wi[j + 2], y[j + 2], z2);
      z3 = fmaf(Wi[j + 3], y[j + 3], z3);
    }
    for (; j <= i; ++j) z0 = fmaf(Wi[j], y[j], z0);
    const float z = (z0 + z1) + (z2 + z3);
    const float q = z * z;
    const float t = s + q;
    comp += fabsf(s) >= fabsf(q) ? (s - t) + q : (q - t) + s;
    s = t;
  }
  return c - 0.5f * (s + comp);
}

template <int D, int COV, int XT>
__global__ void __launch_bounds__(kLseThreads)
lse_kernel(const void* __restrict__ X, int64_t N, int K, const void* __restrict__ prepared,
           PreparedLayout L, float* __restrict__ lse_out, double* __restrict__ ll_part, int m,
           int32_t* __restrict__ ids, float* __restrict__ gamma, DeviceStatus* st,
           const uint32_t* __restrict__ rows, const uint32_t* __restrict__ row_count) {
  using S = LseShape<D, COV>;
  extern __shared__ float sm[];
  float* s_mu = sm;                      // KC*D
  float* s_prec = s_mu + S::KC * D;      // KC*P
  float* s_c = s_prec + S::KC * S::P;    // KC
  __shared__ double red[kLseThreads / 32];

  // Dense mode: point n = group * 128 + thread.  Row-list mode: the points
  // rows[0 .. *row_count) (the rows the tensor-core kernel handed over).
  const int64_t cnt = rows ? (int64_t)*row_count : N;
  const int64_t ngroups = (cnt + kLseThreads - 1) / kLseThreads;
  double ll_acc = 0.0;
  for (int64_t grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
  const int64_t idx = grp * kLseThreads + threadIdx.x;
  const bool valid = idx < cnt;
  const int64_t n = valid ? (rows ? (int64_t)rows[idx] : idx) : 0;
  const float* g_c = at<float>(prepared, L.off_c);
  const float* g_mu = at<float>(prepared, L.off_mu);
  const float* g_prec = at<float>(prepared, L.off_prec);

  float x[D];
  if (COV != GMM_COV_FULL) {
    if (valid) load_row<XT, D>(X, n, x);
    else
#pragma unroll
      for (int d = 0; d < D; ++d) x[d] = 0.f;
  }
  float run_m = -INFINITY, run_s = 0.f;
  float tv[8];
  int ti[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) { tv[j] = -INFINITY; ti[j] = 0x7fffffff; }

  for (int k0 = 0; k0 < K; k0 += S::KC) {
    const int kc = min(S::KC, K - k0);
    __syncthreads();
    for (int i = threadIdx.x; i < kc * D; i += kLseThreads) s_mu[i] = g_mu[(size_t)k0 * D + i];
    for (int i = threadIdx.x; i < kc * S::P; i += kLseThreads)
      s_prec[i] = g_prec[(size_t)k0 * S::P + i];
    for (int i = threadIdx.x; i < kc; i += kLseThreads) s_c[i] = g_c[k0 + i];
    __syncthreads();
    if (!valid) continue;
    for (int kk = 0; kk < kc; ++kk) {
      const float c = s_c[kk];
      if (c == -INFINITY) continue;
      float l;
      if constexpr (COV == GMM_COV_FULL) {
        float y[D];
#pragma unroll
        for (int d = 0; d < D; ++d) y[d] = load_x<XT>(X, (size_t)n * D + d) - s_mu[kk * D + d];
        l = logj_full<D>(y, s_prec + kk * S::P, c);
      } else {
        l = logj_diag<D, COV>(x, s_mu + kk * D, s_prec + kk * S::P, c);
      }
      // online log-sum-exp (running max, rescaled sum)
      if (l > run_m) {
        run_s = run_s * expf(run_m - l) + 1.f;
        run_m = l;
      } else {
        run_s += expf(l - run_m);
      }
      if (m > 0 && l > tv[m - 1]) {
        // insertion into the descending top-m list; a value equal to an
        // entry goes after it, so ties keep the lower component first
        const int k = k0 + kk;
        bool placed = false;
#pragma unroll
        for (int t = 7; t >= 1; --t) {
          if (t < m && !placed) {
            if (l > tv[t - 1]) { tv[t] = tv[t - 1]; ti[t] = ti[t - 1]; }
            else { tv[t] = l; ti[t] = k; placed = true; }
          }
        }
        if (!placed) { tv[0] = l; ti[0] = k; }
      }
    }
  }
  if (valid) {
    const float lse = run_m + logf(run_s);
    if (lse_out) lse_out[n] = lse;
    if (!isfinite(lse)) raise_status(st, GMM_ERR_NONFINITE);
    ll_acc += (double)lse;
    for (int j = 0; j < m; ++j) {
      ids[n * m + j] = ti[j] == 0x7fffffff ? -1 : ti[j];
      gamma[n * m + j] = tv[j] == -INFINITY ? 0.f : expf(tv[j] - lse);
    }
  }
  }  // groups
  if (ll_part) {
    double lsev = warp_sum(ll_acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = lsev;
    __syncthreads();
    if (threadIdx.x == 0) {
      double s = 0.0;
      for (int i = 0; i < kLseThreads / 32; ++i) s += red[i];
      ll_part[blockIdx.x] = s;
    }
  }
}

// Statistics of one component chunk over one point partition.  Per 64-point
// tile: responsibilities, the tile's weighted count t0 and first moment t1
// about the fixed centre c_k, then the tile's second moment M2_t about the
// tile's own weighted mean, merged into the block's running sums with Chan,
// Golub and LeVeque's pairwise update (M2 += M2_t + d d^T S0 t0 / (S0 + t0),
// d = tile mean - running mean) in fp64.  Output per block and component:
// [S0 | S1 about c_k | M2 about the block mean].
template <int D, int COV, int XT>
__global__ void __launch_bounds__(kStatThreads)
stats_kernel(const void* __restrict__ X, int64_t N, int K, const void* __restrict__ prepared,
             PreparedLayout L, const float* __restrict__ lse, int64_t rows_per_part,
             double* __restrict__ part, int accumulate, const uint32_t* __restrict__ rows,
             const uint32_t* __restrict__ row_count) {
  using SS = StatShape<D, COV>;
  constexpr int KC = SS::KC, F = SS::F, SLOTS = SS::SLOTS, T = kStatTile;
  constexpr int P = LseShape<D, COV>::P;
  constexpr int XS = D + 1;  // padded row of the x tile
  constexpr int YS = D + 1;  // padded row of the y tile (full): a warp's rows in different banks
  extern __shared__ double smd[];
  double* s_r0 = smd;                 // KC     running S0 of this block
  double* s_r1 = s_r0 + KC;           // KC*D   running S1 of this block
  double* s_rm = s_r1 + KC * D;       // KC*D   running mean S1 / S0
  double* s_fac = s_rm + KC * D;      // KC     this tile's correction weight
  float* s_x = (float*)(s_fac + KC);  // T*XS
  float* s_g = s_x + T * XS;          // T*KC
  float* s_mu = s_g + T * KC;         // KC*D
  float* s_prec = s_mu + KC * D;      // KC*P
  float* s_c = s_prec + KC * P;       // KC
  float* s_t0 = s_c + KC;             // KC     tile sums
  float* s_t1 = s_t0 + KC;            // KC*D
  float* s_y = s_t1 + KC * D;         // full only: T*KC*YS  (y = x - c)
  short* s_pair = (short*)(s_y + (COV == GMM_COV_FULL ? T * KC * YS : 0));

  const int k0 = blockIdx.x * KC;
  const int kc = min(KC, K - k0);
  // Dense mode: points [0, N).  Row-list mode: the points rows[0 .. *row_count),
  // split evenly over the partitions (the count is only known on the device).
  const int64_t cnt = rows ? (int64_t)*row_count : N;
  if (rows) {
    // at least four tiles per partition: with few handed-over rows most
    // partitions get none, and leave their partial as it is (accumulating)
    // or only zero it (the first block of rows)
    rows_per_part = (cnt + gridDim.y - 1) / gridDim.y;
    rows_per_part = (rows_per_part + T - 1) / T * T;
    if (rows_per_part < 4 * T) rows_per_part = 4 * T;
  }
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_part;
  const int64_t r1 = min(cnt, r0 + rows_per_part);
  if (rows && r0 >= cnt) {
    if (!accumulate) {
      double* out = part + (size_t)blockIdx.y * K * F;
      for (int f = threadIdx.x; f < kc * F; f += kStatThreads) out[(size_t)k0 * F + f] = 0.0;
    }
    return;
  }

  for (int i = threadIdx.x; i < kc * D; i += kStatThreads)
    s_mu[i] = at<float>(prepared, L.off_mu)[(size_t)k0 * D + i];
  for (int i = threadIdx.x; i < kc * P; i += kStatThreads)
    s_prec[i] = at<float>(prepared, L.off_prec)[(size_t)k0 * P + i];
  for (int i = threadIdx.x; i < kc; i += kStatThreads) s_c[i] = at<float>(prepared, L.off_c)[k0 + i];
  for (int i = threadIdx.x; i < KC * (2 * D + 2); i += kStatThreads) smd[i] = 0.0;
  if constexpr (COV == GMM_COV_FULL) {
    for (int e = threadIdx.x; e < D * (D + 1) / 2; e += kStatThreads) {
      // e enumerates the lower triangle row by row: (a, b) with b <= a
      int a = (int)((sqrtf(8.f * e + 1.f) - 1.f) * 0.5f);
      while ((a + 1) * (a + 2) / 2 <= e) ++a;
      while (a * (a + 1) / 2 > e) --a;
      int b = e - a * (a + 1) / 2;
      s_pair[2 * e] = (short)a;
      s_pair[2 * e + 1] = (short)b;
    }
  }

  double accd[SLOTS];
  float tsum[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) { accd[s] = 0.0; tsum[s] = 0.f; }

  for (int64_t t0r = r0; t0r < r1; t0r += T) {
    const int tn = (int)min((int64_t)T, r1 - t0r);
    __syncthreads();
    for (int i = threadIdx.x; i < T * D; i += kStatThreads) {
      int r = i / D, d = i % D;
      const int64_t src = r < tn ? (rows ? (int64_t)rows[t0r + r] : t0r + r) : 0;
      s_x[r * XS + d] = r < tn ? load_x<XT>(X, (size_t)src * D + d) : 0.f;
    }
    __syncthreads();
    // responsibilities of this chunk for the tile
    // lanes of a warp share one component (broadcast reads of its
    // parameters) and walk consecutive rows of the padded x tile
    for (int pidx = threadIdx.x; pidx < T * KC; pidx += kStatThreads) {
      const int kk = pidx / T, r = pidx % T;
      float g = 0.f;
      if (r < tn && kk < kc && s_c[kk] != -INFINITY) {
        float l;
        if constexpr (COV == GMM_COV_FULL) {
          float y[D];
#pragma unroll
          for (int d = 0; d < D; ++d) {
            y[d] = s_x[r * XS + d] - s_mu[kk * D + d];
            s_y[(r * KC + kk) * YS + d] = y[d];
          }
          l = logj_full<D>(y, s_prec + kk * P, s_c[kk]);
        } else {
          // same summation order as every other log-density evaluation
          const float* xr = s_x + r * XS;
          const float* mk = s_mu + kk * D;
          const float* wk = s_prec + kk * P;
          const float d2 = dist2_diag<D, COV>(
              [&](int d) { return xr[d]; }, [&](int d) { return mk[d]; },
              [&](int d) { return COV == GMM_COV_DIAG ? wk[d] : wk[0]; });
          l = s_c[kk] - 0.5f * d2;
        }
        g = expf(l - lse[rows ? (int64_t)rows[t0r + r] : t0r + r]);
      }
      s_g[r * KC + kk] = g;
    }
    __syncthreads();
    // phase A: tile count and first moment about the centre
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int f = threadIdx.x + s * kStatThreads;
      if (f >= kc * F) continue;
      const int kk = f / F, feat = f % F;
      if (feat > D) continue;
      float acc = 0.f;
      if (feat == 0) {
        for (int r = 0; r < tn; ++r) acc += s_g[r * KC + kk];
        s_t0[kk] = acc;
        // weight of the pairwise correction: S0 t0 / (S0 + t0)
        const double R0 = s_r0[kk];
        s_fac[kk] = (R0 > 0.0 && acc > 0.f) ? R0 * (double)acc / (R0 + (double)acc) : 0.0;
      } else {
        const int d = feat - 1;
        if constexpr (COV == GMM_COV_FULL) {
          for (int r = 0; r < tn; ++r) acc = fmaf(s_g[r * KC + kk], s_y[(r * KC + kk) * YS + d], acc);
        } else {
          const float c_d = s_mu[kk * D + d];
          for (int r = 0; r < tn; ++r) acc = fmaf(s_g[r * KC + kk], s_x[r * XS + d] - c_d, acc);
        }
        s_t1[kk * D + d] = acc;
      }
      tsum[s] = acc;
    }
    __syncthreads();
    // phase B: second moment about the tile mean, merged (Chan et al.)
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int f = threadIdx.x + s * kStatThreads;
      if (f >= kc * F) continue;
      const int kk = f / F, feat = f % F;
      if (feat <= D) continue;
      const float t0 = s_t0[kk];
      if (!(t0 > 0.f)) continue;
      int a, b;
      if constexpr (COV == GMM_COV_FULL) {
        const int e = feat - 1 - D;
        a = s_pair[2 * e];
        b = s_pair[2 * e + 1];
      } else {
        a = b = feat - 1 - D;
      }
      const float ma = s_t1[kk * D + a] / t0, mb = s_t1[kk * D + b] / t0;
      float m2 = 0.f;
      if constexpr (COV == GMM_COV_FULL) {
        for (int r = 0; r < tn; ++r) {
          const float* y = s_y + (r * KC + kk) * YS;
          m2 = fmaf(s_g[r * KC + kk], (y[a] - ma) * (y[b] - mb), m2);
        }
      } else {
        const float c_d = s_mu[kk * D + a];
        for (int r = 0; r < tn; ++r) {
          const float u = (s_x[r * XS + a] - c_d) - ma;
          m2 = fmaf(s_g[r * KC + kk], u * u, m2);
        }
      }
      // s_rm holds the running mean (S1 / S0) of the tiles merged so far
      const double fac = s_fac[kk];
      const double da = (double)ma - s_rm[kk * D + a];
      const double db = (double)mb - s_rm[kk * D + b];
      accd[s] += (double)m2 + da * db * fac;
    }
    __syncthreads();
    // phase C: running count and first moment
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int f = threadIdx.x + s * kStatThreads;
      if (f >= kc * F) continue;
      const int kk = f / F, feat = f % F;
      if (feat > D) continue;
      accd[s] += (double)tsum[s];
      if (feat == 0) s_r0[kk] = accd[s];
      else s_r1[kk * D + feat - 1] = accd[s];
    }
    __syncthreads();
    // running mean for the next tile's correction
    for (int i = threadIdx.x; i < kc * D; i += kStatThreads) {
      const double r0 = s_r0[i / D];
      s_rm[i] = r0 > 0.0 ? s_r1[i] / r0 : 0.0;
    }
  }
  // per-block partial [P][K][F]; with `accumulate` the block's sums are
  // merged into the partial already there (same pairwise rule)
  double* out = part + (size_t)blockIdx.y * K * F;
  __syncthreads();
  double outv[SLOTS];
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int f = threadIdx.x + s * kStatThreads;
    outv[s] = accd[s];
    if (f >= kc * F || !accumulate) continue;
    const int kk = f / F, feat = f % F;
    const double* o = out + (size_t)(k0 + kk) * F;
    if (feat <= D) {
      outv[s] = o[feat] + accd[s];
    } else {
      int a, b;
      if constexpr (COV == GMM_COV_FULL) {
        const int e = feat - 1 - D;
        a = s_pair[2 * e];
        b = s_pair[2 * e + 1];
      } else {
        a = b = feat - 1 - D;
      }
      const double S0o = o[0], S0n = s_r0[kk];
      double corr = 0.0;
      if (S0o > 0.0 && S0n > 0.0) {
        const double da = s_r1[kk * D + a] / S0n - o[1 + a] / S0o;
        const double db = s_r1[kk * D + b] / S0n - o[1 + b] / S0o;
        corr = da * db * (S0o * S0n / (S0o + S0n));
      }
      outv[s] = o[feat] + accd[s] + corr;
    }
  }
  __syncthreads();
#pragma unroll
  for (int s = 0; s < SLOTS; ++s) {
    const int f = threadIdx.x + s * kStatThreads;
    if (f >= kc * F) continue;
    const int kk = f / F, feat = f % F;
    out[(size_t)(k0 + kk) * F + feat] = outv[s];
  }
}

template <int D, int COV, int XT>
size_t lse_smem() {
  using S = LseShape<D, COV>;
  return sizeof(float) * (S::KC * D + S::KC * S::P + S::KC);
}

template <int D, int COV, int XT>
size_t stat_smem() {
  using SS = StatShape<D, COV>;
  constexpr int P = LseShape<D, COV>::P;
  size_t b = sizeof(double) * (size_t)SS::KC * (2 * D + 2);
  size_t f = (size_t)kStatTile * (D + 1) + kStatTile * SS::KC + SS::KC * D + SS::KC * P + SS::KC +
             SS::KC + SS::KC * D;
  if (COV == GMM_COV_FULL) f += (size_t)kStatTile * SS::KC * (D + 1);
  b += f * sizeof(float);
  if (COV == GMM_COV_FULL) b += sizeof(short) * 2 * (D * (D + 1) / 2);
  return b;
}

// grid 0: dense, one block per 128 points.  With a row list, `grid` blocks
// walk the list.
template <int D, int COV, int XT>
cudaError_t run_lse(const void* X, int64_t N, int K, const void* prepared, const PreparedLayout& L,
                    float* lse, double* ll_part, int m, int32_t* ids, float* gamma,
                    DeviceStatus* st, const uint32_t* rows, const uint32_t* row_count, int grid,
                    cudaStream_t s) {
  size_t smem = lse_smem<D, COV, XT>();
  auto kern = lse_kernel<D, COV, XT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int64_t blocks = rows ? grid : (N + kLseThreads - 1) / kLseThreads;
  kern<<<(unsigned)blocks, kLseThreads, smem, s>>>(X, N, K, prepared, L, lse, ll_part, m, ids,
                                                   gamma, st, rows, row_count);
  return cudaGetLastError();
}

template <int D, int COV, int XT>
cudaError_t run_stats(const void* X, int64_t N, int K, const void* prepared,
                      const PreparedLayout& L, const float* lse, int parts, double* part,
                      int accumulate, const uint32_t* rows, const uint32_t* row_count,
                      cudaStream_t s) {
  using SS = StatShape<D, COV>;
  size_t smem = stat_smem<D, COV, XT>();
  auto kern = stats_kernel<D, COV, XT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int64_t rpp = (N + parts - 1) / parts;
  rpp = (rpp + kStatTile - 1) / kStatTile * kStatTile;
  dim3 grid((K + SS::KC - 1) / SS::KC, parts);
  kern<<<grid, kStatThreads, smem, s>>>(X, N, K, prepared, L, lse, rpp, part, accumulate, rows,
                                        row_count);
  return cudaGetLastError();
}

}  // namespace simt

template <int V>
using IC = std::integral_constant<int, V>;

// Calls fn(IC<cov>, IC<xdtype>) for the runtime pair.
template <typename Fn>
cudaError_t dispatch_cx(int cov, int xt, Fn&& fn) {
  auto by_x = [&](auto Cc) -> cudaError_t {
    switch (xt) {
      case GMM_F32: return fn(Cc, IC<GMM_F32>{});
      case GMM_F16: return fn(Cc, IC<GMM_F16>{});
      default: return fn(Cc, IC<GMM_BF16>{});
    }
  };
  switch (cov) {
    case GMM_COV_FULL: return by_x(IC<GMM_COV_FULL>{});
    case GMM_COV_DIAG: return by_x(IC<GMM_COV_DIAG>{});
    default: return by_x(IC<GMM_COV_ISO>{});
  }
}

// One instantiation unit per D (simt_d*.cu) defines these two.
template <int D>
cudaError_t simt_lse_d(const void* X, int xdtype, int64_t N, int K, int cov, const void* prepared,
                       float* lse, double* ll_part, int m, int32_t* ids, float* gamma,
                       DeviceStatus* st, const uint32_t* rows, const uint32_t* row_count,
                       int grid, cudaStream_t s);
template <int D>
cudaError_t simt_stats_d(const void* X, int xdtype, int64_t N, int K, int cov,
                         const void* prepared, const float* lse, int parts, double* part,
                         int accumulate, const uint32_t* rows, const uint32_t* row_count,
                         cudaStream_t s);

}  // namespace gmm
