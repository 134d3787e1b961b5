// prepare.cu - per-component preprocessing, one thread block per component.
//
// "Preprocess kernel" of the low-precision GMM operator notes (sec. 3.1):
// factorise the covariance once per EM iteration, all K components in
// parallel, and fold log|Sigma| and -(D/2) log 2pi into one constant so the
// distance step never repeats that work.  Positive-definiteness is checked
// here and repaired with a ridge (sec. 3.3, 4.1) so the distance kernels have
// no branch for it.
#include <math.h>

#include "gmm_internal.cuh"
#include "tc_ptx.cuh"

namespace gmm {

namespace {

constexpr double kLog2Pi = 1.8378770664093454835606594728112;

__device__ double block_sum(double v, double* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  double s = 0.0;
  for (int i = 0; i < nw; ++i) s += red[i];  // fixed order
  return s;
}

// Diagonal / isotropic: inverse variances and log-determinant.
__global__ void prepare_diag_kernel(const float* __restrict__ pi, const float* __restrict__ mu,
                                    const float* __restrict__ var, int D, int K, int nv,
                                    float ridge_rel, PreparedLayout L, void* prepared,
                                    DeviceStatus* st) {
  __shared__ double red[32];
  const int k = blockIdx.x;
  const float* v = var + (size_t)k * nv;
  double tr = 0.0;
  for (int d = threadIdx.x; d < nv; d += blockDim.x) tr += (double)v[d];
  tr = block_sum(tr, red);
  double add = (double)ridge_rel * tr / nv;
  int bad = 0;
  for (int d = threadIdx.x; d < nv; d += blockDim.x) {
    double w = (double)v[d] + add;
    if (!(w > 0.0) || !isfinite(w)) bad = 1;
  }
  bad = __syncthreads_or(bad);
  int flags = 0;
  if (bad) {
    flags |= GMM_FLAG_RIDGE;
    add += 1e-3 * tr / nv;
    bad = !(tr > 0.0);
    for (int d = threadIdx.x; d < nv; d += blockDim.x) {
      double w = (double)v[d] + add;
      if (!(w > 0.0) || !isfinite(w)) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (bad) flags |= GMM_FLAG_NOT_PD;
  }
  float* prec = at<float>(prepared, L.off_prec) + (size_t)k * nv;
  double ld = 0.0;
  for (int d = threadIdx.x; d < nv; d += blockDim.x) {
    double w = (double)v[d] + add;
    prec[d] = bad ? 0.0f : (float)(1.0 / w);
    ld += bad ? 0.0 : log(w);
  }
  ld = block_sum(ld, red);
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    at<float>(prepared, L.off_mu)[(size_t)k * D + d] = mu[(size_t)k * D + d];
  if (threadIdx.x == 0) {
    double logdet = nv == D ? ld : (double)D * ld;
    double p = (double)pi[k];
    double c = (bad || !(p > 0.0)) ? -INFINITY : log(p) - 0.5 * logdet - 0.5 * D * kLog2Pi;
    at<float>(prepared, L.off_c)[k] = (float)c;
    at<int32_t>(prepared, L.off_flags)[k] = flags;
    if (bad && st) raise_status(st, GMM_ERR_NOT_PD);
  }
}

// Full covariance: fp64 Cholesky in shared memory (right-looking), then the
// inverse factor W = L^-1 column by column.  dynamic smem: D*D doubles.
__global__ void prepare_full_kernel(const float* __restrict__ pi, const float* __restrict__ mu,
                                    const float* __restrict__ cov, int D, int K, float ridge_rel,
                                    PreparedLayout L, void* prepared, DeviceStatus* st) {
  extern __shared__ double A[];  // D*D
  __shared__ double red[32];
  __shared__ double s_rd[128];   // 1 / L_jj
  __shared__ double s_col[128];  // the column of W being formed
  const int k = blockIdx.x;
  const float* S = cov + (size_t)k * D * D;
  double tr = 0.0;
  for (int d = threadIdx.x; d < D; d += blockDim.x) tr += (double)S[(size_t)d * D + d];
  tr = block_sum(tr, red);
  double add = (double)ridge_rel * tr / D;
  int flags = 0;
  int fail = 1;
  for (int attempt = 0; attempt < 2 && fail; ++attempt) {
    if (attempt == 1) {
      flags |= GMM_FLAG_RIDGE;
      add += 1e-3 * tr / D;
      if (!(tr > 0.0)) break;
    }
    for (int i = threadIdx.x; i < D * D; i += blockDim.x)
      A[i] = (double)S[i] + ((i / D) == (i % D) ? add : 0.0);
    __syncthreads();
    int bad = 0;
    for (int j = 0; j < D; ++j) {
      // every thread reads the same pivot and takes its root and reciprocal
      const double p = A[j * D + j];
      if (!(p > 0.0) || !isfinite(p)) {
        bad = 1;
        break;
      }
      const double ljj = sqrt(p), rl = 1.0 / ljj;
      for (int i = j + 1 + threadIdx.x; i < D; i += blockDim.x) A[i * D + j] *= rl;
      __syncthreads();
      if (threadIdx.x == 0) A[j * D + j] = ljj;  // every thread has read the pivot
      // trailing update of the lower triangle, A[i][l] -= L[i][j] L[l][j] for
      // j < l <= i, spread evenly: rows j+1+pp and D-1-pp form a pair of
      // D-j elements in all, taken by four threads
      const int m = D - 1 - j, npairs = (m + 1) / 2;
      const int sub = threadIdx.x & 3;
      for (int pp = threadIdx.x >> 2; pp < npairs; pp += blockDim.x >> 2) {
        const int ia = j + 1 + pp, ib = D - 1 - pp;
        const int la = ia - j, tot = ia == ib ? la : la + (ib - j);
        const double lia = A[ia * D + j], lib = A[ib * D + j];
        for (int c = sub; c < tot; c += 4) {
          const bool ra = c < la;
          const int i = ra ? ia : ib, l = j + 1 + (ra ? c : c - la);
          A[i * D + l] = fma(-(ra ? lia : lib), A[l * D + j], A[i * D + l]);
        }
      }
      __syncthreads();
    }
    fail = bad;
    __syncthreads();
  }
  if (fail) flags |= GMM_FLAG_NOT_PD;
  float* W = at<float>(prepared, L.off_prec) + (size_t)k * D * D;
  double ld = 0.0;
  if (!fail) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) ld += log(A[d * D + d]);
  }
  ld = block_sum(ld, red);
  // W = L^-1 in place, columns from the last: with the trailing block
  // already inverted, W[i][j] = -(sum_{t=j+1..i} W[i][t] L[t][j]) / L[j][j].
  // Rows j+1+pp and D-1-pp form a pair, its dot products split over four
  // threads (terms sub, sub+4, ... of the pair's terms; partial sums
  // combined as (s0 + s1) + (s2 + s3)); every L[t][j] is read before column
  // j changes.
  if (!fail) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) s_rd[d] = 1.0 / A[d * D + d];
    __syncthreads();
    const int sub = threadIdx.x & 3;
    for (int j = D - 1; j >= 0; --j) {
      const double wjj = s_rd[j];
      const int m = D - 1 - j, npairs = (m + 1) / 2;
      for (int base = 0; base < npairs; base += blockDim.x >> 2) {
        const int pp = base + (threadIdx.x >> 2);
        double va = 0.0, vb = 0.0;
        int ia = 0, ib = 0;
        if (pp < npairs) {
          ia = j + 1 + pp;
          ib = D - 1 - pp;
          const int la = ia - j, tot = ia == ib ? la : la + (ib - j);
          for (int c = sub; c < tot; c += 4) {
            if (c < la) {
              const int t = j + 1 + c;
              va = fma(A[ia * D + t], A[t * D + j], va);
            } else {
              const int t = j + 1 + c - la;
              vb = fma(A[ib * D + t], A[t * D + j], vb);
            }
          }
        }
        va += __shfl_xor_sync(0xffffffffu, va, 1);
        vb += __shfl_xor_sync(0xffffffffu, vb, 1);
        va += __shfl_xor_sync(0xffffffffu, va, 2);
        vb += __shfl_xor_sync(0xffffffffu, vb, 2);
        if (pp < npairs) {
          if (sub == 0) s_col[ia] = -va * wjj;
          if (sub == 1 && ib != ia) s_col[ib] = -vb * wjj;
        }
      }
      __syncthreads();
      for (int i = j + 1 + threadIdx.x; i < D; i += blockDim.x) A[i * D + j] = s_col[i];
      if (threadIdx.x == 0) A[j * D + j] = wjj;
      __syncthreads();
    }
  }
  for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
    const int i = e / D, j = e % D;
    W[e] = (fail || j > i) ? 0.0f : (float)A[e];
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    at<float>(prepared, L.off_mu)[(size_t)k * D + d] = mu[(size_t)k * D + d];
  if (fc_tc_shape(D, K, GMM_COV_FULL)) {
    // the tensor-core screen's operands: s_k = 2^e with max |W| / s_k in
    // [2^14, 2^15), the B image of fp16(W32 / s_k) (W32 the fp32 W the exact
    // kernels use), b_k = W mu_k and the error-bound coefficients
    //   ex_k = 1.01 ((2^-11 + 2^-16) |W|_F + 2^-25 s_k D),  em_k = 1.01 2^-18 |W|_F |mu_k|
    // (fc_screen.cu derives them).
    double mx = 0.0, f2 = 0.0, m2 = 0.0;
    for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
      const int i = e / D, j = e % D;
      if (!fail && j <= i) {
        const double w = (double)(float)A[e];
        mx = fmax(mx, fabs(w));
        f2 += w * w;
      }
    }
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      const double m = (double)mu[(size_t)k * D + d];
      m2 += m * m;
    }
    __shared__ double s_mx[4];
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    if ((threadIdx.x & 31) == 0) s_mx[threadIdx.x >> 5] = mx;
    f2 = block_sum(f2, red);
    m2 = block_sum(m2, red);
    double M = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) M = fmax(M, s_mx[w]);
    int e2 = 0;
    frexp(M > 0.0 ? M : 1.0, &e2);  // M = f 2^e2, f in [0.5, 1)
    const float sk = (float)ldexp(1.0, e2 - 15);
    const float inv = 1.f / sk;
    float* T = at<float>(prepared, L.off_fcT);
    unsigned char* B = at<unsigned char>(prepared, L.off_fcB);
    if (threadIdx.x == 0) {
      const double F = sqrt(f2) * (1.0 + 1e-6), mun = sqrt(m2) * (1.0 + 1e-6);
      T[k] = sk;
      T[3 * kFcMaxK + k] = (float)(1.01 * 3.814697265625e-06 * F * mun);
      T[2 * kFcMaxK + k] =
          (float)(1.01 * ((0.00048828125 + 1.52587890625e-05) * F + 2.98023223876953125e-08 * sk * D));
    }
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
      double b = 0.0;
      if (!fail)
        for (int j = 0; j <= i; ++j) b += (double)(float)A[i * D + j] * (double)mu[(size_t)k * D + j];
      T[4 * kFcMaxK + k * D + i] = (float)b;
    }
    for (int u = threadIdx.x; u < D * 8; u += blockDim.x) {
      const int i = u >> 3, c = u & 7, n = k * D + i;
      __align__(16) __half h[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int j = 8 * c + t;
        h[t] = __float2half_rn(!fail && j < D && j <= i ? (float)A[i * D + j] * inv : 0.f);
      }
      *reinterpret_cast<uint4*>(B + (size_t)n * 128 + ((c ^ (n & 7)) << 4)) =
          *reinterpret_cast<const uint4*>(h);
    }
  }
  if (threadIdx.x == 0) {
    double p = (double)pi[k];
    double c = (fail || !(p > 0.0)) ? -INFINITY : log(p) - ld - 0.5 * D * kLog2Pi;
    if (fc_tc_shape(D, K, GMM_COV_FULL)) at<float>(prepared, L.off_fcT)[kFcMaxK + k] = (float)c;
    at<float>(prepared, L.off_c)[k] = (float)c;
    at<int32_t>(prepared, L.off_flags)[k] = flags;
    if (fail && st) raise_status(st, GMM_ERR_NOT_PD);
  }
}

// fp16 at or above v >= 0 (round up).
__device__ __forceinline__ __half half_ru(double v) {
  __half h = __double2half(v);
  if ((double)__half2float(h) < v) h = __ushort_as_half((unsigned short)(__half_as_ushort(h) + 1));
  return h;
}

// Margin of the folded screening per unit of row norm: the fp16 rounding of
// both operands (3 x 2^-11) and the tensor-core accumulation allowance
// (3.5e-5 of sum |a b|), with 1e-4 relative for the accumulation error of
// the margin terms themselves and 2e-6 spare.
constexpr double kFoldKappa = 1.5e-3 * 1.0001 + 2e-6;

// Folded operands, part 0: one block of 128 threads per component of the
// padded range: max |b|, |b|^2 and sum mu^2 w in fp64, staged (3 doubles per
// component) in the chunk's extra-row region, which part 1 overwrites.
__global__ void __launch_bounds__(kTcChunk) prepare_fold_sums_kernel(PreparedLayout L,
                                                                     void* prepared) {
  __shared__ double red[3][kTcChunk / 32];
  const int k = blockIdx.x, chunk = k / kTcChunk, row = k % kTcChunk;
  const int D = L.D, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool live = k < L.K && at<float>(prepared, L.off_c)[k] != -INFINITY;
  double mx = 0.0, n2 = 0.0, q = 0.0;
  if (live) {
    const float* mu = at<float>(prepared, L.off_mu) + (size_t)k * D;
    const float* prec = at<float>(prepared, L.off_prec) + (size_t)k * (L.cov == GMM_COV_DIAG ? D : 1);
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      const double w = (double)prec[L.cov == GMM_COV_DIAG ? d : 0];
      const double b1 = (double)mu[d] * w, b2 = -0.5 * w;
      mx = fmax(mx, fmax(fabs(b1), fabs(b2)));
      n2 += b1 * b1 + b2 * b2;
      q += (double)mu[d] * b1;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    q += __shfl_xor_sync(0xffffffffu, q, o);
  }
  if (lane == 0) { red[0][wid] = mx; red[1][wid] = n2; red[2][wid] = q; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double m = 0.0, a2 = 0.0, qq = 0.0;
    for (int i = 0; i < kTcChunk / 32; ++i) { m = fmax(m, red[0][i]); a2 += red[1][i]; qq += red[2][i]; }
    double* stage = reinterpret_cast<double*>(at<unsigned char>(prepared, L.off_tcB) +
                                              (size_t)chunk * L.tcB_chunk_bytes +
                                              (size_t)kTcChunk * 2 * D * 2) + 3 * row;
    stage[0] = m;
    stage[1] = a2;
    stage[2] = qq;
  }
}

// Folded operands, part 1: one block of 128 threads per chunk, thread t for
// component k = 128 chunk + t, from the sums part 0 staged.  Picks the
// chunk's scale S, a power of two with max |b| / S <= 2^14, |bias| / S <=
// 2^25 and max d_k / S <= 2^15 (no fp16 overflow in either step), and writes
// the extra K = 16 row of B, the margins u_k and d_k and the trailer scalars
// (see tc_fold).  d_k covers the 1e-3 + 1e-6 |bias| gap between the expanded
// form and the exact fp32 log-density, the accumulation allowance on the bias
// terms (3.6e-5 |bias|) and the residual of the bias split.  Dead and padding
// components get bias part -inf and zero margins.
__global__ void __launch_bounds__(kTcChunk) prepare_fold_scale_kernel(PreparedLayout L,
                                                                      void* prepared) {
  __shared__ double red[3][kTcChunk / 32];
  __shared__ double sS;
  const int chunk = blockIdx.x, t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int D = L.D;
  const float* cvec = at<float>(prepared, L.off_c);
  const double* stage = reinterpret_cast<const double*>(
      at<unsigned char>(prepared, L.off_tcB) + (size_t)chunk * L.tcB_chunk_bytes +
      (size_t)kTcChunk * 2 * D * 2);
  const double s_mx = stage[3 * t], s_n2 = stage[3 * t + 1], s_q = stage[3 * t + 2];
  __syncthreads();  // every thread has read its sums before the region is rewritten

  const int k = chunk * kTcChunk + t;
  const bool live = k < L.K && cvec[k] != -INFINITY;
  const double bias = live ? (double)cvec[k] - 0.5 * s_q : 0.0;
  // the d_k bound before the split residual (which is below 1e-7 |bias|)
  const double dpre = live ? 1.0001 * (1e-3 + 3.72e-5 * fabs(bias)) : 0.0;
  double m0 = s_mx, m1 = fabs(bias), m2 = dpre;
  for (int o = 16; o > 0; o >>= 1) {
    m0 = fmax(m0, __shfl_xor_sync(0xffffffffu, m0, o));
    m1 = fmax(m1, __shfl_xor_sync(0xffffffffu, m1, o));
    m2 = fmax(m2, __shfl_xor_sync(0xffffffffu, m2, o));
  }
  if (lane == 0) { red[0][wid] = m0; red[1][wid] = m1; red[2][wid] = m2; }
  __syncthreads();
  if (t == 0) {
    double M = 0.0, B = 0.0, Dm = 0.0;
    for (int i = 0; i < kTcChunk / 32; ++i) {
      M = fmax(M, red[0][i]); B = fmax(B, red[1][i]); Dm = fmax(Dm, red[2][i]);
    }
    int e = -1000;
    if (M > 0.0) e = max(e, (int)ceil(log2(M)) - 14);
    if (B > 0.0) e = max(e, (int)ceil(log2(B)) - 25);
    if (Dm > 0.0) e = max(e, (int)ceil(log2(Dm)) - 15);
    if (e == -1000) e = 0;
    sS = ldexp(1.0, e);
  }
  __syncthreads();
  const double S = sS;
  // bias / S = 2^10 b1 + b2 + 2^-10 b3 (fp16 parts), residual r3
  __half p1 = __ushort_as_half((unsigned short)0xFC00), p2 = __double2half(0.0), p3 = p2;
  double r3 = 0.0;
  if (live) {
    const double beta = bias / S;
    p1 = __double2half(beta * 0x1p-10);
    const double r1 = beta - (double)__half2float(p1) * 0x1p10;
    p2 = __double2half(r1);
    const double r2 = r1 - (double)__half2float(p2);
    p3 = __double2half(r2 * 0x1p10);
    r3 = r2 - (double)__half2float(p3) * 0x1p-10;
  }
  const double u = live ? kFoldKappa * sqrt(s_n2) + 0x1p-20 * S : 0.0;
  const double dk = live ? dpre + 1.0001 * 1.01 * fabs(r3) * S : 0.0;
  unsigned char* img = at<unsigned char>(prepared, L.off_tcB) + (size_t)chunk * L.tcB_chunk_bytes +
                       (size_t)kTcChunk * 2 * D * 2;
  const __half zero = __double2half(0.0);
  for (int e = 0; e < kTcExtraK; ++e) {
    __half h = zero;
    if (e == 0) h = p1;
    else if (e == 1) h = p2;
    else if (e == 2) h = p3;
    else if (e == 3 && live) h = half_ru(u * 16.0 / S);
    else if (e == 4 && live) h = half_ru(dk / S);
    *reinterpret_cast<__half*>(img + tc::k16_offset(t, e)) = h;
  }
  float* trail = at<float>(prepared, L.off_tcT) + (size_t)chunk * kTcTrail;
  const float uf = __double2float_ru(u), df = __double2float_ru(dk);
  trail[t] = uf;
  trail[kTcChunk + t] = df;
  // chunk maxima of the margins (for the assignment's m-th lower bound)
  float a0 = uf, a1 = df;
  for (int o = 16; o > 0; o >>= 1) {
    a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, o));
    a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, o));
  }
  __syncthreads();  // red is read above before reuse
  if (lane == 0) { red[0][wid] = a0; red[1][wid] = a1; }
  __syncthreads();
  if (t == 0) {
    float U = 0.f, Dm = 0.f;
    for (int i = 0; i < kTcChunk / 32; ++i) { U = fmaxf(U, (float)red[0][i]); Dm = fmaxf(Dm, (float)red[1][i]); }
    trail[kFoldS] = (float)S;
    trail[kFoldInvS] = (float)(1.0 / S);
    trail[kFoldUMax] = U;
    trail[kFoldDMax] = Dm;
  }
}

// Streamed chunks (more than kTcFoldChunks): one block of 128 threads per
// chunk picks the chunk's common scale S, the smallest power of two with
// max |b| / S <= 2^14 over its components (fp32 maxima: a relative error
// of 2^-23 cannot overflow fp16), and writes it to every scale slot of the
// chunk's trailer.
__global__ void __launch_bounds__(kTcChunk) prepare_stream_scale_kernel(PreparedLayout L,
                                                                        void* prepared) {
  __shared__ float red[kTcChunk / 32];
  __shared__ float sS;
  const int chunk = blockIdx.x, t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int k = chunk * kTcChunk + t, D = L.D;
  const bool live = k < L.K && at<float>(prepared, L.off_c)[k] != -INFINITY;
  float mx = 0.f;
  if (live) {
    const float* mu = at<float>(prepared, L.off_mu) + (size_t)k * D;
    const float* prec = at<float>(prepared, L.off_prec) + (size_t)k * (L.cov == GMM_COV_DIAG ? D : 1);
    for (int d = 0; d < D; ++d) {
      const float w = prec[L.cov == GMM_COV_DIAG ? d : 0];
      mx = fmaxf(mx, fmaxf(fabsf(mu[d] * w), 0.5f * fabsf(w)));
    }
  }
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red[wid] = mx;
  __syncthreads();
  if (t == 0) {
    float M = 0.f;
    for (int i = 0; i < kTcChunk / 32; ++i) M = fmaxf(M, red[i]);
    sS = M > 0.f ? ldexpf(1.f, (int)ceilf(log2f(M)) - 14) : 1.f;
  }
  __syncthreads();
  at<float>(prepared, L.off_tcT)[(size_t)chunk * kTcTrail + t] = sS;
}

// Screening operands for the tensor-core kernel (diagonal / isotropic, D = 64
// or 128), one block per component of the padded range [0, 128 * chunks).
// Row k of chunk k / 128 holds (b1, b2) = (mu w, -w / 2) divided by a power of
// two s_k chosen so max |b| / s_k <= 2^14 (no fp16 overflow whatever the
// variance), rounded to fp16 and stored in the 128-byte swizzled K-major
// layout the MMA reads.  The trailer keeps s_k, |(b1, b2)|_2 (for the
// rounding bound) and the screening bias c_k - (1/2) sum_d mu_d^2 w_d (the
// constant of the expanded form).  Components with bias -inf and padding rows
// get b = 0 and bias -inf.  Folded chunks (tc_fold) divide by the chunk's
// common scale instead, and their trailer comes from
// prepare_fold_scale_kernel.
__global__ void prepare_tc_kernel(PreparedLayout L, void* prepared) {
  __shared__ double red[32];
  __shared__ double s_max;
  const int k = blockIdx.x;
  const int D = L.D, KD = 2 * D;
  const int chunk = k / kTcChunk, row = k % kTcChunk;
  unsigned char* img = at<unsigned char>(prepared, L.off_tcB) + (size_t)chunk * L.tcB_chunk_bytes;
  float* trail = at<float>(prepared, L.off_tcT) + (size_t)chunk * kTcTrail;
  const bool live = k < L.K && at<float>(prepared, L.off_c)[k] != -INFINITY;
  const float* mu = at<float>(prepared, L.off_mu) + (size_t)(live ? k : 0) * D;
  const float* prec = at<float>(prepared, L.off_prec) +
                      (size_t)(live ? k : 0) * (L.cov == GMM_COV_DIAG ? D : 1);
  auto bval = [&](int j) -> double {
    if (!live) return 0.0;
    const int d = j < D ? j : j - D;
    const double w = (double)prec[L.cov == GMM_COV_DIAG ? d : 0];
    return j < D ? (double)mu[d] * w : -0.5 * w;
  };
  double mx = 0.0, n2 = 0.0, q = 0.0;
  for (int j = threadIdx.x; j < KD; j += blockDim.x) {
    const double b = bval(j);
    mx = fmax(mx, fabs(b));
    n2 += b * b;
    if (j < D && live) q += (double)mu[j] * b;  // mu^2 w
  }
  // block max and sums (fixed order)
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    n2 += __shfl_xor_sync(0xffffffffu, n2, o);
    q += __shfl_xor_sync(0xffffffffu, q, o);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __shared__ double s_q;
  if (lane == 0) { red[wid] = mx; red[8 + wid] = n2; red[16 + wid] = q; }
  __syncthreads();
  if (threadIdx.x == 0) {
    double m = 0.0, s = 0.0, qq = 0.0;
    for (int i = 0; i < nw; ++i) { m = fmax(m, red[i]); s += red[8 + i]; qq += red[16 + i]; }
    s_max = m;
    red[31] = s;
    s_q = qq;
  }
  __syncthreads();
  // folded: the chunk's common scale (written by prepare_fold_scale_kernel)
  // the chunk's common scale (written by prepare_fold_scale_kernel or
  // prepare_stream_scale_kernel)
  const bool fold = tc_fold(L.tc_chunks);
  const double scale = fold ? (double)trail[kFoldS] : (double)trail[row];
  for (int j = threadIdx.x; j < KD; j += blockDim.x) {
    const __half h = __double2half(bval(j) / scale);
    *reinterpret_cast<__half*>(img + tc::sw128_offset(row, j, kTcChunk)) = h;
  }
  if (threadIdx.x == 0 && !fold) {
    trail[row] = (float)scale;
    // |(b1, b2)| plus a floor for the operands that the common scale leaves
    // fp16-subnormal (2^-25 S each, at most 2^-21 S |a| in all, which
    // kappa |a| (2^-20 S / 1.5e-3) covers)
    trail[kTcChunk + row] = __double2float_ru(sqrt(red[31]) + 0x1p-20 * scale / 1.5e-3);
    // bias = c_k - sum mu^2 w / 2, with the margin of the fp32 evaluation
    // (1e-3 absolute + 1e-6 relative), rounded outwards
    const double bias = live ? (double)at<float>(prepared, L.off_c)[k] - 0.5 * s_q : 0.0;
    const double dl = 1e-3 + 1e-6 * fabs(bias);
    trail[2 * kTcChunk + row] = live ? __double2float_rd(bias - dl) : -INFINITY;
    trail[3 * kTcChunk + row] = live ? __double2float_ru(bias + dl) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_prepare_tc(int D, int K, int cov, void* prepared, cudaStream_t s) {
  PreparedLayout L = PreparedLayout::make(D, K, cov);
  if (!L.tc_chunks) return cudaSuccess;
  if (tc_fold(L.tc_chunks)) {
    prepare_fold_sums_kernel<<<L.tc_chunks * kTcChunk, kTcChunk, 0, s>>>(L, prepared);
    cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
    prepare_fold_scale_kernel<<<L.tc_chunks, kTcChunk, 0, s>>>(L, prepared);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else {
    prepare_stream_scale_kernel<<<L.tc_chunks, kTcChunk, 0, s>>>(L, prepared);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  prepare_tc_kernel<<<L.tc_chunks * kTcChunk, 128, 0, s>>>(L, prepared);
  return cudaGetLastError();
}

cudaError_t launch_prepare(const gmm_params* p, int D, int K, int cov, float ridge_rel,
                           void* prepared, DeviceStatus* st, cudaStream_t s) {
  PreparedLayout L = PreparedLayout::make(D, K, cov);
  if (cov == GMM_COV_FULL) {
    size_t smem = sizeof(double) * (size_t)D * D;
    cudaError_t e = cudaFuncSetAttribute(prepare_full_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prepare_full_kernel<<<K, 128, smem, s>>>(p->pi, p->mu, p->cov, D, K, ridge_rel, L, prepared,
                                            st);
  } else {
    int nv = cov == GMM_COV_DIAG ? D : 1;
    prepare_diag_kernel<<<K, 128, 0, s>>>(p->pi, p->mu, p->cov, D, K, nv, ridge_rel, L, prepared,
                                          st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_prepare_tc(D, K, cov, prepared, s);
  }
  return cudaGetLastError();
}

}  // namespace gmm
