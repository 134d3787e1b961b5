// mstep.cu - deterministic reduction of the per-block statistics and the
// M-step, one thread block per component.
//
// "M-step kernel" of the low-precision GMM operator notes (sec. 3.1): block
// partial sums first, then a global reduction - here in fp64 over the
// partitions in a fixed order, so two runs give the same bits.  The update
// is the maximum-likelihood one from the sufficient statistics (Flash-GMM
// summary, Method: parameters updated directly from s0, s1, s2):
//   pi' = s0/N,  mu' = c + S1/s0,  Sigma' = M2/s0,
// where S1 is the first moment about the centre c the statistics were taken
// around (the input mean) and M2 the second moment about the weighted mean
// itself, so no large moments cancel.
#include <math.h>

#include "gmm_internal.cuh"

namespace gmm {

namespace {

// part: [P][K][F] fp64, each partial [S0 | S1 about the centre c | M2 about
// the partial's own mean].  The partials are merged in partition order:
// S0 and S1 are summed; M2 = sum_p [M2_p + S0_p (m_p - m)(m_p - m)^T] with
// m_p = S1_p / S0_p and m = S1 / S0 (the pairwise update of Chan, Golub and
// LeVeque, applied to all partitions at once).  centre: the mean the
// statistics were taken about (fp32 [K*D]).  Updates params in place.
// Grid (K, Y): block (k, y) takes the second-moment entries [y B, (y + 1) B)
// of component k (B = blockDim.x, one entry a thread; Y = 1 for diagonal and
// isotropic covariance), every block of k the same sums S0, S1.  Block y = 0
// writes pi and mu; flags_out (zeroed by the launcher) collects every
// block's flags by OR.  dynamic smem: (1 + D) + parts doubles.
__global__ void mstep_kernel(const double* __restrict__ part, int parts, int64_t N, int D, int K,
                             int cov, const float* __restrict__ centre,
                             const int32_t* __restrict__ prep_flags, float var_floor,
                             float min_s0, float* pi, float* mu, float* covp,
                             int32_t* flags_out) {
  extern __shared__ double s[];
  double* inv0 = s + 1 + D;  // 1 / S0_p (0 where S0_p = 0)
  const int k = blockIdx.x, y = blockIdx.y;
  const int F = stat_width(D, cov);
  auto P_ = [&](int p, int f) { return part[((size_t)p * K + k) * F + f]; };
  for (int f = threadIdx.x; f <= D; f += blockDim.x) {
    double acc = 0.0;
    for (int p = 0; p < parts; ++p) acc += P_(p, f);
    s[f] = acc;
  }
  for (int p = threadIdx.x; p < parts; p += blockDim.x) {
    const double c0 = P_(p, 0);
    inv0[p] = c0 > 0.0 ? 1.0 / c0 : 0.0;
  }
  __syncthreads();
  const double s0 = s[0];
  const bool empty = !(s0 >= (double)min_s0) || !(s0 > 0.0);
  const int nm2 = cov == GMM_COV_FULL ? D * (D + 1) / 2 : D;
  __shared__ int s_floor;
  if (threadIdx.x == 0) s_floor = 0;
  // this thread's entry (full: e enumerates the lower triangle row by row)
  const int e = y * blockDim.x + threadIdx.x;
  int a = e, b = e;
  if (cov == GMM_COV_FULL && e < nm2) {
    a = (int)((sqrt(8.0 * e + 1.0) - 1.0) * 0.5);
    while ((a + 1) * (a + 2) / 2 <= e) ++a;
    while (a * (a + 1) / 2 > e) --a;
    b = e - a * (a + 1) / 2;
  }
  double m2 = 0.0;
  if (e < nm2 && s0 > 0.0) {
    const double ma = s[1 + a] / s0, mb = s[1 + b] / s0;
    for (int p = 0; p < parts; ++p) {
      const double c0 = P_(p, 0);
      m2 += P_(p, 1 + D + e);
      if (c0 > 0.0) m2 += c0 * (P_(p, 1 + a) * inv0[p] - ma) * (P_(p, 1 + b) * inv0[p] - mb);
    }
  }
  __syncthreads();
  int floored = 0;
  if (cov == GMM_COV_ISO) {
    // one block (D <= blockDim): the mean of the diagonal
    if (e < nm2) inv0[e] = m2;  // the partition reciprocals are no longer read
    __syncthreads();
    if (!empty && threadIdx.x == 0) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += inv0[d];
      double v = acc / s0 / D;
      if (v < (double)var_floor) { v = var_floor; floored = 1; }
      covp[k] = (float)v;
    }
  } else if (!empty && e < nm2) {
    double v = m2 / s0;
    if (a == b && v < (double)var_floor) { v = var_floor; floored = 1; }
    if (cov == GMM_COV_FULL) {
      float* S = covp + (size_t)k * D * D;
      S[(size_t)a * D + b] = (float)v;
      S[(size_t)b * D + a] = (float)v;
    } else {
      covp[(size_t)k * D + e] = (float)v;
    }
  }
  if (y == 0 && !empty) {
    const double inv = 1.0 / s0;
    const float* c = centre + (size_t)k * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x)
      mu[(size_t)k * D + d] = (float)((double)c[d] + s[1 + d] * inv);
  }
  if (floored) atomicOr(&s_floor, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    if (y == 0) pi[k] = (float)(s0 / (double)N);
    if (flags_out)
      atomicOr(flags_out + k,
               prep_flags[k] | (s_floor ? GMM_FLAG_FLOOR : 0) | (empty ? GMM_FLAG_EMPTY : 0));
  }
}

// Sum of the per-block log-likelihood partials in a fixed order.
__global__ void ll_finalize_kernel(const double* __restrict__ ll_part, int64_t n,
                                   double* __restrict__ out, int accumulate) {
  __shared__ double red[1024 / 32];
  double acc = 0.0;
  // contiguous slice per thread, slices summed in thread order
  const int64_t per = (n + blockDim.x - 1) / blockDim.x;
  const int64_t b = threadIdx.x * per, e = min(n, b + per);
  for (int64_t i = b; i < e; ++i) acc += ll_part[i];
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    *out = accumulate ? *out + s : s;
  }
}

}  // namespace

cudaError_t launch_mstep(const double* part, int parts, int64_t N, int D, int K, int cov,
                         const float* centre, const int32_t* prep_flags, float var_floor,
                         float min_s0, gmm_params* p, int32_t* flags_out, cudaStream_t s) {
  constexpr int kThreads = 256;
  const int nm2 = cov == GMM_COV_FULL ? D * (D + 1) / 2 : D;
  const int ny = cov == GMM_COV_FULL ? (nm2 + kThreads - 1) / kThreads : 1;
  const size_t smem = sizeof(double) * ((size_t)1 + D + (parts > D ? parts : D));
  cudaError_t e = cudaFuncSetAttribute(mstep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  if (flags_out && (e = cudaMemsetAsync(flags_out, 0, sizeof(int32_t) * K, s)) != cudaSuccess)
    return e;
  mstep_kernel<<<dim3(K, ny), kThreads, smem, s>>>(part, parts, N, D, K, cov, centre, prep_flags,
                                                   var_floor, min_s0, p->pi, p->mu, p->cov,
                                                   flags_out);
  return cudaGetLastError();
}

cudaError_t launch_ll_finalize(const double* ll_part, int64_t n, double* out, int accumulate,
                               cudaStream_t s) {
  ll_finalize_kernel<<<1, 1024, 0, s>>>(ll_part, n, out, accumulate);
  return cudaGetLastError();
}

}  // namespace gmm
