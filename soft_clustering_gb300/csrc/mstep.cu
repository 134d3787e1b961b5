// mstep.cu - deterministic reduction of the per-block statistics and the
// M-step, one thread block per component.
//
// "M-step kernel" of the low-precision GMM operator notes (sec. 3.1): block
// partial sums first, then a global reduction - here in fp64 over the
// partitions in a fixed order, so two runs give the same bits.  The update
// is the maximum-likelihood one from the sufficient statistics (Flash-GMM
// summary, Method: parameters updated directly from s0, s1, s2):
//   pi' = s0/N,  mu' = c + S1/s0,  Sigma' = S2/s0 - (S1/s0)(S1/s0)^T,
// where S1, S2 are the first and second moments about the centre c the
// statistics were accumulated around (the input mean), so the subtraction
// loses nothing to cancellation.
#include <math.h>

#include "gmm_internal.cuh"

namespace gmm {

namespace {

// part: [P][K][F] fp64.  centre: the mean the statistics are taken about
// (fp32 [K*D]).  Updates params in place.  dynamic smem: F doubles.
__global__ void mstep_kernel(const double* __restrict__ part, int parts, int64_t N, int D, int K,
                             int cov, const float* __restrict__ centre,
                             const int32_t* __restrict__ prep_flags, float var_floor,
                             float min_s0, float* pi, float* mu, float* covp,
                             int32_t* flags_out) {
  extern __shared__ double s[];
  const int k = blockIdx.x;
  const int F = stat_width(D, cov);
  for (int f = threadIdx.x; f < F; f += blockDim.x) {
    double acc = 0.0;
    for (int p = 0; p < parts; ++p) acc += part[((size_t)p * K + k) * F + f];
    s[f] = acc;
  }
  __syncthreads();
  const double s0 = s[0];
  const bool empty = !(s0 >= (double)min_s0) || !(s0 > 0.0);
  __shared__ int s_floor;
  if (threadIdx.x == 0) s_floor = 0;
  __syncthreads();
  int floored = 0;
  if (!empty) {
    const double inv = 1.0 / s0;
    const float* c = centre + (size_t)k * D;
    if (cov == GMM_COV_FULL) {
      float* S = covp + (size_t)k * D * D;
      // s layout: [s0 | S1 (D) | S2 lower triangle, row by row]
      for (int e = threadIdx.x; e < D * (D + 1) / 2; e += blockDim.x) {
        int a = (int)((sqrt(8.0 * e + 1.0) - 1.0) * 0.5);
        while ((a + 1) * (a + 2) / 2 <= e) ++a;
        while (a * (a + 1) / 2 > e) --a;
        const int b = e - a * (a + 1) / 2;
        const double da = s[1 + a] * inv, db = s[1 + b] * inv;
        double v = s[1 + D + e] * inv - da * db;
        if (a == b && v < (double)var_floor) { v = var_floor; floored = 1; }
        S[(size_t)a * D + b] = (float)v;
        S[(size_t)b * D + a] = (float)v;
      }
    } else if (cov == GMM_COV_DIAG) {
      for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const double dd = s[1 + d] * inv;
        double v = s[1 + D + d] * inv - dd * dd;
        if (v < (double)var_floor) { v = var_floor; floored = 1; }
        covp[(size_t)k * D + d] = (float)v;
      }
    } else if (threadIdx.x == 0) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) {
        const double dd = s[1 + d] * inv;
        acc += s[1 + D + d] * inv - dd * dd;
      }
      double v = acc / D;
      if (v < (double)var_floor) { v = var_floor; floored = 1; }
      covp[k] = (float)v;
    }
    __syncthreads();  // every thread has read mu (centre is the prepared copy)
    for (int d = threadIdx.x; d < D; d += blockDim.x)
      mu[(size_t)k * D + d] = (float)((double)c[d] + s[1 + d] * inv);
  }
  if (floored) atomicOr(&s_floor, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    pi[k] = (float)(s0 / (double)N);
    if (flags_out)
      flags_out[k] = prep_flags[k] | (s_floor ? GMM_FLAG_FLOOR : 0) | (empty ? GMM_FLAG_EMPTY : 0);
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
  size_t smem = sizeof(double) * stat_width(D, cov);
  cudaError_t e = cudaFuncSetAttribute(mstep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  mstep_kernel<<<K, 256, smem, s>>>(part, parts, N, D, K, cov, centre, prep_flags, var_floor,
                                    min_s0, p->pi, p->mu, p->cov, flags_out);
  return cudaGetLastError();
}

cudaError_t launch_ll_finalize(const double* ll_part, int64_t n, double* out, int accumulate,
                               cudaStream_t s) {
  ll_finalize_kernel<<<1, 1024, 0, s>>>(ll_part, n, out, accumulate);
  return cudaGetLastError();
}

}  // namespace gmm
