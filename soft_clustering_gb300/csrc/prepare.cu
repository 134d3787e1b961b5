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
  __shared__ int s_fail;
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
    if (threadIdx.x == 0) s_fail = 0;
    __syncthreads();
    for (int j = 0; j < D; ++j) {
      if (threadIdx.x == 0) {
        double p = A[j * D + j];
        if (!(p > 0.0) || !isfinite(p)) s_fail = 1;
        else A[j * D + j] = sqrt(p);
      }
      __syncthreads();
      if (s_fail) break;
      const double ljj = A[j * D + j];
      for (int i = j + 1 + threadIdx.x; i < D; i += blockDim.x) A[i * D + j] /= ljj;
      __syncthreads();
      const int m = D - j - 1;
      for (int idx = threadIdx.x; idx < m * m; idx += blockDim.x) {
        int i = j + 1 + idx / m, l = j + 1 + idx % m;
        if (l <= i) A[i * D + l] -= A[i * D + j] * A[l * D + j];
      }
      __syncthreads();
    }
    fail = s_fail;
    __syncthreads();
  }
  if (fail) flags |= GMM_FLAG_NOT_PD;
  float* W = at<float>(prepared, L.off_prec) + (size_t)k * D * D;
  double ld = 0.0;
  if (!fail) {
    for (int d = threadIdx.x; d < D; d += blockDim.x) ld += log(A[d * D + d]);
  }
  ld = block_sum(ld, red);
  // Column j of W = L^-1 by forward substitution of L w = e_j (one thread per column).
  for (int j = threadIdx.x; j < D; j += blockDim.x) {
    double wc[128];
    for (int i = 0; i < D; ++i) {
      if (fail || i < j) { wc[i] = 0.0; W[(size_t)i * D + j] = 0.0f; continue; }
      double s = (i == j) ? 1.0 : 0.0;
      for (int t = j; t < i; ++t) s -= A[i * D + t] * wc[t];
      wc[i] = s / A[i * D + i];
      W[(size_t)i * D + j] = (float)wc[i];
    }
  }
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    at<float>(prepared, L.off_mu)[(size_t)k * D + d] = mu[(size_t)k * D + d];
  if (threadIdx.x == 0) {
    double p = (double)pi[k];
    double c = (fail || !(p > 0.0)) ? -INFINITY : log(p) - ld - 0.5 * D * kLog2Pi;
    at<float>(prepared, L.off_c)[k] = (float)c;
    at<int32_t>(prepared, L.off_flags)[k] = flags;
    if (fail && st) raise_status(st, GMM_ERR_NOT_PD);
  }
}

// Screening operands for the tensor-core kernel (diagonal / isotropic, D = 64
// or 128), one block per component of the padded range [0, 128 * chunks).
// Row k of chunk k / 128 holds (b1, b2) = (mu w, -w / 2) divided by a power of
// two s_k chosen so max |b| / s_k <= 2^14 (no fp16 overflow whatever the
// variance), rounded to fp16 and stored in the 128-byte swizzled K-major
// layout the MMA reads.  The trailer keeps s_k, |(b1, b2)|_2 (for the
// rounding bound) and the screening bias c_k - (1/2) sum_d mu_d^2 w_d (the
// constant of the expanded form).  Components with bias -inf and padding rows
// get b = 0 and bias -inf.
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
  const double m = s_max;
  const double scale = m > 0.0 ? ldexp(1.0, (int)ceil(log2(m)) - 14) : 1.0;
  for (int j = threadIdx.x; j < KD; j += blockDim.x) {
    const __half h = __double2half(bval(j) / scale);
    *reinterpret_cast<__half*>(img + tc::sw128_offset(row, j, kTcChunk)) = h;
  }
  if (threadIdx.x == 0) {
    trail[row] = (float)scale;
    trail[kTcChunk + row] = (float)sqrt(red[31]);
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
