// noalloc.cu - gmm_em_step_noalloc: the EM step for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain scratch memory: code that runs inside
// another framework's allocator budget, plugins handed only their input and
// output buffers, or processes that must not call cudaMalloc once set up.
// For them the step's scratch (status word, prepared parameters,
// log-likelihood partials, per-block statistics, flags) lives in the
// file-scope device array below.  It is part of this library's device
// image, so every GPU that loads the library holds it until the process
// exits.  No call here allocates: no cudaMalloc, cudaFree or allocating
// library routine.
#include <stdio.h>


#include "gmm_internal.cuh"

namespace gmm {

cudaError_t launch_prepare(const gmm_params* p, int D, int K, int cov, float ridge_rel,
                           void* prepared, DeviceStatus* st, cudaStream_t s);
cudaError_t simt_lse(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                     const void* prepared, float* lse, double* ll_part, int m, int32_t* ids,
                     float* gamma, DeviceStatus* st, cudaStream_t s);
cudaError_t simt_stats(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                       const void* prepared, const float* lse, int parts, double* part,
                       int accumulate, cudaStream_t s);
cudaError_t launch_mstep(const double* part, int parts, int64_t N, int D, int K, int cov,
                         const float* centre, const int32_t* prep_flags, float var_floor,
                         float min_s0, gmm_params* p, int32_t* flags_out, cudaStream_t s);
cudaError_t launch_ll_finalize(const double* ll_part, int64_t n, double* out, int accumulate,
                               cudaStream_t s);
int stat_parts_for(int64_t N, int D, int K, int cov);

namespace {

// 64 MiB of scratch, shared by every call in the process.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch in the current context, looked up on
// every call (a cached address would outlive a device reset).
cudaError_t scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

struct ScratchLayout {
  size_t off_status, off_prep, off_llpart, off_ll, off_part, off_flags, bytes;
  int parts;
};

ScratchLayout scratch_layout(int64_t N, int D, int K, int cov) {
  ScratchLayout L;
  size_t o = 0;
  L.off_status = o; o = align_up(o + sizeof(DeviceStatus));
  L.off_prep = o;   o = align_up(o + PreparedLayout::make(D, K, cov).bytes);
  L.off_llpart = o; o = align_up(o + sizeof(double) * (size_t)((N + kLseRows - 1) / kLseRows));
  L.off_ll = o;     o = align_up(o + sizeof(double));
  L.parts = stat_parts_for(N, D, K, cov);
  L.off_part = o;   o = align_up(o + sizeof(double) * (size_t)L.parts * K * stat_width(D, cov));
  L.off_flags = o;  o = align_up(o + sizeof(int32_t) * K);
  L.bytes = o;
  return L;
}

gmm_status cuda_fail(cudaError_t e) {
  if (e == cudaSuccess) return GMM_OK;
  fprintf(stderr, "libgmm (gmm_em_step_noalloc): CUDA error %s\n", cudaGetErrorString(e));
  return GMM_ERR_CUDA;
}

}  // namespace
}  // namespace gmm

using namespace gmm;

extern "C" gmm_status gmm_em_step_noalloc(const void* X, gmm_dtype xdtype, int64_t N, int D,
                                          int K, gmm_params* params, gmm_cov_type cov,
                                          const gmm_opts* opts, double* loglik_dev,
                                          float* lse_dev, int32_t* flags_dev, void* stream) {
  if (!X || N < 1 || K < 1 || K > kMaxK || xdtype < GMM_F32 || xdtype > GMM_BF16 ||
      cov < GMM_COV_FULL || cov > GMM_COV_ISO)
    return GMM_ERR_INVALID_ARG;
  if (!(D == 16 || D == 32 || D == 64 || D == 128)) return D > 0 ? GMM_ERR_UNSUPPORTED : GMM_ERR_INVALID_ARG;
  if (!params || !params->pi || !params->mu || !params->cov || !loglik_dev || !lse_dev ||
      ((uintptr_t)X & 15))
    return GMM_ERR_INVALID_ARG;
  const ScratchLayout L = scratch_layout(N, D, K, cov);
  if (L.bytes > kNoAllocScratchBytes) {
    fprintf(stderr,
            "libgmm (gmm_em_step_noalloc): N=%lld D=%d K=%d needs %zu scratch bytes, more than "
            "the %zu built in; use gmm_em_step with a workspace\n",
            (long long)N, D, K, L.bytes, kNoAllocScratchBytes);
    return GMM_ERR_WORKSPACE;
  }
  void* base = nullptr;
  gmm_status r = cuda_fail(scratch_address(&base));
  if (r != GMM_OK) return r;
  const gmm_opts o = opts ? *opts : gmm_default_opts();
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus* st = at<DeviceStatus>(base, L.off_status);
  void* prep = at<char>(base, L.off_prep);
  double* llp = at<double>(base, L.off_llpart);
  double* ll = at<double>(base, L.off_ll);
  double* part = at<double>(base, L.off_part);
  const PreparedLayout PL = PreparedLayout::make(D, K, cov);
  // The status word must start at zero; every other region is fully written
  // by the kernel that produces it before it is read.
  if ((r = cuda_fail(cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s))) != GMM_OK) return r;
  if ((r = cuda_fail(launch_prepare(params, D, K, cov, o.ridge_rel, prep, st, s))) != GMM_OK) return r;
  if ((r = cuda_fail(simt_lse(X, xdtype, N, D, K, cov, prep, lse_dev, llp, 0, nullptr, nullptr,
                              st, s))) != GMM_OK)
    return r;
  if ((r = cuda_fail(launch_ll_finalize(llp, (N + kLseRows - 1) / kLseRows, ll, 0, s))) != GMM_OK) return r;
  if ((r = cuda_fail(simt_stats(X, xdtype, N, D, K, cov, prep, lse_dev, L.parts, part, 0, s))) !=
      GMM_OK)
    return r;
  if ((r = cuda_fail(launch_mstep(part, L.parts, N, D, K, cov, at<float>(prep, PL.off_mu),
                                  at<int32_t>(prep, PL.off_flags), o.var_floor, o.min_s0, params,
                                  flags_dev ? flags_dev : at<int32_t>(base, L.off_flags), s))) !=
      GMM_OK)
    return r;
  r = cuda_fail(cudaMemcpyAsync(loglik_dev, ll, sizeof(double), cudaMemcpyDeviceToDevice, s));
  if (r != GMM_OK) return r;
  // Device-side conditions (not positive definite, non-finite) are in the
  // status word; report them to the caller once this call's work is done.
  DeviceStatus h;
  if ((r = cuda_fail(cudaMemcpyAsync(&h, st, sizeof(int32_t) * 2, cudaMemcpyDeviceToHost, s))) !=
      GMM_OK)
    return r;
  if ((r = cuda_fail(cudaStreamSynchronize(s))) != GMM_OK) return r;
  return (gmm_status)h.code;
}
