// simt_d32.cu - instantiations of the fp32 CUDA-core path for D = 32.
#include "simt_kernels.cuh"

namespace gmm {

template <>
cudaError_t simt_lse_d<32>(const void* X, int xdtype, int64_t N, int K, int cov,
                          const void* prepared, float* lse, double* ll_part, int m, int32_t* ids,
                          float* gamma, DeviceStatus* st, const uint32_t* rows,
                          const uint32_t* row_count, int grid, cudaStream_t s) {
  PreparedLayout L = PreparedLayout::make(32, K, cov);
  return dispatch_cx(cov, xdtype, [&](auto Cc, auto Xc) {
    return simt::run_lse<32, decltype(Cc)::value, decltype(Xc)::value>(
        X, N, K, prepared, L, lse, ll_part, m, ids, gamma, st, rows, row_count, grid, s);
  });
}

template <>
cudaError_t simt_stats_d<32>(const void* X, int xdtype, int64_t N, int K, int cov,
                            const void* prepared, const float* lse, int parts, double* part,
                            int accumulate, const uint32_t* rows,
                            const uint32_t* row_count, cudaStream_t s) {
  PreparedLayout L = PreparedLayout::make(32, K, cov);
  return dispatch_cx(cov, xdtype, [&](auto Cc, auto Xc) {
    return simt::run_stats<32, decltype(Cc)::value, decltype(Xc)::value>(
        X, N, K, prepared, L, lse, parts, part, accumulate, rows, row_count, s);
  });
}

}  // namespace gmm
