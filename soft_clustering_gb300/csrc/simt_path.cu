// simt_path.cu - entry points of the fp32 CUDA-core path, dispatching on D
// to the per-D instantiation units (kernels in simt_kernels.cuh).
#include "simt_kernels.cuh"

namespace gmm {

int simt_stat_chunk(int D, int cov) {
  switch (D) {
    case 16: return cov == GMM_COV_FULL ? simt::StatShape<16, GMM_COV_FULL>::KC : simt::StatShape<16, GMM_COV_DIAG>::KC;
    case 32: return cov == GMM_COV_FULL ? simt::StatShape<32, GMM_COV_FULL>::KC : simt::StatShape<32, GMM_COV_DIAG>::KC;
    case 64: return cov == GMM_COV_FULL ? simt::StatShape<64, GMM_COV_FULL>::KC : simt::StatShape<64, GMM_COV_DIAG>::KC;
    default: return cov == GMM_COV_FULL ? simt::StatShape<128, GMM_COV_FULL>::KC : simt::StatShape<128, GMM_COV_DIAG>::KC;
  }
}

cudaError_t simt_lse_rows(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                          const void* prepared, float* lse, double* ll_part, int m, int32_t* ids,
                          float* gamma, DeviceStatus* st, const uint32_t* rows,
                          const uint32_t* row_count, int grid, cudaStream_t s) {
  switch (D) {
    case 16: return simt_lse_d<16>(X, xdtype, N, K, cov, prepared, lse, ll_part, m, ids, gamma, st, rows, row_count, grid, s);
    case 32: return simt_lse_d<32>(X, xdtype, N, K, cov, prepared, lse, ll_part, m, ids, gamma, st, rows, row_count, grid, s);
    case 64: return simt_lse_d<64>(X, xdtype, N, K, cov, prepared, lse, ll_part, m, ids, gamma, st, rows, row_count, grid, s);
    case 128: return simt_lse_d<128>(X, xdtype, N, K, cov, prepared, lse, ll_part, m, ids, gamma, st, rows, row_count, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t simt_lse(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                     const void* prepared, float* lse, double* ll_part, int m, int32_t* ids,
                     float* gamma, DeviceStatus* st, cudaStream_t s) {
  return simt_lse_rows(X, xdtype, N, D, K, cov, prepared, lse, ll_part, m, ids, gamma, st,
                       nullptr, nullptr, 0, s);
}

// With a row list, the points rows[0 .. *row_count) (count read on the device).
cudaError_t simt_stats_rows(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                            const void* prepared, const float* lse, int parts, double* part,
                            int accumulate, const uint32_t* rows, const uint32_t* row_count,
                            cudaStream_t s) {
  switch (D) {
    case 16: return simt_stats_d<16>(X, xdtype, N, K, cov, prepared, lse, parts, part, accumulate, rows, row_count, s);
    case 32: return simt_stats_d<32>(X, xdtype, N, K, cov, prepared, lse, parts, part, accumulate, rows, row_count, s);
    case 64: return simt_stats_d<64>(X, xdtype, N, K, cov, prepared, lse, parts, part, accumulate, rows, row_count, s);
    case 128: return simt_stats_d<128>(X, xdtype, N, K, cov, prepared, lse, parts, part, accumulate, rows, row_count, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t simt_stats(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                       const void* prepared, const float* lse, int parts, double* part,
                       int accumulate, cudaStream_t s) {
  return simt_stats_rows(X, xdtype, N, D, K, cov, prepared, lse, parts, part, accumulate,
                         nullptr, nullptr, s);
}

}  // namespace gmm
