/*
 * gen_cuda.cu - device side of the seeded synthetic-mixture generator.
 *
 * Draws points straight into device memory with the same gen_point() the
 * host runs (mixture_gen.h), so large data sets never cross the host link and
 * any point can still be regenerated on the host by index.  Built with
 * -fmad=false: fused multiply-adds would change the bits.
 */
#include <cuda_runtime.h>

#include "mixture_gen.h"

namespace {

__global__ void __launch_bounds__(128) gen_points_kernel(gen_mixture m, uint64_t start,
                                                         uint64_t count, int dtype, void* out) {
  double scratch[128];
  const size_t esz = dtype == GEN_F32 ? 4 : 2;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (uint64_t)gridDim.x * blockDim.x) {
    gen_point(&m, start + i, dtype, (char*)out + (size_t)i * m.D * esz, scratch);
  }
}

}  // namespace

/* Draw points [start, start+count) into out_dev (row-major, dtype GEN_*).
 * Table pointers are device addresses.  D must be even and <= 128.
 * Returns 0, 1 for a bad argument, 2 for a launch error.  Asynchronous on
 * `stream` (a cudaStream_t, NULL for the default stream). */
extern "C" int gen_device_points(int kind, int D, int K, uint64_t seed, double noise,
                                 double mid_frac, const double* cdf, const double* mu,
                                 const double* sd, const double* chol, uint64_t start,
                                 uint64_t count, int dtype, void* out_dev, void* stream) {
  if (D <= 0 || D > 128 || (D & 1) || K <= 0 || !out_dev || !cdf || !mu) return 1;
  if ((kind == GEN_MIX_DIAG || kind == GEN_MIX_IVF) && !sd) return 1;
  if (kind == GEN_MIX_FULL && !chol) return 1;
  if (count == 0) return 0;
  gen_mixture m;
  m.kind = kind;
  m.D = D;
  m.K = K;
  m.seed = seed;
  m.noise = noise;
  m.mid_frac = mid_frac;
  m.cdf = cdf;
  m.mu = mu;
  m.sd = sd;
  m.chol = chol;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (count + 127) / 128;
  uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  gen_points_kernel<<<(unsigned)blocks, 128, 0, (cudaStream_t)stream>>>(m, start, count, dtype,
                                                                           out_dev);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
