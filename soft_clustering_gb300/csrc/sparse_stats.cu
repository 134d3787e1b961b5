// sparse_stats.cu - sufficient statistics from the tensor-core E-step's
// responsibility records (Flash-GMM summary, Method: online s0, s1, s2).
//
// The screening kernel writes, per 128-point tile, the (component, point,
// gamma) of every pair it evaluated exactly, in point order.  All other
// pairs carry less than 4.3e-18 of their point's responsibility.  This
// kernel turns the records into per-block statistics without an N x K
// matrix: a block owns one slice of 8192 / D components (its accumulators,
// slice x (1 + 2D) fp32, live in shared memory) and one range of tiles; warp w
// accumulates the records of the components k with k % 8 == w, in record
// order, so the sums are the same on every run.  Moments are taken about the
// component's input mean c_k (y = x - c_k); accumulators are flushed into fp64
// per-block partials every kFlushTiles tiles, and at the end the second
// moment is moved to the block's own weighted mean, giving the
// [S0 | S1 about c | M2 about the block mean] partials the M-step merges.
#include <math.h>

#include "gmm_internal.cuh"

namespace gmm {
namespace {

constexpr int kThreads = 256;
constexpr int kFlushTiles = 16;   // fp32 accumulation span (2048 points)

// Components per block: 64 for D = 128, 128 for D = 64 (about 100 KB of
// shared memory, two blocks per SM).
template <int D>
constexpr int slice_of() { return 8192 / D; }

// records: uint2 {(k << 7) | row_in_tile, bits of gamma}.
template <int D, int XT>
__global__ void __launch_bounds__(kThreads)
sparse_stats_kernel(const void* __restrict__ X, int64_t N, int K, const void* __restrict__ prepared,
                    PreparedLayout L, const uint32_t* __restrict__ tile_cnt,
                    const uint2* __restrict__ recs, int rec_cap, int64_t ntiles,
                    int64_t tiles_per_part, double* __restrict__ part, int accumulate) {
  constexpr int F = 1 + 2 * D;
  constexpr int DPL = D / 32;
  constexpr int kSlice = slice_of<D>();
  extern __shared__ float sm[];
  float* acc = sm;                       // [kSlice][F]
  float* cent = acc + kSlice * F;        // [kSlice][D]
  uint2* srec = (uint2*)(cent + kSlice * D);  // [rec_cap]

  const int s = blockIdx.x;              // component slice
  const int64_t p = blockIdx.y;          // tile partition
  const int k0 = s * kSlice;
  const int kn = min(kSlice, K - k0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* g_mu = at<float>(prepared, L.off_mu);
  for (int i = tid; i < kSlice * D; i += kThreads)
    cent[i] = i < kn * D ? g_mu[(size_t)k0 * D + i] : 0.f;
  for (int i = tid; i < kSlice * F; i += kThreads) acc[i] = 0.f;
  double* out = part + ((size_t)p * K + k0) * F;
  if (!accumulate) {
    for (int i = tid; i < kn * F; i += kThreads) out[i] = 0.0;
  } else {
    // continue a partial from an earlier call: back to the second moment
    // about the centre, S2c = M2 + S1^2 / S0
    for (int i = tid; i < kn * D; i += kThreads) {
      double* o = out + (size_t)(i / D) * F;
      const int d = i % D;
      if (o[0] > 0.0) o[1 + D + d] += o[1 + d] * o[1 + d] / o[0];
    }
  }
  __syncthreads();

  const int64_t t0 = p * tiles_per_part;
  const int64_t t1 = min(ntiles, t0 + tiles_per_part);
  int since_flush = 0;
  auto flush = [&]() {
    __syncthreads();
    for (int i = tid; i < kn * F; i += kThreads) {
      out[i] += (double)acc[i];
      acc[i] = 0.f;
    }
    __syncthreads();
  };
  for (int64_t t = t0; t < t1; ++t) {
    const uint32_t tc_n = tile_cnt[t];
    const int cnt = tc_n < (uint32_t)rec_cap ? (int)tc_n : rec_cap;
    for (int i = tid; i < cnt; i += kThreads) srec[i] = recs[(size_t)t * rec_cap + i];
    __syncthreads();
    for (int base = 0; base < cnt; base += 32) {
      const int i = base + lane;
      uint2 rec = make_uint2(0u, 0u);
      bool own = false;
      if (i < cnt) {
        rec = srec[i];
        const int k = (int)(rec.x >> 7);
        own = (k >= k0) && (k < k0 + kn) && (((k - k0) & 7) == warp);
      }
      unsigned mask = __ballot_sync(0xffffffffu, own);
      while (mask) {
        const int b = __ffs(mask) - 1;
        mask &= mask - 1;
        const uint32_t key = __shfl_sync(0xffffffffu, rec.x, b);
        const float g = __uint_as_float(__shfl_sync(0xffffffffu, rec.y, b));
        const int kl = (int)(key >> 7) - k0;
        const int64_t n = t * 128 + (key & 127);
        if (n >= N) continue;  // (never written for rows past the end)
        float* a = acc + kl * F;
#pragma unroll
        for (int q = 0; q < DPL; ++q) {
          const int d = q * 32 + lane;  // lane-interleaved: conflict-free shared memory
          const float y = load_x<XT>(X, (size_t)n * D + d) - cent[kl * D + d];
          const float gy = g * y;
          a[1 + d] += gy;
          a[1 + D + d] = fmaf(gy, y, a[1 + D + d]);
        }
        if (lane == 0) a[0] += g;
        __syncwarp();
      }
    }
    __syncthreads();
    if (++since_flush == kFlushTiles) {
      flush();
      since_flush = 0;
    }
  }
  flush();
  // second moment about this block's weighted mean: M2 = S2c - S1c^2 / S0
  for (int i = tid; i < kn * D; i += kThreads) {
    const int kl = i / D, d = i % D;
    double* o = out + (size_t)kl * F;
    const double s0 = o[0];
    if (s0 > 0.0) o[1 + D + d] = o[1 + D + d] - o[1 + d] * o[1 + d] / s0;
  }
}

template <int D, int XT>
cudaError_t run_sparse(const void* X, int64_t N, int K, int cov, const void* prepared,
                       const uint32_t* tile_cnt, const uint2* recs, int rec_cap, int parts,
                       double* part, int accumulate, cudaStream_t s) {
  constexpr int F = 1 + 2 * D;
  constexpr int kSlice = slice_of<D>();
  const PreparedLayout L = PreparedLayout::make(D, K, cov);
  const int64_t ntiles = (N + 127) / 128;
  const int slices = (K + kSlice - 1) / kSlice;
  const int64_t tpp = (ntiles + parts - 1) / parts;
  const size_t smem = sizeof(float) * (size_t)kSlice * (F + D) + sizeof(uint2) * (size_t)rec_cap;
  auto kern = sparse_stats_kernel<D, XT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(slices, parts);
  kern<<<grid, kThreads, smem, s>>>(X, N, K, prepared, L, tile_cnt, recs, rec_cap, ntiles, tpp,
                                    part, accumulate);
  return cudaGetLastError();
}

}  // namespace

// Partitions of the tile range so that slices x partitions ~ 2 blocks per SM
// (304 on 152 SMs).  Depends on D and K only, so that every chunk of a
// streamed pass accumulates into the same partials.
int sparse_stats_parts(int D, int K) {
  const int slice = D == 128 ? slice_of<128>() : slice_of<64>();
  const int slices = (K + slice - 1) / slice;
  const int p = (304 + slices - 1) / slices;
  return p < 1 ? 1 : p;
}

// Diagonal / isotropic statistics (the partial layout is the same for both;
// the isotropic M-step averages the diagonal).  prepared: the block written
// for this call's parameters (its mean array is the centre c).  accumulate:
// merge into partials left by an earlier call (chunks of host data).
cudaError_t sparse_stats(const void* X, int xdtype, int64_t N, int D, int K, const void* prepared,
                         int cov, const uint32_t* tile_cnt, const uint2* recs, int rec_cap,
                         int parts, double* part, int accumulate, cudaStream_t s) {
#define GMM_SPARSE(DD, XX) \
  return run_sparse<DD, XX>(X, N, K, cov, prepared, tile_cnt, recs, rec_cap, parts, part, accumulate, s)
  if (D == 128) {
    if (xdtype == GMM_F16) { GMM_SPARSE(128, GMM_F16); }
    if (xdtype == GMM_BF16) { GMM_SPARSE(128, GMM_BF16); }
    GMM_SPARSE(128, GMM_F32);
  }
  if (D == 64) {
    if (xdtype == GMM_F16) { GMM_SPARSE(64, GMM_F16); }
    if (xdtype == GMM_BF16) { GMM_SPARSE(64, GMM_BF16); }
    GMM_SPARSE(64, GMM_F32);
  }
#undef GMM_SPARSE
  return cudaErrorInvalidValue;
}

}  // namespace gmm
