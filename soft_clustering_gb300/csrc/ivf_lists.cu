// ivf_lists.cu - inverted lists for IVF multi-assignment, built on the device
// from the top-m output of gmm_assign_topm.
//
// Flash-GMM summary, "Core insight" (second point) and "Experiments / key
// findings": with soft assignment a vector near a cluster boundary is put in
// the lists of several high-responsibility clusters instead of one.  Entry
// (n, t) of the top-m output joins the list of component ids[n m + t] when
// it is the point's best component (t = 0) or its responsibility is at least
// gamma_min; every list holds its points in ascending order.
//
// Three steps, all with integer counts, so the lists are the same on every
// run:
//   count    entries per (component, block of kPB points), a shared-memory
//            histogram per block, taken over slices of kSlice components
//   scan     per component, over its blocks (exclusive), then over the
//            components: list offsets (int64) and each block's start in
//            every list
//   scatter  one warp per block walks its points in order, 32 entries at a
//            time; __match_any_sync ranks the entries of one component
#include "gmm_internal.cuh"

namespace gmm {
namespace {

constexpr int kPB = 8192;         // points per counting / scattering block
constexpr int kSlice = 12288;     // components per shared-memory histogram pass
constexpr int kCountThreads = 256;
constexpr int kScanThreads = 1024;
constexpr int kSmemCursorK = 12288;  // scatter keeps its cursors in shared memory up to this K

__device__ __forceinline__ bool joins(int t, float g, float gmin) { return t == 0 || g >= gmin; }

__global__ void __launch_bounds__(kCountThreads)
ivf_count_kernel(const int32_t* __restrict__ ids, const float* __restrict__ gamma, int64_t N,
                 int m, int K, float gmin, int64_t nb, uint32_t* __restrict__ counts) {
  __shared__ uint32_t hist[kSlice];
  const int64_t b = blockIdx.x;
  const int64_t e0 = b * kPB * (int64_t)m;
  const int64_t e1 = min(N, (b + 1) * kPB) * (int64_t)m;
  for (int k0 = 0; k0 < K; k0 += kSlice) {
    const int ks = min(kSlice, K - k0);
    for (int i = threadIdx.x; i < ks; i += kCountThreads) hist[i] = 0u;
    __syncthreads();
    for (int64_t e = e0 + threadIdx.x; e < e1; e += kCountThreads) {
      const int k = ids[e];
      const int t = (int)(e % m);
      if (k >= k0 && k < k0 + ks && joins(t, gamma[e], gmin)) atomicAdd(&hist[k - k0], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < ks; i += kCountThreads)
      counts[(size_t)(k0 + i) * nb + b] = hist[i];
    __syncthreads();
  }
}

// Exclusive block-wide prefix (kScanThreads) of one value per thread.
__device__ __forceinline__ uint64_t block_scan64(uint64_t v, uint64_t* wsum, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint64_t t = wsum[lane];
    uint64_t ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t u = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += u;
    }
    wsum[lane] = ti - t;
    if (lane == 31) *total = ti;
  }
  __syncthreads();
  const uint64_t r = wsum[warp] + incl - v;
  __syncthreads();
  return r;
}

// One block per component: counts[k][b] -> offset of block b within list k
// (in place), tot[k] = the list's length.
__global__ void __launch_bounds__(kScanThreads)
ivf_scan_blocks_kernel(uint32_t* __restrict__ counts, int64_t nb, uint64_t* __restrict__ tot) {
  __shared__ uint64_t wsum[kScanThreads / 32];
  __shared__ uint64_t total;
  const int k = blockIdx.x;
  uint32_t* c = counts + (size_t)k * nb;
  uint64_t carry = 0;
  for (int64_t base = 0; base < nb; base += kScanThreads) {
    const int64_t i = base + threadIdx.x;
    const uint64_t v = i < nb ? c[i] : 0u;
    const uint64_t ex = block_scan64(v, wsum, &total);
    if (i < nb) c[i] = (uint32_t)(carry + ex);
    carry += total;
  }
  if (threadIdx.x == 0) tot[k] = carry;
}

// One block: offsets[k] = start of list k, offsets[K] = number of entries.
__global__ void __launch_bounds__(kScanThreads)
ivf_scan_lists_kernel(const uint64_t* __restrict__ tot, int K, int64_t* __restrict__ offsets) {
  __shared__ uint64_t wsum[kScanThreads / 32];
  __shared__ uint64_t total;
  const int kper = (K + kScanThreads - 1) / kScanThreads;
  const int k0 = min(K, (int)threadIdx.x * kper), k1 = min(K, k0 + kper);
  uint64_t mine = 0;
  for (int k = k0; k < k1; ++k) mine += tot[k];
  uint64_t run = block_scan64(mine, wsum, &total);
  for (int k = k0; k < k1; ++k) {
    offsets[k] = (int64_t)run;
    run += tot[k];
  }
  if (threadIdx.x == 0) offsets[K] = (int64_t)total;
}

// One warp per block of kPB points.  The cursor of list k starts at
// offsets[k] + the block's offset within the list and moves by the entries
// placed; cursors live in shared memory (K <= kSmemCursorK) or in the block's
// own column of `counts` (each column is read and written by one warp only).
__global__ void __launch_bounds__(32)
ivf_scatter_kernel(const int32_t* __restrict__ ids, const float* __restrict__ gamma, int64_t N,
                   int m, int K, float gmin, int64_t nb, uint32_t* __restrict__ counts,
                   const int64_t* __restrict__ offsets, int32_t* __restrict__ list_pts,
                   float* __restrict__ list_gamma) {
  extern __shared__ uint32_t scur[];
  const int64_t b = blockIdx.x;
  const int lane = threadIdx.x;
  const bool in_smem = K <= kSmemCursorK;
  if (in_smem)
    for (int k = lane; k < K; k += 32) scur[k] = counts[(size_t)k * nb + b];
  __syncwarp();
  const int64_t e0 = b * kPB * (int64_t)m;
  const int64_t e1 = min(N, (b + 1) * kPB) * (int64_t)m;
  for (int64_t base = e0; base < e1; base += 32) {
    const int64_t e = base + lane;
    int k = -1;
    float g = 0.f;
    if (e < e1) {
      k = ids[e];
      g = gamma[e];
      if (!(k >= 0 && k < K && joins((int)(e % m), g, gmin))) k = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, k);
    uint32_t cur = 0;
    if (k >= 0) cur = in_smem ? scur[k] : counts[(size_t)k * nb + b];
    if (k >= 0) {
      const int64_t pos = offsets[k] + (int64_t)cur + __popc(grp & ((1u << lane) - 1u));
      list_pts[pos] = (int32_t)(e / m);
      list_gamma[pos] = g;
    }
    __syncwarp();
    if (k >= 0 && lane == 31 - __clz(grp)) {
      if (in_smem) scur[k] = cur + __popc(grp);
      else counts[(size_t)k * nb + b] = cur + __popc(grp);
    }
    __syncwarp();
  }
}

struct IvfLayout {
  int64_t nb;
  size_t off_counts, off_tot, bytes;
  static IvfLayout make(int64_t N, int K) {
    IvfLayout L;
    L.nb = (N + kPB - 1) / kPB;
    size_t o = 0;
    L.off_counts = o; o = align_up(o + sizeof(uint32_t) * (size_t)K * L.nb);
    L.off_tot = o;    o = align_up(o + sizeof(uint64_t) * (size_t)K);
    L.bytes = o;
    return L;
  }
};

gmm_status ivf_cuda(cudaError_t e) { return e == cudaSuccess ? GMM_OK : GMM_ERR_CUDA; }

}  // namespace
}  // namespace gmm

using namespace gmm;

extern "C" {

size_t gmm_ivf_lists_ws_bytes(int64_t N, int m, int K) {
  if (N < 1 || N > INT32_MAX || m < 1 || m > 8 || K < 1 || K > (1 << 16)) return 0;
  return IvfLayout::make(N, K).bytes;
}

gmm_status gmm_ivf_lists(const int32_t* ids, const float* gamma, int64_t N, int m, int K,
                         float gamma_min, int64_t* offsets, int32_t* list_pts, float* list_gamma,
                         void* ws, size_t ws_bytes, void* stream) {
  if (!ids || !gamma || !offsets || !list_pts || !list_gamma || !ws) return GMM_ERR_INVALID_ARG;
  if (N < 1 || N > INT32_MAX || m < 1 || m > 8 || K < 1 || K > (1 << 16) || !(gamma_min == gamma_min))
    return GMM_ERR_INVALID_ARG;
  const IvfLayout L = IvfLayout::make(N, K);
  if (ws_bytes < L.bytes) return GMM_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t* counts = at<uint32_t>(ws, L.off_counts);
  uint64_t* tot = at<uint64_t>(ws, L.off_tot);
  {
    ProfScope p("ivf_lists_kernels", s, 4);
    ivf_count_kernel<<<(unsigned)L.nb, kCountThreads, 0, s>>>(ids, gamma, N, m, K, gamma_min, L.nb,
                                                               counts);
    gmm_status r = ivf_cuda(cudaGetLastError());
    if (r != GMM_OK) return r;
    ivf_scan_blocks_kernel<<<K, kScanThreads, 0, s>>>(counts, L.nb, tot);
    if ((r = ivf_cuda(cudaGetLastError())) != GMM_OK) return r;
    ivf_scan_lists_kernel<<<1, kScanThreads, 0, s>>>(tot, K, offsets);
    if ((r = ivf_cuda(cudaGetLastError())) != GMM_OK) return r;
    const size_t smem = K <= kSmemCursorK ? sizeof(uint32_t) * (size_t)K : 0;
    ivf_scatter_kernel<<<(unsigned)L.nb, 32, smem, s>>>(ids, gamma, N, m, K, gamma_min, L.nb,
                                                        counts, offsets, list_pts, list_gamma);
    if ((r = ivf_cuda(cudaGetLastError())) != GMM_OK) return r;
  }
  return GMM_OK;
}

}  // extern "C"
