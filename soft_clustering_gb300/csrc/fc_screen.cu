// fc_screen.cu - tensor-core screen of full-covariance log joints: the
// candidate mask of every point for the kernels of fullcov.cu.
//
// "low-precision GMM operator" notes, sec. 1.2 (Cholesky route: the squared
// Mahalanobis distance is |z|^2 with z = L^-1 (x - mu)) and sec. 3.1 (the
// distance kernel as a matrix product); Flash-GMM summary, Method
// (block-wise responsibilities over all components of a tile).
//
// For a tile of 128 points the contraction Z~ = X [W~_1; ...; W~_K]^T runs on
// the tensor cores (tcgen05.mma, kind::f16: X as stored in fp16, W~_k =
// fp16(W_k / s_k) with s_k a power of two, fp32 accumulators in TMEM, K*D <=
// 1024 columns in at most two halves of 512; D = 32 or 64, the contraction
// dimension padded with zeros to 64).  Per point and component the
// epilogue forms z~ = s_k Z~_k - b_k (b_k = W_k mu_k in fp32) and bounds the
// exact z = W_k (x - mu_k):
//   |z~ - z| <= E = (2^-11 + 2^-16) |W_k|_F |x| + 2^-18 |W_k|_F |mu_k|
//                   + 2^-25 s_k D |x| + 2^-15 |z~|
// (fp16 rounding of W_k / s_k: 2^-11 relative, or 2^-25 s_k absolute where it
// falls subnormal; the fp32 accumulation of 64 exact products: 2^-17
// relative to the sum of their magnitudes; the fp32 bias: 64 roundings of
// its terms; the subtraction and |z~| itself: 2^-15 |z~|; each product sum
// bounded by Cauchy-Schwarz), so the true log joint l = c - |z|^2 / 2 lies in
//   [c - (|z~| + E)^2 / 2,  c - max(0, |z~| - E)^2 / 2].
// The mask holds every component whose upper bound reaches the largest lower
// bound less 41 nats: every component within 40 nats of the point's best.  A
// point with a non-finite coordinate gets every component (the exact kernels
// then report it).
//
// One persistent CTA of 8 warps per SM.  The B image and the per-component
// constants (written by gmm_prepare) arrive by bulk copies once.  Per tile the
// columns go in quarters of 256 (four components at D = 64) through two TMEM
// buffers, so the contraction of quarter q + 1 runs while the epilogue reads
// quarter q; warps w and w + 4 share TMEM lanes 32 (w % 4) .. + 31 (a point
// each) and split every quarter's components.  The next tile's rows are
// loaded into registers while the current tile is screened.
#include <math.h>

#include "gmm_internal.cuh"
#include "tc_ptx.cuh"

namespace gmm {
namespace {

constexpr int kScrThreads = 256;   // 8 warps: two threads per point
constexpr int kScrRows = 128;      // points per tile (MMA M, TMEM lanes)
constexpr int kScrGrid = 152;
constexpr int kQCols = 256;        // columns per quarter (MMA N) and per TMEM buffer
constexpr uint32_t kScrWait = 1u << 22;

struct ScrArgs {
  const __half* X;
  int64_t N;
  int K;
  const unsigned char* B;  // prepared B image [K D][128]
  const float* T;          // prepared constants [4 kFcMaxK + K D]
  uint32_t* mask;          // [N]
  DeviceStatus* st;
};

// Shared memory from a 1024-byte aligned base: B image, A tile, constants,
// exchange between the two threads of a point, barriers.
struct ScrLayout {
  size_t b_img, a_img, cst, xch, bar, slot, bytes;
  __host__ __device__ static ScrLayout make(int D, int K) {
    ScrLayout L;
    size_t o = 0;
    L.b_img = o; o += (size_t)K * D * 128;
    o = (o + 1023) / 1024 * 1024;
    L.a_img = o; o += (size_t)kScrRows * 128;
    L.cst = o;   o += sizeof(float) * (4 * kFcMaxK + (size_t)K * D);
    L.xch = o;   o += sizeof(float) * 4 * kScrRows;
    L.bar = (o + 7) / 8 * 8; o = L.bar + 3 * 8;
    L.slot = o;  o += 8;
    L.bytes = o + 1024;  // room to align the base
    return L;
  }
};

template <int D>
__global__ void __launch_bounds__(kScrThreads, 1) fc_screen_kernel(const ScrArgs a) {
  constexpr int CPQ = kQCols / D;  // components per quarter
  constexpr int KS = 4;            // K steps of 16 (contraction dimension padded to 64)
  extern __shared__ unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  const int K = a.K;
  const ScrLayout L = ScrLayout::make(D, K);
  unsigned char* sB = sm + L.b_img;
  unsigned char* sA = sm + L.a_img;
  float* cs = reinterpret_cast<float*>(sm + L.cst);  // s_k | bias_k | ex_k | em_k | b_k
  float* xch = reinterpret_cast<float*>(sm + L.xch);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);  // full[2], operands
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + L.slot);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int r = tid & (kScrRows - 1), hh = tid >> 7;  // the point (TMEM lane) and half

  if (warp == 0) {
    tc::tmem_alloc(slot, 2 * kQCols);
    tc::tmem_relinquish();
  }
  const uint32_t b_bytes = (uint32_t)(K * D * 128);
  const uint32_t t_bytes = (uint32_t)(sizeof(float) * (4 * kFcMaxK + K * D));
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_init(&bar[2], 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&bar[2], b_bytes + t_bytes);
    for (uint32_t o = 0; o < b_bytes; o += 16384)
      tc::bulk_g2s(sB + o, a.B + o, min(16384u, b_bytes - o), &bar[2]);
    tc::bulk_g2s(cs, a.T, t_bytes, &bar[2]);
  }
  const int64_t ntiles = (a.N + kScrRows - 1) / kScrRows;
  // this thread's half of its point's row: chunks 4 hh .. 4 hh + 3
  uint4 xr[4];
  auto fetch = [&](int64_t t) {
    const int64_t row = t * kScrRows + r;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = 4 * hh + c;
      xr[c] = (cc < D / 8 && row < a.N)
                  ? __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)row * D) + cc)
                  : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if ((int64_t)blockIdx.x < ntiles) fetch(blockIdx.x);
  const bool loaded = __syncthreads_and(tc::mbar_wait(&bar[2], 0, kScrWait)) != 0;
  if (!loaded && tid == 0) raise_status(a.st, GMM_ERR_TIMEOUT);
  tc::tc_fence_after();
  const uint32_t tmem = *slot;
  uint32_t valid = 0u;
  for (int k = 0; k < K; ++k)
    if (cs[kFcMaxK + k] > -INFINITY) valid |= 1u << k;
  const int nq = (K * D + kQCols - 1) / kQCols;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  uint32_t uses[2] = {0u, 0u};
  bool ok = loaded;

  auto issue = [&](int q) {  // thread 0: quarter q into TMEM buffer q & 1
    tc::tc_fence_after();
    const int n0 = q * kQCols, nn = min(kQCols, K * D - n0);
    const uint32_t idesc = tc::idesc_f16_f32(kScrRows, nn);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint64_t da = tc::sdesc_k128(tc::smem_addr(sA + ks * 32));
      const uint64_t db = tc::sdesc_k128(tc::smem_addr(sB + (size_t)n0 * 128 + ks * 32));
      tc::mma_f16(tmem + (uint32_t)((q & 1) * kQCols), da, db, idesc, ks > 0 ? 1u : 0u);
    }
    tc::mma_commit(&bar[q & 1]);
  };

  for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
    const int64_t row = t * kScrRows + r;
    // the A tile (128-byte swizzled rows) and this half's |x|^2
    float nx2 = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int cc = 4 * hh + c;
      const __half2* h2 = reinterpret_cast<const __half2*>(&xr[c]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(h2[q]);
        nx2 = fmaf(f.x, f.x, nx2);
        nx2 = fmaf(f.y, f.y, nx2);
      }
      *reinterpret_cast<uint4*>(sA + r * 128 + ((cc ^ (r & 7)) << 4)) = xr[c];
    }
    xch[hh * kScrRows + r] = nx2;
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) issue(0);
    if (t + gridDim.x < ntiles) fetch(t + gridDim.x);
    const float nxx = xch[r] + xch[kScrRows + r];
    const float nx = sqrtf(nxx) * (1.f + 1e-5f);
    // upper bounds of this thread's components: quarter q, k = q CPQ + 2 j + hh
    float hi[4][CPQ / 2];
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int j = 0; j < CPQ / 2; ++j) hi[q][j] = -INFINITY;
    float best_lo = -INFINITY;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q >= nq) break;
      if (tid == 0 && q + 1 < nq) issue(q + 1);
      const bool got = tc::mbar_wait(&bar[q & 1], uses[q & 1] & 1u, kScrWait);
      ++uses[q & 1];
      ok = __syncthreads_and(got) != 0;
      if (!ok) {
        if (tid == 0) raise_status(a.st, GMM_ERR_TIMEOUT);
        break;
      }
      tc::tc_fence_after();
#pragma unroll
      for (int j = 0; j < CPQ / 2; ++j) {
        const int kk = 2 * j + hh, k = q * CPQ + kk;
        if (k >= K) break;
        const float sk = cs[k], ck = cs[kFcMaxK + k];
        const float* bk = cs + 4 * kFcMaxK + k * D;
        float z2a = 0.f, z2b = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          tc::tmem_ld32(tmem + lane_base + (uint32_t)((q & 1) * kQCols + kk * D + c0), v);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float z0 = fmaf(sk, v[i], -bk[c0 + i]);
            const float z1 = fmaf(sk, v[i + 1], -bk[c0 + i + 1]);
            z2a = fmaf(z0, z0, z2a);
            z2b = fmaf(z1, z1, z2b);
          }
        }
        const float nz = sqrtf(z2a + z2b);
        const float E = cs[2 * kFcMaxK + k] * nx + cs[3 * kFcMaxK + k] + 3.0517578125e-05f * nz;
        const float dl = fmaxf(0.f, nz - E), dh = nz + E;
        hi[q][j] = ck - 0.5f * dl * dl;
        if (ck > -INFINITY) best_lo = fmaxf(best_lo, ck - 0.5f * dh * dh);
      }
      tc::tc_fence_before();
      __syncthreads();
    }
    if (!ok) break;
    // the two threads of a point: the best lower bound, then the mask
    xch[2 * kScrRows + hh * kScrRows + r] = best_lo;
    __syncthreads();
    const float b2 = fmaxf(xch[2 * kScrRows + r], xch[3 * kScrRows + r]);
    uint32_t m = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int j = 0; j < CPQ / 2; ++j) {
        const int k = q * CPQ + 2 * j + hh;
        if (k < K && hi[q][j] >= b2 - 41.f) m |= 1u << k;
      }
    __syncthreads();  // both halves have read the lower bounds
    reinterpret_cast<uint32_t*>(xch)[hh * kScrRows + r] = m;
    __syncthreads();
    if (hh == 0 && row < a.N) {
      uint32_t mm = m | reinterpret_cast<const uint32_t*>(xch)[kScrRows + r];
      if (!isfinite(nxx) || !(b2 > -INFINITY) || isnan(b2)) mm = valid;
      a.mask[row] = mm & valid;
    }
    __syncthreads();  // the exchange area and the A tile are free again
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 2 * kQCols);
  }
}

}  // namespace

// The screen covers fp16 X with the shapes fc_tc_shape admits.
bool fc_screen_eligible(int D, int K, int xdtype) {
  return xdtype == GMM_F16 && fc_tc_shape(D, K, GMM_COV_FULL);
}

cudaError_t fc_screen(const void* X, int64_t N, int D, int K, const void* prepared,
                      uint32_t* mask, DeviceStatus* st, cudaStream_t s) {
  const PreparedLayout PL = PreparedLayout::make(D, K, GMM_COV_FULL);
  ScrArgs a;
  a.X = static_cast<const __half*>(X);
  a.N = N; a.K = K;
  a.B = at<unsigned char>(prepared, PL.off_fcB);
  a.T = at<float>(prepared, PL.off_fcT);
  a.mask = mask; a.st = st;
  // at least 116 KB of shared memory, so a single block holds an SM's TMEM
  size_t smem = ScrLayout::make(D, K).bytes;
  if (smem < (size_t)116 * 1024) smem = (size_t)116 * 1024;
  const int64_t ntiles = (N + kScrRows - 1) / kScrRows;
  const int grid = (int)(ntiles < kScrGrid ? ntiles : kScrGrid);
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    ProfScope prof("fc_screen_kernel", s);
    kern<<<grid, kScrThreads, smem, s>>>(a);
    return cudaGetLastError();
  };
  if (D == 32) return go(fc_screen_kernel<32>);
  if (D == 64) return go(fc_screen_kernel<64>);
  return cudaErrorInvalidValue;
}

}  // namespace gmm
