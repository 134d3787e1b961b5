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
#include <math.h>

#include "gmm_internal.cuh"
#include "tc_ptx.cuh"

namespace gmm {
namespace {

constexpr int kScrThreads = 128;   // 4 warps: a point (TMEM lane) per thread
constexpr int kScrRows = 128;      // points per tile (MMA M)
constexpr int kScrGrid = 152;
constexpr int kScrMaxK = 32;
constexpr int kHalfCols = 512;     // TMEM columns
constexpr uint32_t kScrWait = 1u << 22;

struct ScrArgs {
  const __half* X;
  int64_t N;
  int K;
  const float* W;      // [K][D][D] W = L^-1 (lower)
  const float* mu;     // [K][D]
  const float* bias;   // [K]
  uint32_t* mask;      // [N]
  DeviceStatus* st;
};

// Shared memory (offsets from a 1024-byte aligned base): B image (K*D rows of
// 128 bytes, 128-byte swizzle), A tile, b_k, per-component constants.
struct ScrLayout {
  size_t b_img, a_img, bk, cst, red, bar, slot, bytes;
  __host__ __device__ static ScrLayout make(int D, int K) {
    ScrLayout L;
    size_t o = 0;
    L.b_img = o; o += (size_t)K * D * 128;
    o = (o + 1023) / 1024 * 1024;
    L.a_img = o; o += (size_t)kScrRows * 128;
    L.bk = o;    o += sizeof(float) * (size_t)K * D;
    L.cst = o;   o += sizeof(float) * 4 * kScrMaxK;
    L.red = o;   o += sizeof(float) * 3 * (kScrThreads / 32);
    L.bar = (o + 7) / 8 * 8; o = L.bar + 8;
    L.slot = o;  o += 8;
    L.bytes = o + 1024;  // room to align the base
    return L;
  }
};

template <int D>
__global__ void __launch_bounds__(kScrThreads, 1) fc_screen_kernel(const ScrArgs a) {
  constexpr int CPH = kHalfCols / D;  // components per TMEM half
  constexpr int KS = 4;               // K steps of 16 (K dimension padded to 64)
  extern __shared__ unsigned char smraw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  const int K = a.K;
  const ScrLayout L = ScrLayout::make(D, K);
  unsigned char* sB = sm + L.b_img;
  unsigned char* sA = sm + L.a_img;
  float* sb = reinterpret_cast<float*>(sm + L.bk);          // b_k = W_k mu_k  [K*D]
  float* cs = reinterpret_cast<float*>(sm + L.cst);         // s_k, c_k, ex_k, em_k
  float* red = reinterpret_cast<float*>(sm + L.red);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L.bar);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + L.slot);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (warp == 0) {
    tc::tmem_alloc(slot, kHalfCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(bar, 1);
    tc::mbar_fence_init();
  }
  // per component: the scale, |W|_F and |mu| (block reductions), the bias
  for (int k = 0; k < K; ++k) {
    const float* Wk = a.W + (size_t)k * D * D;
    float mx = 0.f, f2 = 0.f, m2 = 0.f;
    for (int e = tid; e < D * D; e += kScrThreads) {
      const int i = e / D, j = e % D;
      if (j <= i) {
        const float w = __ldg(Wk + e);
        mx = fmaxf(mx, fabsf(w));
        f2 = fmaf(w, w, f2);
      }
    }
    for (int d = tid; d < D; d += kScrThreads) {
      const float m = __ldg(a.mu + (size_t)k * D + d);
      m2 = fmaf(m, m, m2);
    }
    for (int o = 16; o > 0; o >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      f2 += __shfl_xor_sync(0xffffffffu, f2, o);
      m2 += __shfl_xor_sync(0xffffffffu, m2, o);
    }
    __syncthreads();
    if (lane == 0) { red[warp] = mx; red[4 + warp] = f2; red[8 + warp] = m2; }
    __syncthreads();
    if (tid == 0) {
      float M = 0.f, F2 = 0.f, M2 = 0.f;
      for (int w = 0; w < kScrThreads / 32; ++w) {
        M = fmaxf(M, red[w]);
        F2 += red[4 + w];
        M2 += red[8 + w];
      }
      // s = 2^e with max |W| / s in [2^14, 2^15)
      int e2 = 0;
      frexpf(M > 0.f ? M : 1.f, &e2);  // M = f 2^e2, f in [0.5, 1)
      const float s = ldexpf(1.f, e2 - 15);
      const float F = sqrtf(F2) * (1.f + 1e-5f);
      const float mun = sqrtf(M2) * (1.f + 1e-5f);
      cs[k] = s;
      cs[kScrMaxK + k] = __ldg(a.bias + k);
      cs[2 * kScrMaxK + k] = 1.01f * ((0.00048828125f + 1.52587890625e-05f) * F +
                                     2.98023223876953125e-08f * s * (float)D);
      cs[3 * kScrMaxK + k] = 1.01f * 3.814697265625e-06f * F * mun;
    }
  }
  __syncthreads();
  // B image: row n = k D + i holds fp16(W_k[i][j] / s_k) for j <= i, else 0;
  // and b_k = W_k mu_k
  for (int u = tid; u < K * D * 8; u += kScrThreads) {
    const int n = u >> 3, c = u & 7, k = n / D, i = n % D;
    const float inv = 1.f / cs[k];
    const float* Wr = a.W + ((size_t)k * D + i) * D;
    __align__(16) __half h[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int j = 8 * c + t;
      h[t] = __float2half_rn(j < D && j <= i ? __ldg(Wr + j) * inv : 0.f);
    }
    *reinterpret_cast<uint4*>(sB + n * 128 + ((c ^ (n & 7)) << 4)) = *reinterpret_cast<const uint4*>(h);
  }
  for (int n = tid; n < K * D; n += kScrThreads) {
    const int k = n / D, i = n % D;
    const float* Wr = a.W + ((size_t)k * D + i) * D;
    const float* mk = a.mu + (size_t)k * D;
    float s = 0.f;
    for (int j = 0; j <= i; ++j) s = fmaf(__ldg(Wr + j), __ldg(mk + j), s);
    sb[n] = s;
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *slot;
  uint32_t valid = 0u;
  for (int k = 0; k < K; ++k)
    if (cs[kScrMaxK + k] > -INFINITY) valid |= 1u << k;
  const int halves = (K * D + kHalfCols - 1) / kHalfCols;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  uint32_t phase = 0;
  bool ok = true;
  const int64_t ntiles = (a.N + kScrRows - 1) / kScrRows;
  for (int64_t t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
    const int64_t row = t * kScrRows + tid;
    const bool in = row < a.N;
    // the A tile: this thread's row, 128-byte swizzled, K padded to 64
    float nx2 = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (c < D / 8 && in) {
        v = __ldg(reinterpret_cast<const uint4*>(a.X + (size_t)row * D) + c);
        const __half2* h2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(h2[q]);
          nx2 = fmaf(f.x, f.x, nx2);
          nx2 = fmaf(f.y, f.y, nx2);
        }
      }
      *reinterpret_cast<uint4*>(sA + tid * 128 + ((c ^ (tid & 7)) << 4)) = v;
    }
    const float nx = sqrtf(nx2) * (1.f + 1e-5f);
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    float hi[kScrMaxK];
    float best_lo = -INFINITY;
#pragma unroll
    for (int k = 0; k < kScrMaxK; ++k) hi[k] = -INFINITY;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (h >= halves) break;
      if (tid == 0) {
        tc::tc_fence_after();
        const int ncols = min(kHalfCols, K * D - h * kHalfCols);
        for (int n0 = 0; n0 < ncols; n0 += 256) {
          const int nn = min(256, ncols - n0);
          const uint32_t idesc = tc::idesc_f16_f32(kScrRows, nn);
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const uint64_t da = tc::sdesc_k128(tc::smem_addr(sA + ks * 32));
            const uint64_t db = tc::sdesc_k128(tc::smem_addr(sB + (size_t)(h * kHalfCols + n0) * 128 + ks * 32));
            tc::mma_f16(tmem + (uint32_t)n0, da, db, idesc, ks > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(bar);
      }
      const bool got = tc::mbar_wait(bar, phase, kScrWait);
      phase ^= 1u;
      ok = __syncthreads_and(got) != 0;  // the same outcome in every thread
      if (!ok && tid == 0) raise_status(a.st, GMM_ERR_TIMEOUT);
      tc::tc_fence_after();
      if (ok) {
#pragma unroll
        for (int kk = 0; kk < CPH; ++kk) {
          const int k = h * CPH + kk;
          if (k >= K || k >= kScrMaxK) break;
          const float s = cs[k], ck = cs[kScrMaxK + k];
          float z2a = 0.f, z2b = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float v[32];
            tc::tmem_ld32(tmem + lane_base + (uint32_t)(kk * D + c0), v);
            const float* bk = sb + k * D + c0;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float z0 = fmaf(s, v[i], -bk[i]);
              const float z1 = fmaf(s, v[i + 1], -bk[i + 1]);
              z2a = fmaf(z0, z0, z2a);
              z2b = fmaf(z1, z1, z2b);
            }
          }
          const float nz = sqrtf(z2a + z2b);
          const float E = cs[2 * kScrMaxK + k] * nx + cs[3 * kScrMaxK + k] + 3.0517578125e-05f * nz;
          const float dl = fmaxf(0.f, nz - E), dh = nz + E;
          const float lo = ck - 0.5f * dh * dh;
          hi[k] = ck - 0.5f * dl * dl;
          if (ck > -INFINITY) best_lo = fmaxf(best_lo, lo);
        }
      }
      tc::tc_fence_before();
      __syncthreads();
      if (!ok) break;
    }
    if (ok && in) {
      uint32_t m = 0u;
#pragma unroll
      for (int k = 0; k < kScrMaxK; ++k)
        if (k < K && hi[k] >= best_lo - 41.f) m |= 1u << k;
      if (!isfinite(nx2) || !(best_lo > -INFINITY) || isnan(best_lo)) m = valid;
      a.mask[row] = m & valid;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kHalfCols);
  }
}

}  // namespace

// The screen covers fp16 X with D in {32, 64} and K D <= 1024.
bool fc_screen_eligible(int D, int K, int xdtype) {
  return xdtype == GMM_F16 && (D == 32 || D == 64) && K >= 1 && K <= kScrMaxK &&
         K * D <= 2 * kHalfCols;
}

cudaError_t fc_screen(const void* X, int64_t N, int D, int K, const void* prepared,
                      uint32_t* mask, DeviceStatus* st, cudaStream_t s) {
  const PreparedLayout PL = PreparedLayout::make(D, K, GMM_COV_FULL);
  ScrArgs a;
  a.X = static_cast<const __half*>(X);
  a.N = N; a.K = K;
  a.W = at<float>(prepared, PL.off_prec);
  a.mu = at<float>(prepared, PL.off_mu);
  a.bias = at<float>(prepared, PL.off_c);
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
