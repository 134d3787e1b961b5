// fullcov.cu - E-step and sufficient statistics of full-covariance mixtures
// with few components, driven by per-point candidate masks.
//
// "low-precision GMM operator" notes, sec. 1.2 (the Cholesky route:
// z = L^-1 (x - mu), d^2 = z.z) and sec. 3.2 (fused distance and posterior,
// fp32 log-sum-exp); Flash-GMM summary, Method (s0 = sum g, s1 = sum g x,
// s2 = sum g x x^T).
//
// A point's candidate mask has one bit per component (K <= 32).  Every
// component within 40 nats of the point's best log joint has its bit set (the
// tensor-core screen of fc_screen.cu guarantees it; without the screen every
// component with a finite bias is set), and the others carry less than
// 4.3e-18 of the point's responsibility.  Two kernels:
//   fc_lse    persistent blocks holding every component's W = L^-1 (rows
//             padded to a multiple of four floats, zero beyond the diagonal),
//             mean and bias in shared memory.  Per tile of 128 points: the
//             (component, point) pairs of the masks in component-major order,
//             a thread per pair (the lanes of a warp mostly share a component,
//             so W is read by broadcast), the exact log joint; then a thread
//             per point: LSE_n over its candidates in component order, and
//             the log-likelihood.
//   fc_stats  a block per (component, partition of the points): the
//             partition's candidates of the component, their log joints
//             recomputed with four threads a point (bit-identical to fc_lse),
//             g = exp(l - LSE_n) and y = x - mu gathered into chunks of up to
//             256 points; per chunk s0, the chunk mean and the second moment
//             about it in fp32 (4 x 4 register tiles of the lower triangle),
//             merged into the block's fp64 sums with the pairwise update of
//             Chan, Golub and LeVeque.  The partial written per (partition,
//             component) is [S0 | S1 about mu | M2 about the block mean].
// Every sum has a fixed order, so the results are the same on every run.
#include <math.h>

#include <type_traits>

#include "gmm_internal.cuh"

namespace gmm {
namespace {

constexpr int kFcT = 128;          // points per fc_lse tile
constexpr int kFcThreads = 512;    // fc_lse block
constexpr int kFcGrid = 152;       // fc_lse blocks (fixed: the log-likelihood partial count)
constexpr int kFsThreads = 256;    // fc_stats block
constexpr int kFsTile = 256;       // partition points per mask tile (one per thread)
constexpr int kFsChunk = 256;      // candidate points per fp32 chunk
constexpr int kFcMaxK = 32;        // one mask word per point

// Floats of one component's padded W.  The rows 4m .. 4m + 3 hold 4(m + 1)
// floats each (zero beyond the diagonal), stored interleaved by 16-byte
// blocks from offset 8 m (m + 1): block b of row 4m + q at 16 b + 4 q, so the
// four rows of a group read together fall in four different bank groups.
__host__ __device__ constexpr int fc_wfloats(int D) { return 8 * (D / 4) * (D / 4 + 1); }
// Component stride in fc_lse (four more floats move the next component's
// rows to other banks).
__host__ __device__ constexpr int fc_wstride(int D) { return fc_wfloats(D) + 4; }

struct FcArgs {
  const void* X;          // the rows, [N][D]
  int64_t N;
  int K;
  const float* W;         // prepared W = L^-1, [K][D][D] row-major (lower)
  const float* mu;        // [K][D]
  const float* bias;      // [K]  log pi - log|S|/2 - (D/2) log 2 pi, -inf excluded
  const uint32_t* mask;   // [N]  candidate masks
  float* lse;             // [N]
  double* ll_part;        // [gridDim.x] of fc_lse
  double* stat;           // [P][K][F] fp64 partials
  int accumulate;
  DeviceStatus* st;
};

// Loads D coordinates starting at element e0 (a multiple of 4) as float4s.
template <int XT>
__device__ __forceinline__ float4 load4(const void* X, size_t e0) {
  if constexpr (XT == GMM_F32) {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(X) + e0));
  } else {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(X) + e0));
    float2 a, b;
    if constexpr (XT == GMM_F16) {
      a = __half22float2(*reinterpret_cast<const __half2*>(&q.x));
      b = __half22float2(*reinterpret_cast<const __half2*>(&q.y));
    } else {
      a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.x));
      b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&q.y));
    }
    return make_float4(a.x, a.y, b.x, b.y);
  }
}

// Partial d^2 over the rows i = q (mod 4) of z = W y: row i summed in two
// packed pairs of partial sums, ((z0 + z1) + (z2 + z3)); the squares added in
// increasing i with Neumaier's compensation.  d^2 = (p0 + p1) + (p2 + p3).
template <int D>
__device__ __forceinline__ float fc_part(const float* __restrict__ Wk, const float2 (&y2)[D / 2],
                                         int q) {
  constexpr int M = D / 4;
  float s = 0.f, c = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float* w = Wk + 8 * m * (m + 1) + 4 * q;
    float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
#pragma unroll
    for (int bk = 0; bk <= m; ++bk) {
      const float4 wv = *reinterpret_cast<const float4*>(w + 16 * bk);
      a = fma2(make_float2(wv.x, wv.y), y2[2 * bk], a);
      b = fma2(make_float2(wv.z, wv.w), y2[2 * bk + 1], b);
    }
    const float z = __fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(b.x, b.y));
    const float zz = __fmul_rn(z, z);
    const float t = __fadd_rn(s, zz);
    c = __fadd_rn(c, s >= zz ? __fadd_rn(__fsub_rn(s, t), zz) : __fadd_rn(__fsub_rn(zz, t), s));
    s = t;
  }
  return __fadd_rn(s, c);
}

// Stages component k's W rows (padded, zero beyond the diagonal) at dst.
template <int D>
__device__ __forceinline__ void stage_w(float* dst, const float* __restrict__ Wk, int i) {
  const int m = i >> 2, q = i & 3;
  float* row = dst + 8 * m * (m + 1) + 4 * q;
  for (int j = 0; j < 4 * (m + 1); ++j)
    row[16 * (j >> 2) + (j & 3)] = j <= i ? __ldg(Wk + (size_t)i * D + j) : 0.f;
}

template <int D, int XT>
__global__ void __launch_bounds__(kFcThreads, 1) fc_lse_kernel(const FcArgs a) {
  constexpr int WS = fc_wstride(D), XS = D + 4, NW = kFcT / 32;
  extern __shared__ __align__(16) float sm[];
  const int K = a.K;
  float* sW = sm;                                    // K * WS
  float* sMu = sW + K * WS;                          // K * D
  float* sC = sMu + K * D;                           // kFcMaxK
  float* xs = sC + kFcMaxK;                          // kFcT * XS
  float* lval = xs + kFcT * XS;                      // kFcT * K
  uint32_t* cm = reinterpret_cast<uint32_t*>(lval + kFcT * K);  // K * NW
  uint32_t* msk = cm + K * NW;                       // kFcT
  int* offs = reinterpret_cast<int*>(msk + kFcT);    // kFcMaxK + 4
  uint8_t* prow = reinterpret_cast<uint8_t*>(offs + kFcMaxK + 4);  // kFcT * K
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < K * D; e += kFcThreads) {
    const int k = e / D, i = e % D;
    stage_w<D>(sW + k * WS, a.W + (size_t)k * D * D, i);
    sMu[e] = __ldg(a.mu + e);
  }
  for (int k = tid; k < kFcMaxK; k += kFcThreads) sC[k] = k < K ? __ldg(a.bias + k) : -INFINITY;
  __syncthreads();
  uint32_t valid = 0u;
  for (int k = 0; k < K; ++k)
    if (sC[k] > -INFINITY) valid |= 1u << k;
  const int64_t ntiles = (a.N + kFcT - 1) / kFcT;
  double ll = 0.0;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r0 = t * kFcT;
    const int rows = (int)min((int64_t)kFcT, a.N - r0);
    __syncthreads();  // the previous tile's tables are no longer read
    // masks (component-major bit columns by ballot) and the rows of X
    if (tid < kFcT) {
      const uint32_t m = tid < rows ? __ldg(a.mask + r0 + tid) & valid : 0u;
      msk[tid] = m;
      for (int k = 0; k < K; ++k) {
        const uint32_t b = __ballot_sync(0xffffffffu, (m >> k) & 1u);
        if (lane == 0) cm[k * NW + warp] = b;
      }
    }
    for (int e = tid; e < kFcT * (D / 4); e += kFcThreads) {
      const int r = e / (D / 4), c4 = e % (D / 4);
      const float4 v = r < rows ? load4<XT>(a.X, (size_t)(r0 + r) * D + 4 * c4)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
      *reinterpret_cast<float4*>(xs + r * XS + 4 * c4) = v;
    }
    __syncthreads();
    // pair offsets per component
    if (warp == 0) {
      int cnt = 0;
      if (lane < K)
        for (int w = 0; w < NW; ++w) cnt += __popc(cm[lane * NW + w]);
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      if (lane < K) offs[lane + 1] = inc;
      if (lane == 0) offs[0] = 0;
    }
    __syncthreads();
    // the pair list: component-major, rows ascending
    if (tid < kFcT) {
      const uint32_t m = msk[tid], lt = (1u << lane) - 1u;
      for (int k = 0; k < K; ++k) {
        if (!((m >> k) & 1u)) continue;
        int pos = offs[k] + __popc(cm[k * NW + warp] & lt);
        for (int w = 0; w < warp; ++w) pos += __popc(cm[k * NW + w]);
        prow[pos] = (uint8_t)tid;
      }
    }
    __syncthreads();
    const int np = offs[K];
    int kk = 0;
    for (int p = tid; p < np; p += kFcThreads) {
      while (offs[kk + 1] <= p) ++kk;
      const int r = prow[p];
      float2 y2[D / 2];
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 xv = *reinterpret_cast<const float4*>(xs + r * XS + 4 * c4);
        const float4 mv = *reinterpret_cast<const float4*>(sMu + kk * D + 4 * c4);
        y2[2 * c4] = sub2(make_float2(xv.x, xv.y), make_float2(mv.x, mv.y));
        y2[2 * c4 + 1] = sub2(make_float2(xv.z, xv.w), make_float2(mv.z, mv.w));
      }
      const float* Wk = sW + kk * WS;
      const float d2 = __fadd_rn(__fadd_rn(fc_part<D>(Wk, y2, 0), fc_part<D>(Wk, y2, 1)),
                                 __fadd_rn(fc_part<D>(Wk, y2, 2), fc_part<D>(Wk, y2, 3)));
      lval[p] = __fsub_rn(sC[kk], __fmul_rn(0.5f, d2));
    }
    __syncthreads();
    // LSE_n over the point's candidates in component order
    if (tid < rows) {
      const uint32_t m = msk[tid], lt = (1u << lane) - 1u;
      auto pos_of = [&](int k) {
        int pos = offs[k] + __popc(cm[k * NW + warp] & lt);
        for (int w = 0; w < warp; ++w) pos += __popc(cm[k * NW + w]);
        return pos;
      };
      float mx = -INFINITY;
      for (uint32_t b = m; b; b &= b - 1u) mx = fmaxf(mx, lval[pos_of(__ffs(b) - 1)]);
      float sum = 0.f;
      for (uint32_t b = m; b; b &= b - 1u) sum += expf(lval[pos_of(__ffs(b) - 1)] - mx);
      const float l = sum > 0.f ? mx + logf(sum) : -INFINITY;
      if (!isfinite(l)) raise_status(a.st, GMM_ERR_NONFINITE);
      a.lse[r0 + tid] = l;
      ll += (double)l;
    }
  }
  __shared__ double red[kFcThreads / 32];
  ll = warp_sum(ll);
  __syncthreads();
  if (lane == 0) red[warp] = ll;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < kFcThreads / 32; ++w) s += red[w];
    a.ll_part[blockIdx.x] = s;
  }
}

template <int D>
struct FsShape {
  static constexpr int M = D / 4;
  static constexpr int NB = M * (M + 1) / 2;    // 4 x 4 blocks of the lower triangle
  static constexpr int YS = D + 4;              // padded chunk row
  static constexpr int G = kFsThreads / D;      // row groups of the chunk's first moment
  static_assert(NB <= kFsThreads, "one thread per block of the second moment");
};

// fc_stats shared memory: the component's W (padded rows) and mean, the
// chunk (y rows and g), chunk mean, first-moment partials, fp64 running sums
// and the mask tile's candidate list.
template <int D>
struct FsLayout {
  using S = FsShape<D>;
  static constexpr size_t W = 0;
  static constexpr size_t MU = W + sizeof(float) * fc_wfloats(D);
  static constexpr size_t YSO = MU + sizeof(float) * D;
  static constexpr size_t GCH = YSO + sizeof(float) * kFsChunk * S::YS;
  static constexpr size_t MC = GCH + sizeof(float) * kFsChunk;
  static constexpr size_t S1P = MC + sizeof(float) * D;
  static constexpr size_t SC = S1P + sizeof(float) * S::G * D;          // fp64 from here
  static constexpr size_t DM = SC + sizeof(double) * 4;
  static constexpr size_t S1R = DM + sizeof(double) * D;
  static constexpr size_t MR = S1R + sizeof(double) * D;
  static constexpr size_t M2R = MR + sizeof(double) * D;
  static constexpr size_t CAND = M2R + sizeof(double) * S::NB * 16;
  static constexpr size_t WCNT = CAND + sizeof(uint32_t) * kFsTile;
  static constexpr size_t BYTES = WCNT + sizeof(int) * (kFsThreads / 32);
};

template <int D, int XT>
__global__ void __launch_bounds__(kFsThreads, 2) fc_stats_kernel(const FcArgs a, int64_t rows_per_part) {
  using S = FsShape<D>;
  using L = FsLayout<D>;
  constexpr int YS = S::YS, F = 1 + D + D * (D + 1) / 2;
  extern __shared__ __align__(16) unsigned char smb[];
  float* sW = reinterpret_cast<float*>(smb + L::W);
  float* sMu = reinterpret_cast<float*>(smb + L::MU);
  float* ys = reinterpret_cast<float*>(smb + L::YSO);
  float* gch = reinterpret_cast<float*>(smb + L::GCH);
  float* mc = reinterpret_cast<float*>(smb + L::MC);
  float* s1p = reinterpret_cast<float*>(smb + L::S1P);
  double* sc = reinterpret_cast<double*>(smb + L::SC);  // S0 running, S0 chunk, factor
  double* dm = reinterpret_cast<double*>(smb + L::DM);
  double* s1r = reinterpret_cast<double*>(smb + L::S1R);
  double* mr = reinterpret_cast<double*>(smb + L::MR);
  double* m2r = reinterpret_cast<double*>(smb + L::M2R);
  uint32_t* cand = reinterpret_cast<uint32_t*>(smb + L::CAND);
  int* wcnt = reinterpret_cast<int*>(smb + L::WCNT);
  const int k = blockIdx.x, p = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r0 = (int64_t)p * rows_per_part;
  const int64_t r1 = min(a.N, r0 + rows_per_part);
  double* out = a.stat + ((size_t)p * a.K + k) * F;
  const float ck = __ldg(a.bias + k);
  if (r0 >= r1 || ck == -INFINITY) {
    if (!a.accumulate)
      for (int f = tid; f < F; f += kFsThreads) out[f] = 0.0;
    return;
  }
  for (int i = tid; i < D; i += kFsThreads) {
    stage_w<D>(sW, a.W + (size_t)k * D * D, i);
    sMu[i] = __ldg(a.mu + (size_t)k * D + i);
    s1r[i] = 0.0;
    mr[i] = 0.0;
  }
  for (int i = tid; i < S::NB * 16; i += kFsThreads) m2r[i] = 0.0;
  if (tid == 0) sc[0] = 0.0;
  __syncthreads();

  // One chunk of `fill` points: s0, mean and second moment about it in fp32,
  // then merged into the running fp64 sums.
  auto process_chunk = [&](int fill) {
    // s0 (warp 0, fixed order) and the first moment (G row groups, then in order)
    if (warp == 0) {
      float s = 0.f;
      for (int n = lane; n < fill; n += 32) s += gch[n];
      s = warp_sum(s);
      if (lane == 0) sc[1] = (double)s;
    }
    {
      const int d = tid % D, g = tid / D;
      float s = 0.f;
      for (int n = g; n < fill; n += S::G) s = fmaf(gch[n], ys[n * YS + d], s);
      s1p[g * D + d] = s;
    }
    __syncthreads();
    const double s0c = sc[1];
    if (!(s0c > 0.0)) {
      __syncthreads();
      return;
    }
    if (tid < D) {
      float s1 = 0.f;
      for (int g = 0; g < S::G; ++g) s1 += s1p[g * D + tid];
      const float m = s1 / (float)s0c;
      mc[tid] = m;
      dm[tid] = (double)m - mr[tid];
      s1r[tid] += (double)s1;
      mr[tid] = s1r[tid] / (sc[0] + s0c);
    }
    if (tid == 0) sc[2] = sc[0] > 0.0 ? sc[0] * s0c / (sc[0] + s0c) : 0.0;
    __syncthreads();
    if (tid == 0) sc[0] += s0c;
    if (tid < S::NB) {
      int A = (int)((sqrtf(8.f * tid + 1.f) - 1.f) * 0.5f);
      while ((A + 1) * (A + 2) / 2 <= tid) ++A;
      while (A * (A + 1) / 2 > tid) --A;
      const int B = tid - A * (A + 1) / 2;
      const float4 ma = *reinterpret_cast<const float4*>(mc + 4 * A);
      const float4 mb = *reinterpret_cast<const float4*>(mc + 4 * B);
      float2 acc[4][2];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);
#pragma unroll 4
      for (int n = 0; n < fill; ++n) {
        const float g = gch[n];
        const float4 ya = *reinterpret_cast<const float4*>(ys + n * YS + 4 * A);
        const float4 yb = *reinterpret_cast<const float4*>(ys + n * YS + 4 * B);
        const float2 b01 = sub2(make_float2(yb.x, yb.y), make_float2(mb.x, mb.y));
        const float2 b23 = sub2(make_float2(yb.z, yb.w), make_float2(mb.z, mb.w));
        const float ua[4] = {__fmul_rn(g, __fsub_rn(ya.x, ma.x)), __fmul_rn(g, __fsub_rn(ya.y, ma.y)),
                             __fmul_rn(g, __fsub_rn(ya.z, ma.z)), __fmul_rn(g, __fsub_rn(ya.w, ma.w))};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] = fma2(make_float2(ua[i], ua[i]), b01, acc[i][0]);
          acc[i][1] = fma2(make_float2(ua[i], ua[i]), b23, acc[i][1]);
        }
      }
      const double fac = sc[2];
      double* m2 = m2r + tid * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const double da = dm[4 * A + i];
        const float v[4] = {acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y};
#pragma unroll
        for (int j = 0; j < 4; ++j) m2[i * 4 + j] += (double)v[j] + fac * da * dm[4 * B + j];
      }
    }
    __syncthreads();
  };

  int fill = 0;
  for (int64_t t0 = r0; t0 < r1; t0 += kFsTile) {
    const int rows = (int)min((int64_t)kFsTile, r1 - t0);
    // the tile's candidates of component k, rows ascending
    const bool bit = tid < rows && ((__ldg(a.mask + t0 + tid) >> k) & 1u);
    const uint32_t bal = __ballot_sync(0xffffffffu, bit);
    if (lane == 0) wcnt[warp] = __popc(bal);
    __syncthreads();
    int base = 0, ncand = 0;
    for (int w = 0; w < kFsThreads / 32; ++w) {
      if (w < warp) base += wcnt[w];
      ncand += wcnt[w];
    }
    if (bit) cand[base + __popc(bal & ((1u << lane) - 1u))] = (uint32_t)(t0 + tid);
    __syncthreads();
    // groups of 64 candidates, four threads each (thread q: rows i = q mod 4)
    for (int g0 = 0; g0 < ncand; g0 += kFsThreads / 4) {
      const int ng = min(kFsThreads / 4, ncand - g0);
      if (fill + ng > kFsChunk) {
        process_chunk(fill);
        fill = 0;
      }
      const int pi = tid >> 2, q = tid & 3;
      const uint32_t row = cand[g0 + min(pi, ng - 1)];
      float2 y2[D / 2];
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 xv = load4<XT>(a.X, (size_t)row * D + 4 * c4);
        const float4 mv = *reinterpret_cast<const float4*>(sMu + 4 * c4);
        y2[2 * c4] = sub2(make_float2(xv.x, xv.y), make_float2(mv.x, mv.y));
        y2[2 * c4 + 1] = sub2(make_float2(xv.z, xv.w), make_float2(mv.z, mv.w));
      }
      const float part = fc_part<D>(sW, y2, q);
      // ((p0 + p1) + (p2 + p3)), as fc_lse
      const float u = __fadd_rn(part, __shfl_down_sync(0xffffffffu, part, 1));
      const float d2 = __fadd_rn(u, __shfl_down_sync(0xffffffffu, u, 2));
      const float l = __fsub_rn(ck, __fmul_rn(0.5f, d2));
      const float g = __shfl_sync(0xffffffffu, expf(l - __ldg(a.lse + row)), lane & ~3);
      if (pi < ng) {
        // thread q stores the 16-byte chunks q, q + 4, ... of y (the four
        // threads of a point write adjacent chunks: no bank conflict)
        float* yr = ys + (fill + pi) * YS;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          float2 v0 = y2[0], v1 = y2[1];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq)
            if (qq == q) { v0 = y2[2 * (4 * c + qq)]; v1 = y2[2 * (4 * c + qq) + 1]; }
          *reinterpret_cast<float4*>(yr + 4 * (4 * c + q)) = make_float4(v0.x, v0.y, v1.x, v1.y);
        }
        if (q == 0) gch[fill + pi] = g;
      }
      __syncthreads();
      fill += ng;
    }
  }
  if (fill > 0) process_chunk(fill);
  // the block's [S0 | S1 about mu | M2 about the block mean] into slot p
  // (the second moments first: merging reads the old first moments)
  const double S0n = sc[0];
  const double S0o = a.accumulate ? out[0] : 0.0;
  for (int e = tid; e < D * (D + 1) / 2; e += kFsThreads) {
    int aa = (int)((sqrtf(8.f * e + 1.f) - 1.f) * 0.5f);
    while ((aa + 1) * (aa + 2) / 2 <= e) ++aa;
    while (aa * (aa + 1) / 2 > e) --aa;
    const int bb = e - aa * (aa + 1) / 2;
    const int A = aa >> 2, B = bb >> 2;
    double v = m2r[(A * (A + 1) / 2 + B) * 16 + (aa & 3) * 4 + (bb & 3)];
    if (a.accumulate) {
      v += out[1 + D + e];
      if (S0o > 0.0 && S0n > 0.0) {
        const double da = s1r[aa] / S0n - out[1 + aa] / S0o;
        const double db = s1r[bb] / S0n - out[1 + bb] / S0o;
        v += da * db * (S0o * S0n / (S0o + S0n));
      }
    }
    out[1 + D + e] = v;
  }
  __syncthreads();
  for (int d = tid; d < D; d += kFsThreads) out[1 + d] = a.accumulate ? out[1 + d] + s1r[d] : s1r[d];
  __syncthreads();  // every thread has read out[0] before it changes
  if (tid == 0) out[0] = S0o + S0n;
}

// Masks without a screen: every component with a finite bias.
__global__ void fc_mask_all_kernel(uint32_t* mask, int64_t N, int K, const float* bias) {
  uint32_t valid = 0u;
  for (int k = 0; k < K; ++k)
    if (__ldg(bias + k) > -INFINITY) valid |= 1u << k;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < N;
       i += (int64_t)gridDim.x * blockDim.x)
    mask[i] = valid;
}

size_t fc_lse_smem(int D, int K) {
  return sizeof(float) * ((size_t)K * fc_wstride(D) + (size_t)K * D + kFcMaxK +
                          (size_t)kFcT * (D + 4) + (size_t)kFcT * K) +
         sizeof(uint32_t) * ((size_t)K * (kFcT / 32) + kFcT) + sizeof(int) * (kFcMaxK + 4) +
         (size_t)kFcT * K;
}

template <int D, int XT>
cudaError_t run_fc(const FcArgs& a, int parts, cudaStream_t s) {
  const size_t sl = fc_lse_smem(D, a.K);
  cudaError_t e = cudaFuncSetAttribute(fc_lse_kernel<D, XT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (a.N + kFcT - 1) / kFcT;
  {
    ProfScope prof("fc_lse_kernel", s);
    fc_lse_kernel<D, XT><<<(int)min((int64_t)kFcGrid, ntiles), kFcThreads, sl, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const size_t ss = FsLayout<D>::BYTES;
  e = cudaFuncSetAttribute(fc_stats_kernel<D, XT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)ss);
  if (e != cudaSuccess) return e;
  int64_t rpp = (a.N + parts - 1) / parts;
  rpp = (rpp + kFsTile - 1) / kFsTile * kFsTile;
  {
    ProfScope prof("fc_stats_kernel", s);
    fc_stats_kernel<D, XT><<<dim3(a.K, parts), kFsThreads, ss, s>>>(a, rpp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool fc_screen_eligible(int D, int K, int xdtype);
cudaError_t fc_screen(const void* X, int64_t N, int D, int K, const void* prepared,
                      uint32_t* mask, DeviceStatus* st, cudaStream_t s);

// Full covariance, D in {16, 32, 64}, at most 32 components whose W fit the
// shared memory of one fc_lse block.
bool fc_eligible(int D, int K, int cov) {
  if (cov != GMM_COV_FULL || !(D == 16 || D == 32 || D == 64) || K < 1 || K > kFcMaxK) return false;
  return fc_lse_smem(D, K) <= (size_t)200 * 1024;
}

// Log-likelihood partials fc_estep writes (fc_lse blocks).
int fc_ll_parts(int64_t N) {
  const int64_t nt = (N + kFcT - 1) / kFcT;
  return (int)(nt < kFcGrid ? nt : kFcGrid);
}

// The E-step and statistics of N rows: masks (those the tensor-core screen
// leaves when `screen` and it applies, else every component), LSE_n into lse, log-likelihood
// partials into ll_part[0 .. fc_ll_parts(N)), statistics into partial slots
// [0, parts) of stat (merged into them when accumulating).
cudaError_t fc_estep(const void* X, int xdtype, int64_t N, int D, int K, const void* prepared,
                     uint32_t* mask, bool screen, float* lse, double* ll_part, double* stat,
                     int parts, int accumulate, DeviceStatus* st, cudaStream_t s) {
  const PreparedLayout L = PreparedLayout::make(D, K, GMM_COV_FULL);
  FcArgs a;
  a.X = X; a.N = N; a.K = K;
  a.W = at<float>(prepared, L.off_prec);
  a.mu = at<float>(prepared, L.off_mu);
  a.bias = at<float>(prepared, L.off_c);
  a.mask = mask; a.lse = lse; a.ll_part = ll_part; a.stat = stat;
  a.accumulate = accumulate; a.st = st;
  if (screen && fc_screen_eligible(D, K, xdtype)) {
    const cudaError_t e = fc_screen(X, N, D, K, prepared, mask, st, s);
    if (e != cudaSuccess) return e;
  } else {
    ProfScope prof("fc_mask_kernel", s);
    fc_mask_all_kernel<<<304, 256, 0, s>>>(mask, N, K, a.bias);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto by_x = [&](auto dd) -> cudaError_t {
    constexpr int DD = decltype(dd)::value;
    if (xdtype == GMM_F16) return run_fc<DD, GMM_F16>(a, parts, s);
    if (xdtype == GMM_BF16) return run_fc<DD, GMM_BF16>(a, parts, s);
    return run_fc<DD, GMM_F32>(a, parts, s);
  };
  if (D == 16) return by_x(std::integral_constant<int, 16>{});
  if (D == 32) return by_x(std::integral_constant<int, 32>{});
  if (D == 64) return by_x(std::integral_constant<int, 64>{});
  return cudaErrorInvalidValue;
}

}  // namespace gmm
