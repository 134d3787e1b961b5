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
//             partition's candidates of the component queued in a ring and
//             taken in chunks of 256 points, their log joints recomputed a
//             thread per point (bit-identical to fc_lse), g = exp(l - LSE_n)
//             and y = x - mu; per chunk s0, the chunk mean and the second
//             moment about it in fp32 (a thread per register block of the
//             lower triangle and slice of the chunk's points, the slices
//             then summed in order), merged into the block's fp64 sums with
//             the pairwise update of Chan, Golub and LeVeque.  The partial
//             written per (partition, component) is
//             [S0 | S1 about mu | M2 about the block mean].
// Every sum has a fixed order, so the results are the same on every run.
#include <math.h>

#include <type_traits>

#include "gmm_internal.cuh"

namespace gmm {
namespace {

constexpr int kFcT = 128;          // points per fc_lse tile
constexpr int kFcThreads = 256;    // fc_lse block (two pairs a thread)
constexpr int kFcGrid = 152;       // fc_lse blocks (fixed: the log-likelihood partial count)
constexpr int kFsThreads = 256;    // fc_stats block
constexpr int kFsTile = 1024;      // partition points per mask tile (four per thread)
constexpr int kFsChunk = 256;      // candidate points per fp32 chunk
constexpr int kFsRing = 2048;      // pending candidates (ring)

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

// fc_part for two points under the same component: every W load serves
// both, the arithmetic of each is that of fc_part.
template <int D>
__device__ __forceinline__ void fc_part2(const float* __restrict__ Wk, const float2 (&ya)[D / 2],
                                         const float2 (&yb)[D / 2], int q, float& pa, float& pb) {
  constexpr int M = D / 4;
  float sa = 0.f, ca = 0.f, sb = 0.f, cb = 0.f;
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float* w = Wk + 8 * m * (m + 1) + 4 * q;
    float2 a0 = make_float2(0.f, 0.f), a1 = a0, b0 = a0, b1 = a0;
#pragma unroll
    for (int bk = 0; bk <= m; ++bk) {
      const float4 wv = *reinterpret_cast<const float4*>(w + 16 * bk);
      a0 = fma2(make_float2(wv.x, wv.y), ya[2 * bk], a0);
      a1 = fma2(make_float2(wv.z, wv.w), ya[2 * bk + 1], a1);
      b0 = fma2(make_float2(wv.x, wv.y), yb[2 * bk], b0);
      b1 = fma2(make_float2(wv.z, wv.w), yb[2 * bk + 1], b1);
    }
    const float za = __fadd_rn(__fadd_rn(a0.x, a0.y), __fadd_rn(a1.x, a1.y));
    const float zb = __fadd_rn(__fadd_rn(b0.x, b0.y), __fadd_rn(b1.x, b1.y));
    const float qa = __fmul_rn(za, za), qb = __fmul_rn(zb, zb);
    const float ta = __fadd_rn(sa, qa), tb = __fadd_rn(sb, qb);
    ca = __fadd_rn(ca, sa >= qa ? __fadd_rn(__fsub_rn(sa, ta), qa) : __fadd_rn(__fsub_rn(qa, ta), sa));
    cb = __fadd_rn(cb, sb >= qb ? __fadd_rn(__fsub_rn(sb, tb), qb) : __fadd_rn(__fsub_rn(qb, tb), sb));
    sa = ta;
    sb = tb;
  }
  pa = __fadd_rn(sa, ca);
  pb = __fadd_rn(sb, cb);
}

// Raw 16-byte chunk of stored coordinates -> four or eight floats.
template <int XT>
__device__ __forceinline__ void raw_to_float2(const uint4& u, float2* f) {
  if constexpr (XT == GMM_F32) {
    f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
    f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (XT == GMM_F16) f[q] = __half22float2(*reinterpret_cast<const __half2*>(&w[q]));
      else f[q] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q]));
    }
  }
}

// Stages the W of components [0, nk) (padded rows, zero beyond the diagonal)
// at dst with component stride `stride`, one element a thread per step.
template <int D>
__device__ __forceinline__ void stage_w(float* dst, int stride, const float* __restrict__ W, int nk,
                                        int tid, int nthreads) {
#pragma unroll 8
  for (int e = tid; e < nk * D * D; e += nthreads) {
    const int k = e / (D * D), i = (e / D) % D, j = e % D;
    const int m = i >> 2, q = i & 3;
    if (j < 4 * (m + 1))
      dst[k * stride + 8 * m * (m + 1) + 4 * q + 16 * (j >> 2) + (j & 3)] = j <= i ? __ldg(W + e) : 0.f;
  }
}

// The per-tile shared memory of fc_lse (one set per half block).
template <int D, int XT>
struct FlTile {
  static constexpr int RB = D * (XT == GMM_F32 ? 4 : 2);  // bytes of a stored row
  __host__ __device__ static size_t bytes(int K) {
    return (size_t)kFcT * RB + sizeof(float) * (size_t)kFcT * K +
           sizeof(uint32_t) * ((size_t)K * (kFcT / 32) + kFcT) + sizeof(int) * (2 * kFcMaxK + 4) +
           (((size_t)kFcT * K + 15) / 16) * 16;
  }
};

// NH independent halves of the block (NH = 2: warps 0-3 and 4-7) take
// alternate tiles with their own tile tables and named barriers, so one half
// evaluates while the other waits at a barrier; W, the means and biases are
// shared.  With NH = 1 the next tile's rows are prefetched into registers.
template <int D, int XT, int NH>
__global__ void __launch_bounds__(kFcThreads, 1) fc_lse_kernel(const FcArgs a) {
  constexpr int WS = fc_wstride(D), NW = kFcT / 32;
  constexpr int TH = kFcThreads / NH;          // threads of a half
  constexpr int ESZ = XT == GMM_F32 ? 4 : 2;
  constexpr int RB = D * ESZ;                 // bytes of a stored row
  constexpr int C16 = RB / 16;                // its 16-byte chunks
  constexpr int VPC = 16 / ESZ;               // coordinates per chunk
  constexpr int XPT = kFcT * C16 / TH;        // chunks of the tile a thread loads
  constexpr bool PREFETCH = NH == 1;
  static_assert(TH >= kFcT && XPT * TH == kFcT * C16, "tile split");
  extern __shared__ __align__(16) float sm[];
  const int K = a.K;
  float* sW = sm;                                    // K * WS
  float* sMu = sW + K * WS;                          // K * D
  float* sC = sMu + K * D;                           // kFcMaxK
  const int tid0 = threadIdx.x, half = tid0 / TH, tid = tid0 % TH;
  const int lane = tid & 31, warp = tid >> 5;        // within the half
  unsigned char* xs = reinterpret_cast<unsigned char*>(sC + kFcMaxK) + half * FlTile<D, XT>::bytes(K);
  float* lval = reinterpret_cast<float*>(xs + kFcT * RB);             // kFcT * K
  uint32_t* cm = reinterpret_cast<uint32_t*>(lval + kFcT * K);  // K * NW
  uint32_t* msk = cm + K * NW;                       // kFcT
  int* offs = reinterpret_cast<int*>(msk + kFcT);    // kFcMaxK + 1: pairs
  int* toff = offs + kFcMaxK + 1;                    // kFcMaxK + 1: tasks (two pairs each)
  uint8_t* prow = reinterpret_cast<uint8_t*>(toff + kFcMaxK + 3);  // kFcT * K
  auto hsync = [&]() {
    if constexpr (NH == 1) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"r"(1 + half), "r"(TH) : "memory");
  };
  stage_w<D>(sW, WS, a.W, K, tid0, kFcThreads);
  for (int e = tid0; e < K * D; e += kFcThreads) sMu[e] = __ldg(a.mu + e);
  for (int k = tid0; k < kFcMaxK; k += kFcThreads) sC[k] = k < K ? __ldg(a.bias + k) : -INFINITY;
  __syncthreads();
  uint32_t valid = 0u;
  for (int k = 0; k < K; ++k)
    if (sC[k] > -INFINITY) valid |= 1u << k;
  const int64_t ntiles = (a.N + kFcT - 1) / kFcT;
  double ll = 0.0;
  unsigned long long npairs = 0;  // pairs of this half's tiles (its thread 0)
  uint32_t mnext = 0u;
  uint4 xnext[PREFETCH ? XPT : 1];
  auto load_x = [&](int64_t t, uint4* dst, bool to_smem) {
    const int64_t r0 = t * kFcT;
    const int rows = (int)min((int64_t)kFcT, a.N - r0);
#pragma unroll
    for (int c = 0; c < XPT; ++c) {
      const int e = tid + c * TH, r = e / C16, q = e % C16;
      const uint4 v = r < rows ? __ldg(reinterpret_cast<const uint4*>(
                                     static_cast<const unsigned char*>(a.X) + (size_t)(r0 + r) * RB) + q)
                               : make_uint4(0u, 0u, 0u, 0u);
      if (to_smem) reinterpret_cast<uint4*>(xs)[e] = v;
      else dst[c] = v;
    }
  };
  auto load_mask = [&](int64_t t) {
    const int64_t r0 = t * kFcT;
    const int rows = (int)min((int64_t)kFcT, a.N - r0);
    return tid < rows && tid < kFcT ? __ldg(a.mask + r0 + tid) : 0u;
  };
  const int64_t t_first = (int64_t)blockIdx.x * NH + half, t_step = (int64_t)gridDim.x * NH;
  if constexpr (PREFETCH) {
    if (t_first < ntiles) {
      mnext = load_mask(t_first);
      load_x(t_first, xnext, false);
    }
  }
  for (int64_t t = t_first; t < ntiles; t += t_step) {
    const int64_t r0 = t * kFcT;
    const int rows = (int)min((int64_t)kFcT, a.N - r0);
    hsync();  // the previous tile's tables are no longer read
    // masks (component-major bit columns by ballot) and the rows of X
    if constexpr (!PREFETCH) mnext = load_mask(t);
    if (tid < kFcT) {
      const uint32_t m = mnext & valid;
      msk[tid] = m;
      for (int k = 0; k < K; ++k) {
        const uint32_t b = __ballot_sync(0xffffffffu, (m >> k) & 1u);
        if (lane == 0) cm[k * NW + warp] = b;
      }
    }
    if constexpr (PREFETCH) {
#pragma unroll
      for (int c = 0; c < XPT; ++c) reinterpret_cast<uint4*>(xs)[tid + c * TH] = xnext[c];
      if (t + t_step < ntiles) {
        mnext = load_mask(t + t_step);
        load_x(t + t_step, xnext, false);
      }
    } else {
      load_x(t, nullptr, true);
    }
    hsync();
    // pair and task offsets per component (a task: two pairs of a component)
    if (warp == 0) {
      int cnt = 0;
      if (lane < K)
        for (int w = 0; w < NW; ++w) cnt += __popc(cm[lane * NW + w]);
      int inc = cnt, tin = (cnt + 1) >> 1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        const int v = __shfl_up_sync(0xffffffffu, tin, o);
        if (lane >= o) { inc += u; tin += v; }
      }
      if (lane < K) { offs[lane + 1] = inc; toff[lane + 1] = tin; }
      if (lane == 0) { offs[0] = 0; toff[0] = 0; }
    }
    hsync();
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
    hsync();
    const int nt = toff[K];
    if (tid == 0) npairs += (uint32_t)offs[K];
    int kk = 0;
    for (int tk = tid; tk < nt; tk += TH) {
      while (toff[kk + 1] <= tk) ++kk;
      const int p = offs[kk] + 2 * (tk - toff[kk]);
      const bool two = p + 1 < offs[kk + 1];
      const int ra = prow[p], rb = prow[two ? p + 1 : p];
      float2 ya[D / 2], yb[D / 2];
#pragma unroll
      for (int c = 0; c < C16; ++c) {
        float2 fa[VPC / 2], fb[VPC / 2];
        raw_to_float2<XT>(*reinterpret_cast<const uint4*>(xs + ra * RB + 16 * c), fa);
        raw_to_float2<XT>(*reinterpret_cast<const uint4*>(xs + rb * RB + 16 * c), fb);
#pragma unroll
        for (int v = 0; v < VPC / 2; ++v) {
          const float2 mv = *reinterpret_cast<const float2*>(sMu + kk * D + c * VPC + 2 * v);
          ya[c * (VPC / 2) + v] = sub2(fa[v], mv);
          yb[c * (VPC / 2) + v] = sub2(fb[v], mv);
        }
      }
      const float* Wk = sW + kk * WS;
      float pa[4], pb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) fc_part2<D>(Wk, ya, yb, q, pa[q], pb[q]);
      const float da = __fadd_rn(__fadd_rn(pa[0], pa[1]), __fadd_rn(pa[2], pa[3]));
      const float db = __fadd_rn(__fadd_rn(pb[0], pb[1]), __fadd_rn(pb[2], pb[3]));
      lval[p] = __fsub_rn(sC[kk], __fmul_rn(0.5f, da));
      if (two) lval[p + 1] = __fsub_rn(sC[kk], __fmul_rn(0.5f, db));
    }
    hsync();
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
  // the block's log-likelihood: warps in order (both halves), fixed
  __shared__ double red[kFcThreads / 32];
  ll = warp_sum(ll);
  __syncthreads();
  if ((tid0 & 31) == 0) red[tid0 >> 5] = ll;
  __syncthreads();
  if (tid0 == 0) {
    double s = 0.0;
    for (int w = 0; w < kFcThreads / 32; ++w) s += red[w];
    a.ll_part[blockIdx.x] = s;
  }
  if (tid == 0 && npairs) atomicAdd(&a.st->cand_pairs, npairs);
}

template <int D>
struct FsShape {
  static constexpr int BE = D >= 64 ? 8 : 4;     // edge of a second-moment register block
  static constexpr int MB = D / BE;
  static constexpr int NBB = MB * (MB + 1) / 2;  // blocks of the lower triangle
  static constexpr int NS = kFsThreads / NBB;    // slices of the chunk's points
  static constexpr int BE2 = BE * BE;
  static constexpr int PS = BE2 + 4;             // padded stride of a slice partial
  static constexpr int YS = D + 4;               // padded chunk row
  static constexpr int G = kFsThreads / D;       // row groups of the chunk's first moment
  static_assert(NS >= 1, "one thread per block and slice");
  static_assert(NS * NBB * PS <= kFsChunk * YS, "slice partials fit in the chunk rows");
};

// fc_stats shared memory: the component's W (padded rows) and mean, the
// chunk (y rows and g), chunk mean, first-moment partials, fp64 running sums
// and the ring of pending candidates.
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
  static constexpr size_t CAND = M2R + sizeof(double) * S::NBB * S::BE2;
  static constexpr size_t WCNT = CAND + sizeof(uint32_t) * kFsRing;
  static constexpr size_t BYTES = WCNT + sizeof(int) * (kFsThreads / 32);
  static_assert(kFsTile == 4 * kFsThreads, "four mask words a thread");
  static_assert(kFsRing >= kFsChunk + kFsTile && (kFsRing & (kFsRing - 1)) == 0,
                "a power-of-two ring holding a tile past a partial chunk");
};

template <int D, int XT>
__global__ void __launch_bounds__(kFsThreads, 2) fc_stats_kernel(const FcArgs a, int64_t rows_per_part) {
  using S = FsShape<D>;
  using L = FsLayout<D>;
  constexpr int YS = S::YS, BE = S::BE, BE2 = S::BE2, F = 1 + D + D * (D + 1) / 2;
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
  stage_w<D>(sW, 0, a.W + (size_t)k * D * D, 1, tid, kFsThreads);
  for (int i = tid; i < D; i += kFsThreads) {
    sMu[i] = __ldg(a.mu + (size_t)k * D + i);
    s1r[i] = 0.0;
    mr[i] = 0.0;
  }
  for (int i = tid; i < S::NBB * BE2; i += kFsThreads) m2r[i] = 0.0;
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
    // thread (block bi, slice sl): block bi = (A, B) of the lower triangle over
    // the points sl, sl + NS, ...; g (y_a - m_a) (y_b - m_b) in fp32 about the
    // chunk mean m
    const int bi = tid % S::NBB, sl = tid / S::NBB;
    int A = 0;
    while ((A + 1) * (A + 2) / 2 <= bi) ++A;
    const int B = bi - A * (A + 1) / 2;
    float2 acc[BE][BE / 2];
#pragma unroll
    for (int i = 0; i < BE; ++i)
#pragma unroll
      for (int j = 0; j < BE / 2; ++j) acc[i][j] = make_float2(0.f, 0.f);
    if (sl < S::NS) {
      float2 ma[BE / 2], mb[BE / 2];
#pragma unroll
      for (int v = 0; v < BE / 2; ++v) {
        ma[v] = *reinterpret_cast<const float2*>(mc + BE * A + 2 * v);
        mb[v] = *reinterpret_cast<const float2*>(mc + BE * B + 2 * v);
      }
#pragma unroll 1
      for (int n = sl; n < fill; n += S::NS) {
        const float g = gch[n];
        float2 ca[BE / 2], cb[BE / 2];
#pragma unroll
        for (int v = 0; v < BE / 4; ++v) {
          const float4 qa = *reinterpret_cast<const float4*>(ys + n * YS + BE * A + 4 * v);
          const float4 qb = *reinterpret_cast<const float4*>(ys + n * YS + BE * B + 4 * v);
          ca[2 * v] = sub2(make_float2(qa.x, qa.y), ma[2 * v]);
          ca[2 * v + 1] = sub2(make_float2(qa.z, qa.w), ma[2 * v + 1]);
          cb[2 * v] = sub2(make_float2(qb.x, qb.y), mb[2 * v]);
          cb[2 * v + 1] = sub2(make_float2(qb.z, qb.w), mb[2 * v + 1]);
        }
#pragma unroll
        for (int i = 0; i < BE; ++i) {
          const float u = __fmul_rn(g, (i & 1) ? ca[i / 2].y : ca[i / 2].x);
#pragma unroll
          for (int j = 0; j < BE / 2; ++j) acc[i][j] = fma2(make_float2(u, u), cb[j], acc[i][j]);
        }
      }
    }
    __syncthreads();  // every read of the rows is done: the slice partials go there
    float* part = ys;
    if (sl < S::NS) {
      float* pp = part + (sl * S::NBB + bi) * S::PS;
#pragma unroll
      for (int i = 0; i < BE; ++i)
#pragma unroll
        for (int j = 0; j < BE / 4; ++j)
          *reinterpret_cast<float4*>(pp + i * BE + 4 * j) =
              make_float4(acc[i][2 * j].x, acc[i][2 * j].y, acc[i][2 * j + 1].x, acc[i][2 * j + 1].y);
    }
    __syncthreads();
    // the slices summed in order, merged into the fp64 sums
    const double fac = sc[2];
    for (int e = tid; e < S::NBB * BE2; e += kFsThreads) {
      const int bb = e / BE2, r = e % BE2;
      float v = 0.f;
      for (int q = 0; q < S::NS; ++q) v = __fadd_rn(v, part[(q * S::NBB + bb) * S::PS + r]);
      int Ae = 0;
      while ((Ae + 1) * (Ae + 2) / 2 <= bb) ++Ae;
      const int Be = bb - Ae * (Ae + 1) / 2;
      m2r[e] += (double)v + fac * dm[BE * Ae + r / BE] * dm[BE * Be + r % BE];
    }
    __syncthreads();
  };

  // One chunk: a thread per candidate of the ring from `head`: y = x - mu,
  // the exact log joint (bit-identical to fc_lse) and g = exp(l - LSE_n).
  auto solve = [&](uint32_t head, int ng) {
    if (tid < ng) {
      const uint32_t row = cand[(head + tid) & (kFsRing - 1)];
      const float lr = __ldg(a.lse + row);
      float2 y2[D / 2];
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4) {
        const float4 xv = load4<XT>(a.X, (size_t)row * D + 4 * c4);
        const float4 mv = *reinterpret_cast<const float4*>(sMu + 4 * c4);
        y2[2 * c4] = sub2(make_float2(xv.x, xv.y), make_float2(mv.x, mv.y));
        y2[2 * c4 + 1] = sub2(make_float2(xv.z, xv.w), make_float2(mv.z, mv.w));
      }
      // ((p0 + p1) + (p2 + p3)), as fc_lse
      const float d2 = __fadd_rn(__fadd_rn(fc_part<D>(sW, y2, 0), fc_part<D>(sW, y2, 1)),
                                 __fadd_rn(fc_part<D>(sW, y2, 2), fc_part<D>(sW, y2, 3)));
      const float l = __fsub_rn(ck, __fmul_rn(0.5f, d2));
      float* yr = ys + tid * YS;
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4)
        *reinterpret_cast<float4*>(yr + 4 * c4) =
            make_float4(y2[2 * c4].x, y2[2 * c4].y, y2[2 * c4 + 1].x, y2[2 * c4 + 1].y);
      gch[tid] = expf(l - lr);
    }
    __syncthreads();
    process_chunk(ng);
  };

  // Mask tiles of kFsTile points, four consecutive points a thread (the next
  // tile's masks are requested before this one is used); the candidates of k
  // appended to the ring in point order; every full chunk of the ring taken
  // at once, so each chunk is evaluated by all the block's threads.
  uint32_t head = 0u, tail = 0u;
  uint4 mnext = make_uint4(0u, 0u, 0u, 0u);
  auto fetch = [&](int64_t t0) {
    const int64_t rr = t0 + 4 * tid;
    if (rr + 3 < r1) {
      mnext = __ldg(reinterpret_cast<const uint4*>(a.mask + rr));
    } else {
      mnext.x = rr < r1 ? __ldg(a.mask + rr) : 0u;
      mnext.y = rr + 1 < r1 ? __ldg(a.mask + rr + 1) : 0u;
      mnext.z = rr + 2 < r1 ? __ldg(a.mask + rr + 2) : 0u;
      mnext.w = rr + 3 < r1 ? __ldg(a.mask + rr + 3) : 0u;
    }
  };
  if (r0 < r1) fetch(r0);
  for (int64_t t0 = r0; t0 < r1; t0 += kFsTile) {
    const uint32_t bits = ((mnext.x >> k) & 1u) | (((mnext.y >> k) & 1u) << 1) |
                          (((mnext.z >> k) & 1u) << 2) | (((mnext.w >> k) & 1u) << 3);
    if (t0 + kFsTile < r1) fetch(t0 + kFsTile);
    // block-wide exclusive count of the candidates before this thread's points
    const int cnt = __popc(bits);
    int inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) wcnt[warp] = inc;
    __syncthreads();
    int base = inc - cnt, ncand = 0;
    for (int w = 0; w < kFsThreads / 32; ++w) {
      if (w < warp) base += wcnt[w];
      ncand += wcnt[w];
    }
    // fewer than kFsChunk are pending, so the tile's at most kFsTile fit
    for (uint32_t b = bits; b; b &= b - 1u)
      cand[(tail + (uint32_t)base++) & (kFsRing - 1)] = (uint32_t)(t0 + 4 * tid + __ffs(b) - 1);
    __syncthreads();
    tail += (uint32_t)ncand;
    for (; tail - head >= (uint32_t)kFsChunk; head += kFsChunk) solve(head, kFsChunk);
  }
  if (tail != head) solve(head, (int)(tail - head));
  // the block's [S0 | S1 about mu | M2 about the block mean] into slot p
  // (the second moments first: merging reads the old first moments)
  const double S0n = sc[0];
  const double S0o = a.accumulate ? out[0] : 0.0;
  for (int e = tid; e < D * (D + 1) / 2; e += kFsThreads) {
    int aa = (int)((sqrtf(8.f * e + 1.f) - 1.f) * 0.5f);
    while ((aa + 1) * (aa + 2) / 2 <= e) ++aa;
    while (aa * (aa + 1) / 2 > e) --aa;
    const int bb = e - aa * (aa + 1) / 2;
    const int A = aa / BE, B = bb / BE;
    double v = m2r[(A * (A + 1) / 2 + B) * BE2 + (aa % BE) * BE + bb % BE];
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

// fc_lse shared memory: W, means, biases and nh sets of tile tables.
size_t fc_lse_smem(int D, int K, int xdtype, int nh) {
  const size_t rb = (size_t)D * (xdtype == GMM_F32 ? 4 : 2);
  const size_t tile = (size_t)kFcT * rb + sizeof(float) * (size_t)kFcT * K +
                      sizeof(uint32_t) * ((size_t)K * (kFcT / 32) + kFcT) +
                      sizeof(int) * (2 * kFcMaxK + 4) + (((size_t)kFcT * K + 15) / 16) * 16;
  return sizeof(float) * ((size_t)K * fc_wstride(D) + (size_t)K * D + kFcMaxK) + nh * tile;
}

template <int D, int XT>
cudaError_t run_fc(const FcArgs& a, int parts, cudaStream_t s) {
  // two half blocks when their tile tables fit next to W
  const bool two = fc_lse_smem(D, a.K, XT, 2) <= (size_t)220 * 1024;
  const size_t sl = fc_lse_smem(D, a.K, XT, two ? 2 : 1);
  auto kern = two ? fc_lse_kernel<D, XT, 2> : fc_lse_kernel<D, XT, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl);
  if (e != cudaSuccess) return e;
  const int64_t ntiles = (a.N + kFcT - 1) / kFcT;
  {
    ProfScope prof("fc_lse_kernel", s);
    kern<<<(int)min((int64_t)kFcGrid, ntiles), kFcThreads, sl, s>>>(a);
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
  return fc_lse_smem(D, K, GMM_F32, 1) <= (size_t)200 * 1024;
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
