// dense_rows.cu - exact log-sum-exp and sufficient statistics of the points
// whose candidate lists overflowed in the screening kernel.
//
// In the first EM iterations from theta_0 a point keeps tens to hundreds of
// components within 40 nats of its best log joint (every one of them is
// evaluated exactly: "low-precision GMM operator" notes, sec. 3.2 / 4.2,
// fp32 log-densities and log-sum-exp; Flash-GMM summary, Method: statistics
// of all components of a tile).  Evaluated one pair at a time inside the
// screening kernel, each pair would fetch its component's mean and inverse
// variances (1 KB at D = 128) from L2.  Here the screening kernel leaves such
// points with their candidate masks (one bit per component, the exact 40-nat
// window of the rigorous screen), and three kernels take them with the
// parameters staged in shared memory:
//   dense_lse     block (half a mask chunk: 64 components, partition): a
//                 warp per point, its four groups of eight lanes taking
//                 every fourth of the point's candidates, each evaluated in the
//                 centred fp32 form sum_d w_d (x_d - mu_d)^2 (lane: D/8
//                 dimensions, then a butterfly sum over the group), the
//                 groups' running max and sum (base 2) combined into the
//                 point's over the half chunk
//   dense_combine LSE_n from the chunks' (max, sum), the log-likelihood
//   dense_stats   block (group of 8192/D components, partition): a thread
//                 per (component, 16 dimensions: every eighth 16-byte chunk
//                 of the row at D = 128) keeps the component's sums
//                 s0, sum g (x - mu) and sum g v^2 (v = x - c, c a shift
//                 inside the component's new cluster: the block's first
//                 candidate point, moved once to its first point of
//                 responsibility >= 1/2) in registers over the block's points,
//                 g = exp(l - LSE_n) recomputed for every
//                 candidate; at the end they join the block's fp64 partial
//                 slot with the pairwise update of Chan, Golub and LeVeque.
// Every sum has a fixed order, so the results are the same on every run.
#include <math.h>

#include "gmm_internal.cuh"

namespace gmm {
namespace {

constexpr int kChunk = kTcChunk;  // components per mask chunk
constexpr int kThreads = 256;
constexpr int kCombineGrid = 256;  // blocks of the combine kernel (log-likelihood partials)
constexpr int kRowsPerTile = 64;   // points per tile of the statistics kernel

template <int XT>
__device__ __forceinline__ void load_x_vec(const void* X, size_t e0, int n, float* v) {
  if constexpr (XT == GMM_F32) {
    const float* p = static_cast<const float*>(X) + e0;
    if (n == 4) {
      const float4 q = __ldg(reinterpret_cast<const float4*>(p));
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
      const float2 q = __ldg(reinterpret_cast<const float2*>(p));
      v[0] = q.x; v[1] = q.y;
    }
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(X) + e0;
    uint32_t u[2];
    if (n == 4) {
      const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
      u[0] = q.x; u[1] = q.y;
    } else {
      u[0] = __ldg(reinterpret_cast<const unsigned int*>(p));
    }
    for (int i = 0; i < n / 2; ++i) {
      float2 f;
      if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
}

struct DenseArgs {
  const void* X;            // the slab's rows
  const uint32_t* rows;     // points left to these kernels (slab rows, ascending)
  const uint32_t* count;    // how many (on the device)
  int D, K, nch;
  const float* mu;          // prepared means [K][D]
  const float* prec;        // prepared inverse variances [K][D] (iso: [K])
  const float* bias;        // prepared log pi - log|S|/2 - (D/2) log 2 pi [K]
  bool iso;
  const uint32_t* cmask;    // [slab rows][nch][4] candidate masks
  float2* part;             // [points][2 nch] (max, sum) per half chunk, base 2
  float* lse;               // the slab's LSE_n
  double* ll_part;          // [kCombineGrid]
  double* stat;             // [P][K][1 + 2D] fp64 partials
  int accumulate;
  DeviceStatus* st;
};

// Components per block of the log-sum-exp kernel: half a mask chunk, so that
// three blocks fit an SM.
constexpr int kLseComps = kChunk / 2;

template <int D, int XT>
__global__ void __launch_bounds__(kThreads, 3) dense_lse_kernel(const DenseArgs a) {
  constexpr int CPL = D / 32;  // 4-dimension pieces per lane: lane g of a group of eight
                               // holds dimensions 4 (g + 8 i) .. + 3, i < CPL
  constexpr int RS = D + 4;    // padded table row (floats)
  extern __shared__ __align__(16) float smf[];
  float* s_mu = smf;                    // [64][RS]
  float* s_w = s_mu + kLseComps * RS;   // [64][RS]
  float* s_c = s_w + kLseComps * RS;    // [64]
  const uint32_t n = *a.count;
  if (n == 0) return;
  // block x: half hf of mask chunk j (mask words 2 hf, 2 hf + 1)
  const int j = blockIdx.x >> 1, hf = blockIdx.x & 1, P = gridDim.y;
  const int kc0 = j * kChunk + hf * kLseComps;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = lane >> 3, gl = lane & 7;
  for (int i = tid; i < kLseComps * D; i += kThreads) {
    const int kr = i / D, d = i % D, k = kc0 + kr;
    float m = 0.f, w = 0.f;
    if (k < a.K) {
      m = __ldg(a.mu + (size_t)k * D + d);
      w = a.iso ? __ldg(a.prec + k) : __ldg(a.prec + (size_t)k * D + d);
    }
    s_mu[kr * RS + d] = m;
    s_w[kr * RS + d] = w;
  }
  for (int i = tid; i < kLseComps; i += kThreads) {
    const int k = kc0 + i;
    s_c[i] = k < a.K ? __ldg(a.bias + k) : -INFINITY;
  }
  __syncthreads();
  // a warp per point; group q of eight lanes takes the point's candidates of
  // rank q, q + 4, q + 8, ... among the half chunk's (column order), so the
  // four groups' counts differ by at most one.  The log-sum-exp runs in
  // base 2 (values l log2(e)).  The next point's row,
  // masks and coordinates are requested before this one is evaluated.
  constexpr float kLog2e = 1.4426950408889634f;
  const uint32_t stride = (uint32_t)P * (kThreads / 32);
  uint32_t i = blockIdx.y * (kThreads / 32) + warp;
  float xn[CPL][4];
  uint2 mn = make_uint2(0u, 0u);
  auto fetch = [&](uint32_t ii) {
    const uint32_t row = a.rows[ii];
#pragma unroll
    for (int c = 0; c < CPL; ++c) load_x_vec<XT>(a.X, (size_t)row * D + 4 * (gl + 8 * c), 4, xn[c]);
    mn = __ldg(reinterpret_cast<const uint2*>(a.cmask + ((size_t)row * a.nch + j) * 4 + 2 * hf));
  };
  if (i < n) fetch(i);
  uint32_t npairs = 0;  // pairs this thread's group evaluated (counted by every lane)
  for (; i < n; i += stride) {
    float x[CPL][4];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int t = 0; t < 4; ++t) x[c][t] = xn[c][t];
    // the half chunk's candidates dealt over the groups by rank: group q
    // takes the candidates of rank q, q + 4, ... in column order
    uint64_t bits = ((uint64_t)mn.y << 32) | mn.x;
    if (i + stride < n) fetch(i + stride);
    const int ntot = __popcll(bits);
    const int steps = (ntot + 3) >> 2;  // the same for every group of the warp
    npairs += ntot > grp ? (uint32_t)((ntot - grp + 3) >> 2) : 0u;
#pragma unroll
    for (int q = 0; q < 3; ++q)
      if (q < grp) bits &= bits - 1u;
    float mx = -INFINITY, sum = 0.f;
    for (int st = 0; st < steps; ++st) {
      const int col = bits ? __ffsll((long long)bits) - 1 : -1;
#pragma unroll
      for (int q = 0; q < 4; ++q) bits &= bits - 1u;
      float acc = 0.f;
      if (col >= 0) {
        float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const float4 m4 = *reinterpret_cast<const float4*>(s_mu + col * RS + 4 * (gl + 8 * c));
          const float4 w4 = *reinterpret_cast<const float4*>(s_w + col * RS + 4 * (gl + 8 * c));
          const float2 u01 = sub2(make_float2(x[c][0], x[c][1]), make_float2(m4.x, m4.y));
          const float2 u23 = sub2(make_float2(x[c][2], x[c][3]), make_float2(m4.z, m4.w));
          a01 = fma2(mul2(u01, u01), make_float2(w4.x, w4.y), a01);
          a23 = fma2(mul2(u23, u23), make_float2(w4.z, w4.w), a23);
        }
        acc = (a01.x + a23.x) + (a01.y + a23.y);
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (col >= 0) {
        const float l2 = (s_c[col] - 0.5f * acc) * kLog2e;
        // the group's running log-sum-exp (base 2)
        if (l2 > mx) {
          sum = sum * exp2f(mx - l2) + 1.f;
          mx = l2;
        } else {
          sum += exp2f(l2 - mx);
        }
      }
    }
    // the four groups' partial sums, combined in group order
    float gm[4], gs[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      gm[q] = __shfl_sync(0xffffffffu, mx, q * 8);
      gs[q] = __shfl_sync(0xffffffffu, sum, q * 8);
    }
    if (lane == 0) {
      float M = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (gs[q] > 0.f) M = fmaxf(M, gm[q]);
      float S = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (gs[q] > 0.f) S += gs[q] * exp2f(gm[q] - M);
      a.part[(size_t)i * (2 * a.nch) + blockIdx.x] = make_float2(M, S);
    }
  }
  // the block's pair count: lane 8 g of each warp holds group g's
  __shared__ unsigned long long s_pairs;
  if (tid == 0) s_pairs = 0ull;
  __syncthreads();
  if (gl == 0 && npairs) atomicAdd(&s_pairs, (unsigned long long)npairs);
  __syncthreads();
  if (tid == 0 && s_pairs) atomicAdd(&a.st->cand_pairs, s_pairs);
}

__global__ void __launch_bounds__(kThreads) dense_combine_kernel(const DenseArgs a) {
  __shared__ double red[kThreads / 32];
  const uint32_t n = *a.count;
  double acc = 0.0;
  for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < n; i += gridDim.x * kThreads) {
    const float2* p = a.part + (size_t)i * (2 * a.nch);
    float M = -INFINITY;
    for (int j = 0; j < 2 * a.nch; ++j)
      if (p[j].y > 0.f) M = fmaxf(M, p[j].x);
    float S = 0.f;
    for (int j = 0; j < 2 * a.nch; ++j)
      if (p[j].y > 0.f) S += p[j].y * exp2f(p[j].x - M);
    // the partials are in base 2 (values l log2(e))
    const float l = (M + log2f(S)) * 0.6931471805599453f;
    if (!isfinite(l)) raise_status(a.st, GMM_ERR_NONFINITE);
    a.lse[a.rows[i]] = l;
    acc += (double)l;
  }
  acc = warp_sum(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double s = 0.0;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    a.ll_part[blockIdx.x] = s;
  }
}

// 16 dimensions per thread, D/16 threads per component, 512 threads: a block
// takes 8192/D components (64 at D = 128, 128 at D = 64).
constexpr int kStatThreads = 512;
template <int D>
struct DsShape {
  static constexpr int DPT = 16;
  static constexpr int TPC = D / DPT;
  static constexpr int CPB = kStatThreads / TPC;
  static constexpr int WPR = CPB / 32;  // mask words of a block's components per point
};

template <int D, int XT>
__global__ void __launch_bounds__(kStatThreads, 1) dense_stats_kernel(const DenseArgs a) {
  using SH = DsShape<D>;
  constexpr int DPT = SH::DPT, TPC = SH::TPC, CPB = SH::CPB, WPR = SH::WPR, F = 1 + 2 * D;
  constexpr int ESZ = XT == GMM_F32 ? 4 : 2;
  constexpr int ROWB = D * ESZ;
  constexpr int C16 = ROWB / 16;
  constexpr int TC16 = DPT * ESZ / 16;           // 16-byte chunks of a thread's dimensions
  constexpr int VPC = 16 / ESZ;                  // values per chunk
  constexpr int XPT = kRowsPerTile * C16 / kStatThreads;  // chunks of the tile per thread
  static_assert(XPT >= 1 && XPT * kStatThreads == kRowsPerTile * C16, "tile load split");
  __shared__ __align__(16) unsigned char xs[kRowsPerTile * ROWB];
  __shared__ float lse_t[kRowsPerTile];
  __shared__ uint32_t cm[CPB][kRowsPerTile / 32];
  const uint32_t n = *a.count;
  if (n == 0 && a.accumulate) return;  // nothing to add to the partials
  const int tid = threadIdx.x;
  const int kl = tid / TPC, h = tid % TPC;
  const int g = blockIdx.x, p = blockIdx.y, P = gridDim.y;
  const int k = g * CPB + kl;
  const bool kin = k < a.K;
  // thread h holds the 16-byte chunks h, h + TPC, h + 2 TPC, ... of a row, so
  // the TPC threads reading one row at a time touch TPC distinct chunks of
  // one span of 16 TPC bytes (at D = 128 a quarter warp reads 128 bytes with
  // no shared-memory bank conflict)
  auto dim_of = [&](int i) { return ((i / VPC) * TPC + h) * VPC + i % VPC; };
  const unsigned grp_mask = ((1u << TPC) - 1u) << ((tid & 31) & ~(TPC - 1));
  const float ck = kin ? __ldg(a.bias + k) : -INFINITY;
  constexpr int DP = DPT / 2;  // dimension pairs
  // the sums are taken about a shift inside the component's new cluster:
  // the first candidate point of the block (sf = its x - mu), so that a
  // component that moves far relative to its spread keeps its second moment
  // the means live in shared memory (float4 q of thread t at q * threads + t:
  // consecutive threads, consecutive 16 bytes), the rest in registers
  extern __shared__ float4 smu[];  // [DPT / 4][kStatThreads] means, then as many shifts
  float4* ssf = smu + (DPT / 4) * kStatThreads;
  float2 w[DP], s1[DP], s2[DP];
  float s0 = 0.f;
  bool shifted = false, heavy = false;
#pragma unroll
  for (int i = 0; i < DP; ++i) {
    const int d = dim_of(2 * i);  // pairs never straddle a chunk
    const float2 m = kin ? __ldg(reinterpret_cast<const float2*>(a.mu + (size_t)k * D + d)) : make_float2(0.f, 0.f);
    float* sm4 = reinterpret_cast<float*>(&smu[(i / 2) * kStatThreads + tid]) + 2 * (i & 1);
    sm4[0] = m.x;
    sm4[1] = m.y;
    if (!kin) w[i] = make_float2(0.f, 0.f);
    else if (a.iso) w[i] = make_float2(__ldg(a.prec + k), __ldg(a.prec + k));
    else w[i] = __ldg(reinterpret_cast<const float2*>(a.prec + (size_t)k * D + d));
    s1[i] = s2[i] = make_float2(0.f, 0.f);
  }
  // the block's components are mask words [wk0, wk0 + WPR) of mask chunk j
  const int j = (g * CPB) / kChunk, wk0 = ((g * CPB) % kChunk) / 32;
  const uint32_t ntiles = (n + kRowsPerTile - 1) / kRowsPerTile;
  // the next tile's data is fetched into registers while this one is used:
  // its rows of X (XPT chunks a thread), LSE and candidate masks
  uint4 xr[XPT];
  float lr = 0.f;
  uint32_t mr = 0u, rr = 0u;
  auto fetch = [&](uint32_t t) {
    const uint32_t i0 = t * kRowsPerTile;
    const int rows = (int)min((uint32_t)kRowsPerTile, n - i0);
#pragma unroll
    for (int c = 0; c < XPT; ++c) {
      const int e = tid + c * kStatThreads, r = e / C16, q = e % C16;
      xr[c] = r < rows ? __ldg(reinterpret_cast<const uint4*>(
                             static_cast<const unsigned char*>(a.X) +
                             (size_t)__ldg(a.rows + i0 + r) * ROWB) + q)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid < kRowsPerTile) {
      rr = tid < rows ? __ldg(a.rows + i0 + tid) : 0u;
      lr = tid < rows ? a.lse[rr] : 0.f;
    }
    if (tid < kRowsPerTile * WPR) {  // warp w: mask word w % WPR of rows 32 (w / WPR) + lane
      const int w = tid >> 5, r = (w / WPR) * 32 + (tid & 31), wq = w % WPR;
      mr = r < rows ? __ldg(a.cmask + ((size_t)__ldg(a.rows + i0 + r) * a.nch + j) * 4 + wk0 + wq)
                    : 0u;
    }
  };
  if ((uint32_t)p < ntiles) fetch(p);
  for (uint32_t t = p; t < ntiles; t += P) {
    __syncthreads();  // the previous tile's tables are no longer read
#pragma unroll
    for (int c = 0; c < XPT; ++c) {
      const int e = tid + c * kStatThreads, r = e / C16, q = e % C16;
      *reinterpret_cast<uint4*>(xs + r * ROWB + ((q ^ (r & 7)) << 4)) = xr[c];
    }
    if (tid < kRowsPerTile) lse_t[tid] = lr;
    // candidate masks, point-major -> component-major: a 32 x 32 bit
    // transpose per warp, one ballot per component
    if (tid < kRowsPerTile * WPR) {
      const int ln = tid & 31, w = tid >> 5;
      uint32_t mine = 0u;
#pragma unroll 8
      for (int b = 0; b < 32; ++b) {
        const uint32_t v = __ballot_sync(0xffffffffu, (mr >> b) & 1u);
        if (ln == b) mine = v;
      }
      cm[(w % WPR) * 32 + ln][w / WPR] = mine;
    }
    __syncthreads();
    if (t + P < ntiles) fetch(t + P);
    if (!kin || ck == -INFINITY) continue;
#pragma unroll 1
    for (int rw = 0; rw < kRowsPerTile / 32; ++rw) {
      uint32_t m = cm[kl][rw];
      while (m) {
        const int r = rw * 32 + __ffs(m) - 1;
        m &= m - 1u;
        float2 y[DP];  // x - mu
#pragma unroll
        for (int c16 = 0; c16 < TC16; ++c16) {
          const uint4 u = *reinterpret_cast<const uint4*>(
              xs + r * ROWB + (((c16 * TPC + h) ^ (r & 7)) << 4));
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
          if constexpr (XT == GMM_F32) {
            y[c16 * 2 + 0] = make_float2(__uint_as_float(w4[0]), __uint_as_float(w4[1]));
            y[c16 * 2 + 1] = make_float2(__uint_as_float(w4[2]), __uint_as_float(w4[3]));
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if constexpr (XT == GMM_F16) y[c16 * 4 + q] = __half22float2(*reinterpret_cast<const __half2*>(&w4[q]));
              else y[c16 * 4 + q] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[q]));
            }
          }
        }
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int i = 0; i < DP; i += 2) {
          const float4 m4 = smu[(i / 2) * kStatThreads + tid];
          y[i] = sub2(y[i], make_float2(m4.x, m4.y));
          y[i + 1] = sub2(y[i + 1], make_float2(m4.z, m4.w));
          acc[0] = fma2(mul2(y[i], y[i]), w[i], acc[0]);
          acc[1] = fma2(mul2(y[i + 1], y[i + 1]), w[i + 1], acc[1]);
        }
        float d2 = (acc[0].x + acc[1].x) + (acc[0].y + acc[1].y);
#pragma unroll
        for (int o = 1; o < TPC; o <<= 1) d2 += __shfl_xor_sync(grp_mask, d2, o);
        const float gm = exp2f((ck - 0.5f * d2 - lse_t[r]) * 1.4426950408889634f);
        const float2 g2 = make_float2(gm, gm);
        // the second moment is taken about a shift: the first candidate
        // point, moved once to the first point of responsibility >= 1/2 (the
        // sum so far carried over: S2 -= 2 d S1c - S0 d^2, with
        // S1c = S1 - S0 sf the first moment about the old shift); every
        // thread of the component sees the same points and g.  The first
        // moment stays about mu.
        if (!shifted || (!heavy && gm >= 0.5f)) {
#pragma unroll
          for (int i = 0; i < DP; i += 2) {
            const float4 old4 = ssf[(i / 2) * kStatThreads + tid];
            const float2 of0 = shifted ? make_float2(old4.x, old4.y) : make_float2(0.f, 0.f);
            const float2 of1 = shifted ? make_float2(old4.z, old4.w) : make_float2(0.f, 0.f);
            const float2 dl0 = sub2(y[i], of0), dl1 = sub2(y[i + 1], of1);
            const float2 s00 = make_float2(s0, s0);  // S0 before this point
            const float2 c0 = fma2(make_float2(-s0, -s0), of0, s1[i]);      // S1c
            const float2 c1 = fma2(make_float2(-s0, -s0), of1, s1[i + 1]);
            s2[i] = fma2(mul2(s00, dl0), dl0, fma2(make_float2(-2.f * dl0.x, -2.f * dl0.y), c0, s2[i]));
            s2[i + 1] = fma2(mul2(s00, dl1), dl1,
                             fma2(make_float2(-2.f * dl1.x, -2.f * dl1.y), c1, s2[i + 1]));
            ssf[(i / 2) * kStatThreads + tid] = make_float4(y[i].x, y[i].y, y[i + 1].x, y[i + 1].y);
          }
          heavy = gm >= 0.5f;
          shifted = true;
        }
        s0 += gm;
#pragma unroll
        for (int i = 0; i < DP; i += 2) {
          const float4 f4 = ssf[(i / 2) * kStatThreads + tid];
          const float2 v0 = sub2(y[i], make_float2(f4.x, f4.y));  // x - (mu + sf)
          const float2 v1 = sub2(y[i + 1], make_float2(f4.z, f4.w));
          s1[i] = fma2(g2, y[i], s1[i]);
          s1[i + 1] = fma2(g2, y[i + 1], s1[i + 1]);
          const float2 g0 = mul2(g2, v0), g1 = mul2(g2, v1);
          s2[i] = fma2(g0, v0, s2[i]);
          s2[i + 1] = fma2(g1, v1, s2[i + 1]);
        }
      }
    }
  }
  // this block's sums join slot p's fp64 partial [S0 | S1 about mu | M2 about the mean]
  if (kin) {
    double* o = a.stat + ((size_t)p * a.K + k) * F;
    const double b0 = (double)s0;
    const double S0o = a.accumulate ? o[0] : 0.0;
    const double S0 = S0o + b0;
#pragma unroll
    for (int i = 0; i < DPT; ++i) {
      const int d = dim_of(i);
      // the first moment about mu; the second about the shift, so the
      // moment about the block mean comes from the first moment about the
      // shift (S1 - S0 sf, in fp64)
      const double b1 = (double)((i & 1) ? s1[i / 2].y : s1[i / 2].x);
      const double q2 = (double)((i & 1) ? s2[i / 2].y : s2[i / 2].x);
      const float sfi = shifted ? reinterpret_cast<const float*>(&ssf[(i / 4) * kStatThreads + tid])[i & 3] : 0.f;
      const double c1 = b1 - b0 * (double)sfi;
      const double m2b = b0 > 0.0 ? q2 - c1 * c1 / b0 : 0.0;
      double S1 = b1, M2 = m2b;
      if (a.accumulate) {
        const double o1 = o[1 + d], om = o[1 + D + d];
        S1 = o1 + b1;
        M2 = om + m2b;
        if (S0o > 0.0 && b0 > 0.0) {
          const double dm = b1 / b0 - o1 / S0o;
          M2 += dm * dm * (S0o * b0 / S0);
        }
      }
      o[1 + d] = S1;
      o[1 + D + d] = M2;
    }
    __syncwarp(grp_mask);  // every thread of the component has read o[0] before it changes
    if (h == 0) o[0] = S0;
  }
}

template <int D, int XT>
cudaError_t run_dense(const DenseArgs& a, int pa, int pb, cudaStream_t s) {
  const size_t smem_a = sizeof(float) * ((size_t)2 * kLseComps * (D + 4) + kLseComps);
  cudaError_t e = cudaFuncSetAttribute(dense_lse_kernel<D, XT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_a);
  if (e != cudaSuccess) return e;
  {
    ProfScope prof("dense_lse_kernel", s);
    dense_lse_kernel<D, XT><<<dim3(2 * a.nch, pa), kThreads, smem_a, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope prof("dense_combine_kernel", s);
    dense_combine_kernel<<<kCombineGrid, kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope prof("dense_stats_kernel", s);
    const int ng = (a.K + DsShape<D>::CPB - 1) / DsShape<D>::CPB;
    const size_t smem_s = 2 * sizeof(float) * DsShape<D>::DPT * kStatThreads;
    if ((e = cudaFuncSetAttribute(dense_stats_kernel<D, XT>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_s)) != cudaSuccess)
      return e;
    dense_stats_kernel<D, XT><<<dim3(ng, pb), kStatThreads, smem_s, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

int dense_ll_parts() { return kCombineGrid; }

// Partitions of the dense statistics blocks (fixed by D and K: the order of
// the sums never depends on the device or on N).
int dense_stat_parts(int D, int K) {
  const int cpb = kStatThreads / (D / 16);
  const int ng = (K + cpb - 1) / cpb;
  const int p = 152 / ng;  // one wave of one block per SM
  return p < 1 ? 1 : p;
}

// The points rows[0 .. *count) of a slab (X: the slab's rows): LSE_n into
// lse, the log-likelihood into ll_part[0 .. dense_ll_parts()), statistics into
// partial slots [0, dense_stat_parts(D, K)) of stat.  part: scratch of
// (slab rows) x 2 nch float2.
cudaError_t dense_rows(const void* X, int xdtype, int D, int K, int cov, const void* prepared,
                       const uint32_t* rows, const uint32_t* count, const uint32_t* cmask,
                       float2* part, float* lse, double* ll_part, double* stat, int accumulate,
                       DeviceStatus* st, cudaStream_t s) {
  const PreparedLayout L = PreparedLayout::make(D, K, cov);
  DenseArgs a;
  a.X = X; a.rows = rows; a.count = count; a.D = D; a.K = K;
  a.nch = (K + kChunk - 1) / kChunk;
  a.mu = at<float>(prepared, L.off_mu);
  a.prec = at<float>(prepared, L.off_prec);
  a.bias = at<float>(prepared, L.off_c);
  a.iso = cov == GMM_COV_ISO;
  a.cmask = cmask; a.part = part; a.lse = lse; a.ll_part = ll_part; a.stat = stat;
  a.accumulate = accumulate; a.st = st;
  int pa = 152 * 3 / (2 * a.nch);  // one wave of three blocks per SM
  if (pa < 1) pa = 1;
  const int pb = dense_stat_parts(D, K);
  if (D == 128) {
    if (xdtype == GMM_F16) return run_dense<128, GMM_F16>(a, pa, pb, s);
    if (xdtype == GMM_BF16) return run_dense<128, GMM_BF16>(a, pa, pb, s);
    return run_dense<128, GMM_F32>(a, pa, pb, s);
  }
  if (D == 64) {
    if (xdtype == GMM_F16) return run_dense<64, GMM_F16>(a, pa, pb, s);
    if (xdtype == GMM_BF16) return run_dense<64, GMM_BF16>(a, pa, pb, s);
    return run_dense<64, GMM_F32>(a, pa, pb, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gmm
