// chunk_stats.cu - sufficient statistics of the tensor-core E-step, one
// thread block per (group of 8192/D components, partition of point tiles)
// (Flash-GMM summary, Method: online s0 = sum g, s1 = sum g x, s2 = sum g x^2
// per tile, no N x K matrix; "low-precision GMM operator" notes, sec. 3.1:
// block partials, then a global reduction).
//
// The screening kernel leaves, per 128-point tile, records {key, l}: the
// exact fp32 log joint l of every (point, component) pair it evaluated (all
// pairs within 40 nats of the point's best; every other pair carries less
// than 4.3e-18 of the point's responsibility), and LSE_n of every point.  A
// record flagged "single" is a point's only candidate: responsibility 1, its
// log joint not evaluated, so its log-likelihood term is computed here.  A
// tile whose records did not fit its buffer is taken densely: every pair of
// the tile and component group is evaluated exactly here.
//
// Thread (component kl of the group, part h of its dimensions: 32 each) keeps its
// component's sums in registers over the block's tiles: s0, the first and
// second moments about the input mean c_k = mu_k (rounded to bf16), in fp32,
// each tile's rows in ascending order (the records are placed into a dense
// per-tile table first, so the order never depends on how they were
// written).  At the end of the slab the block's sums join the fp64 partial
// [S0 | S1 about c | M2 about the partial's mean] of its slot with the
// pairwise update of Chan, Golub and LeVeque.  Fixed order throughout: the
// same bits on every run.
#include <math.h>

#include "gmm_internal.cuh"

namespace gmm {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 256;

// 32 dimensions per thread, D/32 threads per component, 256 threads: a block
// takes 8192/D components (128 at D = 64, 64 at D = 128).
template <int D>
struct CsShape {
  static constexpr int TPC = D / 32;         // threads per component
  static constexpr int DPT = 32;              // dimensions per thread
  static constexpr int THREADS = kThreads;
  static constexpr int CPB = kThreads / TPC;  // components per block
};

// Shared-memory layout: X tile (stored type, 16-byte chunks XOR-swizzled by
// row), the dense table of log joints [128 rows][128 components] (dense
// tiles: the group's precisions [components][D + 1] instead), LSE of the rows,
// row masks per component (records, singles).
template <int D, int XT>
struct CsSmem {
  static constexpr int CPB = CsShape<D>::CPB;
  static constexpr int ESZ = XT == GMM_F32 ? 4 : 2;
  static constexpr int ROWB = D * ESZ;
  static constexpr int OFF_X = 0;
  static constexpr int OFF_LV = OFF_X + kBM * ROWB;
  static constexpr int LV_BYTES = (kBM * CPB > CPB * (D + 1) ? kBM * CPB : CPB * (D + 1)) * 4;
  static constexpr int OFF_LSE = OFF_LV + LV_BYTES;
  static constexpr int OFF_MASK = OFF_LSE + kBM * 4;
  static constexpr int OFF_SMASK = OFF_MASK + CPB * 4 * 4;
  static constexpr int OFF_RED = OFF_SMASK + CPB * 4 * 4;
  static constexpr int BYTES = OFF_RED + 32 * 8;
};

// byte offset of 16-byte chunk c16 of row r in the swizzled tile
template <int ROWB>
__device__ __forceinline__ int xs_off(int r, int c16) {
  return r * ROWB + ((c16 ^ (r & 7)) << 4);
}

struct CsArgs {
  const void* X;          // slab rows of X
  int64_t N;              // rows in the slab
  int K;
  const void* prepared;
  PreparedLayout L;
  const float* lse;       // LSE_n of the slab's rows
  const uint2* recs;      // [tiles][rec_cap]
  const uint32_t* tile_cnt;
  int rec_cap;
  double* part;           // [P][K][F] fp64 partials
  int accumulate;         // continue the partials of earlier slabs
  double* ll_part;        // [gridDim.x * gridDim.y]: single-candidate log-likelihood
};

template <int D, int XT>
__global__ void __launch_bounds__(CsShape<D>::THREADS, 1) chunk_stats_kernel(const CsArgs a) {
  using SH = CsShape<D>;
  using SM = CsSmem<D, XT>;
  constexpr int TPC = SH::TPC, DPT = SH::DPT, CPB = SH::CPB, F = 1 + 2 * D;
  constexpr int ROWB = SM::ROWB, ESZ = SM::ESZ;
  constexpr int C16 = ROWB / 16;            // 16-byte chunks per row
  constexpr int TC16 = DPT * ESZ / 16;      // chunks per thread's dimensions
  extern __shared__ __align__(128) unsigned char sm[];
  unsigned char* xs = sm + SM::OFF_X;
  float* lv = (float*)(sm + SM::OFF_LV);
  float* lse_s = (float*)(sm + SM::OFF_LSE);
  uint32_t* mask = (uint32_t*)(sm + SM::OFF_MASK);
  uint32_t* smask = (uint32_t*)(sm + SM::OFF_SMASK);
  double* red = (double*)(sm + SM::OFF_RED);

  const int tid = threadIdx.x;
  const int kl = tid / TPC, h = tid % TPC;
  const int c = blockIdx.x, p = blockIdx.y, P = gridDim.y;
  const int k = c * CPB + kl;
  const bool kin = k < a.K;
  const int d0 = h * DPT;
  const float* g_mu = at<float>(a.prepared, a.L.off_mu);
  const float* g_prec = at<float>(a.prepared, a.L.off_prec);
  const float* g_c = at<float>(a.prepared, a.L.off_c);
  const bool iso = a.L.cov == GMM_COV_ISO;
  const float ck = kin ? __ldg(g_c + k) : -INFINITY;
  const bool live = kin && ck != -INFINITY;
  // the lanes that share this thread's component
  const unsigned pair_mask = ((1u << TPC) - 1u) << ((tid & 31) & ~(TPC - 1));

  // The sums are taken about c' = the mean rounded to bf16 (held packed,
  // two dimensions a register); the merge below moves the first moment to
  // the fp32 mean, and the second moment about the block's own mean does not
  // depend on the centre.
  __nv_bfloat162 cen2[DPT / 2];
  float s1[DPT], s2[DPT], s0 = 0.f;
#pragma unroll
  for (int i = 0; i < DPT / 2; ++i) {
    const float m0 = kin ? __ldg(g_mu + (size_t)k * D + d0 + 2 * i) : 0.f;
    const float m1 = kin ? __ldg(g_mu + (size_t)k * D + d0 + 2 * i + 1) : 0.f;
    cen2[i] = __floats2bfloat162_rn(m0, m1);
  }
#pragma unroll
  for (int i = 0; i < DPT; ++i) s1[i] = s2[i] = 0.f;
  auto cen = [&](int dd) -> float {
    const float2 f = __bfloat1622float2(cen2[dd >> 1]);
    return (dd & 1) ? f.y : f.x;
  };
  double ll_acc = 0.0;

  // squared Mahalanobis partial of this thread's dimensions, x from the tile
  auto d2_part = [&](int r, const float* w_row, int w_stride) -> float {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < TC16; ++j) {
      float v[16 / ESZ];
      const uint4 u = *reinterpret_cast<const uint4*>(xs + xs_off<ROWB>(r, d0 * ESZ / 16 + j));
      if constexpr (XT == GMM_F32) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
      } else {
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 f;
          if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&w4[i]));
          else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[i]));
          v[2 * i] = f.x; v[2 * i + 1] = f.y;
        }
      }
#pragma unroll
      for (int i = 0; i < 16 / ESZ; ++i) {
        const int dd = j * (16 / ESZ) + i;
        const float t = v[i] - cen(dd);
        const float w = iso ? w_row[0] : w_row[(size_t)dd * w_stride];
        acc[dd & 3] = fmaf(t * t, w, acc[dd & 3]);
      }
    }
    return (acc[0] + acc[2]) + (acc[1] + acc[3]);
  };

  const int64_t ntiles = (a.N + kBM - 1) / kBM;
  for (int64_t t = p; t < ntiles; t += P) {
    __syncthreads();  // the previous tile's tables are no longer read
    const int64_t r0 = t * kBM;
    const int rows = (int)min((int64_t)kBM, a.N - r0);
    for (int i = tid; i < 2 * CPB * 4; i += SH::THREADS) mask[i] = 0u;  // mask and smask
    // the tile's rows of X, 16-byte chunks, swizzled
    const unsigned char* gx = static_cast<const unsigned char*>(a.X) + (size_t)r0 * ROWB;
    for (int i = tid; i < rows * C16; i += SH::THREADS) {
      const int r = i / C16, q = i % C16;
      *reinterpret_cast<uint4*>(xs + xs_off<ROWB>(r, q)) =
          __ldg(reinterpret_cast<const uint4*>(gx + (size_t)r * ROWB) + q);
    }
    for (int i = tid; i < kBM; i += SH::THREADS) lse_s[i] = i < rows ? a.lse[r0 + i] : 0.f;
    const uint32_t tc = a.tile_cnt[t];
    const bool dense = tc > (uint32_t)a.rec_cap;
    __syncthreads();
    if (!dense) {
      // records of this component group -> table and row masks
      const uint2* rp = a.recs + (size_t)t * a.rec_cap;
      const uint32_t kc0 = (uint32_t)c * CPB;
      for (uint32_t i = tid; i < tc; i += SH::THREADS) {
        const uint2 rec = rp[i];
        const uint32_t kk = (rec.x >> 7) & kRecKMask;
        if (kk - kc0 < (uint32_t)CPB) {
          const int kr = (int)(kk - kc0), r = (int)(rec.x & 127u);
          lv[r * CPB + kr] = __uint_as_float(rec.y);
          atomicOr(&mask[kr * 4 + (r >> 5)], 1u << (r & 31));
          if (rec.x & kRecSingle) atomicOr(&smask[kr * 4 + (r >> 5)], 1u << (r & 31));
        }
      }
    } else {
      // every row the screen kept, every live component; the group's
      // precisions take the table's place: w[kl][d], rows of D + 1
      for (int i = tid; i < CPB * D; i += SH::THREADS) {
        const int kr = i / D, d = i % D;
        const int kk = c * CPB + kr;
        float w = 0.f;
        if (kk < a.K) w = iso ? (d == 0 ? __ldg(g_prec + kk) : 0.f) : __ldg(g_prec + (size_t)kk * D + d);
        lv[kr * (D + 1) + d] = w;
      }
      // every row with a finite LSE_n (a row without one is non-finite input,
      // which the screening kernel reports)
      for (int i = tid; i < CPB * 4; i += SH::THREADS) {
        const int w = i & 3;
        uint32_t v = 0u;
        for (int b = 0; b < 32; ++b) {
          const int r = w * 32 + b;
          if (r < rows && isfinite(lse_s[r])) v |= 1u << b;
        }
        mask[i] = v;
      }
    }
    __syncthreads();
    if (!live) continue;
    const float* w_row = dense ? lv + kl * (D + 1) + (iso ? 0 : d0) : nullptr;
    const float* gw = iso ? g_prec + k : g_prec + (size_t)k * D + d0;
#pragma unroll 1
    for (int wq = 0; wq < 4; ++wq) {
      uint32_t m = mask[kl * 4 + wq];
      const uint32_t sm1 = dense ? 0u : smask[kl * 4 + wq];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1u;
        const int r = wq * 32 + b;
        const bool single = (sm1 >> b) & 1u;
        float g;
        if (dense || single) {
          // the exact log joint, this thread's dimensions then the pair's sum
          float part = dense ? d2_part(r, w_row, 1) : d2_part(r, gw, 1);
#pragma unroll
          for (int o = 1; o < TPC; o <<= 1) part += __shfl_xor_sync(pair_mask, part, o);
          const float l = ck - 0.5f * part;
          if (single) {
            g = 1.f;
            if (h == 0) ll_acc += (double)l;
          } else {
            g = expf(l - lse_s[r]);
          }
        } else {
          g = expf(lv[r * CPB + kl] - lse_s[r]);
        }
        s0 += g;
#pragma unroll
        for (int j = 0; j < TC16; ++j) {
          float v[16 / ESZ];
          const uint4 u = *reinterpret_cast<const uint4*>(xs + xs_off<ROWB>(r, d0 * ESZ / 16 + j));
          if constexpr (XT == GMM_F32) {
            v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
            v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
          } else {
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float2 f;
              if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&w4[i]));
              else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[i]));
              v[2 * i] = f.x; v[2 * i + 1] = f.y;
            }
          }
#pragma unroll
          for (int i = 0; i < 16 / ESZ; ++i) {
            const int dd = j * (16 / ESZ) + i;
            const float y = v[i] - cen(dd);
            const float gy = g * y;
            s1[dd] += gy;
            s2[dd] = fmaf(gy, y, s2[dd]);
          }
        }
      }
    }
  }

  // this block's sums join slot p's fp64 partial of the component
  if (kin) {
    double* o = a.part + ((size_t)p * a.K + k) * F;
    const double b0 = (double)s0;
    const double S0o = a.accumulate ? o[0] : 0.0;
    const double S0 = S0o + b0;
#pragma unroll
    for (int i = 0; i < DPT; ++i) {
      const int d = d0 + i;
      // first moment about the fp32 mean: sum g (x - c') + b0 (c' - mu)
      const double shift = (double)cen(i) - (double)__ldg(g_mu + (size_t)k * D + d);
      const double b1c = (double)s1[i];
      const double b1 = b1c + b0 * shift;
      const double m2b = b0 > 0.0 ? (double)s2[i] - b1c * b1c / b0 : 0.0;
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
    __syncwarp(pair_mask);  // every thread of the component has read o[0] before it changes
    if (h == 0) o[0] = S0;
  }
  // the single-candidate points' log-likelihood of this block
  const double lw = warp_sum(ll_acc);
  if ((tid & 31) == 0) red[tid >> 5] = lw;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < SH::THREADS / 32; ++w) s += red[w];
    a.ll_part[(size_t)blockIdx.y * gridDim.x + blockIdx.x] = s;
  }
}

template <int D, int XT>
cudaError_t run_cs(const CsArgs& args, int nch, int P, cudaStream_t s) {
  constexpr size_t smem = CsSmem<D, XT>::BYTES;
  auto kern = chunk_stats_kernel<D, XT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(nch, P), CsShape<D>::THREADS, smem, s>>>(args);
  return cudaGetLastError();
}

}  // namespace

// Component groups and point partitions of the statistics blocks: about one
// block per SM in all, fixed by D and K alone so the order of the sums never
// depends on the device or on N.
int chunk_stats_blocks(int D, int K) {
  const int cpb = kThreads / (D / 32);
  return (K + cpb - 1) / cpb;
}
int chunk_stats_parts(int D, int K) {
  const int nch = chunk_stats_blocks(D, K);
  int p = (152 + nch - 1) / nch;
  return p < 1 ? 1 : p;
}

// Statistics of one slab of rows from the screening kernel's records into
// partial slots [0, P) of `part`; the slab's single-candidate log-likelihood
// into ll_part[0 .. nch * P).
cudaError_t chunk_stats(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                        const void* prepared, const float* lse, const uint2* recs,
                        const uint32_t* tile_cnt, int rec_cap, double* part, int accumulate,
                        double* ll_part, cudaStream_t s) {
  CsArgs a;
  a.X = X; a.N = N; a.K = K; a.prepared = prepared; a.L = PreparedLayout::make(D, K, cov);
  a.lse = lse; a.recs = recs; a.tile_cnt = tile_cnt; a.rec_cap = rec_cap;
  a.part = part; a.accumulate = accumulate; a.ll_part = ll_part;
  const int nch = chunk_stats_blocks(D, K);
  const int P = chunk_stats_parts(D, K);
  if (D == 128) {
    if (xdtype == GMM_F16) return run_cs<128, GMM_F16>(a, nch, P, s);
    if (xdtype == GMM_BF16) return run_cs<128, GMM_BF16>(a, nch, P, s);
    return run_cs<128, GMM_F32>(a, nch, P, s);
  }
  if (D == 64) {
    if (xdtype == GMM_F16) return run_cs<64, GMM_F16>(a, nch, P, s);
    if (xdtype == GMM_BF16) return run_cs<64, GMM_BF16>(a, nch, P, s);
    return run_cs<64, GMM_F32>(a, nch, P, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gmm
