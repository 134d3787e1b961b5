// tc_screen.cu - E-step on the tensor cores: screen every point-component
// pair with one fp16 tcgen05 contraction, then compute the few pairs that
// matter exactly on CUDA cores.
//
// For diagonal / isotropic covariance the log joint density is
//   l_nk = c_k + sum_d x_d (mu_kd w_kd) + x_d^2 (-w_kd / 2),   w = 1/var,
// a dense contraction [x, x^2] . [b1, b2] ("low-precision GMM operator"
// notes, sec. 1.2-1.3; Flash-GMM summary, Method: all-K distances per tile).
// Its terms are large and cancel (|x.b1| ~ 1e4 against l ~ 1e2 for tight
// clusters), so fp16 operands with fp32 accumulation give only a screen.
// Each screened value v (accumulator units; scale s_k, bias_k = c_k -
// sum mu^2 w / 2) comes with a rigorous bound on its error,
//   |s v + bias - l| <= kappa |[x, x^2]|_2 |[b1, b2]|_2 + 1e-6 (|s v| + |bias|) + 1e-3,
// from the fp16 rounding of b and x^2 (2^-11 each), of fp32 inputs (2^-11),
// fp32 accumulation and the fp32 evaluation of the sum (the relative term:
// its |s v| part is at most 1e-6 |[x, x^2]| |[b1, b2]| and joins kappa, its
// bias part and the 1e-3 are folded into the prepared bias - delta and
// bias + delta).  A component is kept when its upper bound reaches within
// T = 40 nats of the largest lower bound; every kept pair is then evaluated
// exactly in the centred fp32 form sum_d w_d (x_d - mu_d)^2, and LSE_n, the
// log-likelihood, top-m and the responsibilities come from those exact
// values (sec. 3.2, 4.2: fp32 log-sum-exp).  Components more than 40 nats
// below the best carry less than 4.3e-18 of a point's responsibility.  A
// point whose candidate list overflows (15 entries; per column half when the
// parameters are streamed) is handed to the CUDA-core path: one bit per row, turned into an ascending row list by
// fb_compact so that the order never depends on timing.
//
// Roles (one CTA per SM, persistent over 128-point tiles in a fixed order):
//   warps 0-7   epilogue.  Resident parameters (K <= 256): two groups of four
//               warps take alternate tiles, warp 4g + q reading TMEM lane
//               quarter q (32 points) over every column, so one group's
//               refine and records overlap the other group's sweeps; four
//               TMEM buffers, two per group.  Streamed parameters: warp w
//               reads lane quarter w % 4 and column half w / 4 of each chunk,
//               the two warps of a quarter combining their bounds and partial
//               log-sum-exp through shared memory (up to 30 candidates a row)
//   warps 8-11  producers: one point row per thread -> [x, x^2] fp16 tile in
//               shared memory (128-byte swizzled K-major), row norms; the
//               next tile's rows are loaded before the buffer is free
//   warp  12    lane 0 issues bulk copies of the parameter chunks and their
//               trailers and the tcgen05.mma instructions; the warp owns the
//               TMEM allocation
#include <float.h>
#include <math.h>

#include "gmm_internal.cuh"
#include "tc_ptx.cuh"

namespace gmm {
namespace {

constexpr int kBM = 128;          // points per tile (MMA M)
constexpr int kBN = kTcChunk;     // components per chunk (MMA N)
constexpr int kHalf = kBN / 2;    // columns of a chunk per warp (streamed parameters)
constexpr int kCS = 15;           // candidates per list, streamed parameters (per column half)
constexpr int kCSG = 13;          // candidates per point list, resident parameters
constexpr float kT = 40.f;        // nats
// Cauchy-Schwarz factor of the screening error: 3 x 2^-11 rounding plus the
// accumulation allowance (1.5e-3), plus 2e-6 that covers the relative fp32
// margin 1e-6 |s v| <= 1e-6 |a| |b| of evaluating s v + bias
constexpr float kKappa = 1.5e-3f + 2e-6f;
constexpr int kEpiWarps = 8;
constexpr int kProdWarp0 = 8;     // warps 8-11
constexpr int kMmaWarp = 12;
constexpr int kThreads = 13 * 32;
constexpr uint32_t kWait = 1u << 22;

enum { MODE_EM = 0, MODE_ASSIGN = 1 };


struct ScreenArgs {
  const void* X;
  int64_t N;
  int K;
  int m;                 // top-m (assign mode)
  const void* prepared;
  PreparedLayout L;
  float* lse;            // [N] or null (assign mode: null skips the output)
  int want_lse;          // EM: LSE_n of every point is wanted (else a point with a single
                         // candidate keeps gamma 1 without its exact log joint)
  double* ll_part;       // [gridDim.x] (EM) or null
  int32_t* ids;          // [N*m] (assign)
  float* gamma;          // [N*m] (assign)
  uint32_t* fb_mask;     // assign: [tiles * 4] bit r % 32 of word n / 32: row n
                         // handed to the CUDA-core path
  uint32_t* cmask;       // EM: [rows][chunks][4] candidate masks
                         // (word 2h + b: columns 64h + 32b .. + 31 of the chunk)
  uint32_t* dmask;       // EM: [tiles * 4] rows left to the dense-row kernels
  uint2* recs;           // EM: [tiles][rec_cap] records {key, exact log joint}
  uint32_t* tile_cnt;    // EM: [tiles] records of the tile (> rec_cap: they did not fit)
  int rec_cap;
  DeviceStatus* st;
};

// GRP: the grouped epilogue (resident, folded parameters, K <= 256): two
// groups of four warps take alternate tiles, each warp all columns of 32
// rows; four TMEM buffers, no trailer in shared memory.  Otherwise (parameters streamed with B):
// eight warps, the two of a lane quarter splitting each chunk's columns; two
// TMEM buffers and trailer slots.
template <int D, bool GRP>
struct Shape {
  static constexpr int KD = 2 * D;
  static constexpr int KSTEPS = KD / 16;
  static constexpr int CS = GRP ? kCSG : kCS;              // candidates per list
  static constexpr int A_BYTES = kBM * KD * 2;
  static constexpr int AX_BYTES = GRP ? kBM * kTcExtraK * 2 : 0;  // folded extra step of A
  static constexpr int B_MAIN = kBN * KD * 2;
  static constexpr int B_BYTES = B_MAIN + (GRP ? kTcExtraBytes : 0);  // one chunk's image
  static constexpr int T_BYTES = kTcTrail * 4;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_AX = OFF_A + A_BYTES;
  static constexpr int OFF_B = OFF_AX + AX_BYTES;           // 2 buffers
  static constexpr int NT = GRP ? 0 : 2;                    // trailer slots (folded: none)
  static constexpr int OFF_T = OFF_B + 2 * B_BYTES;
  static constexpr int OFF_RN = OFF_T + NT * T_BYTES;       // 2 x 128 row norms
  static constexpr int OFF_CUB = OFF_RN + 2 * kBM * 4;      // [2][CS][128] float
  static constexpr int OFF_CK = OFF_CUB + 2 * CS * kBM * 4;    // [2][CS][128] u16
  static constexpr int OFF_X = OFF_CK + 2 * CS * kBM * 2;      // exchange between warps
  // grouped: record counts [2 groups][2][128] u16; streamed: per half best
  // and m-th lower bound, max and sum of the exact values, counts
  static constexpr int X_BYTES = GRP ? 2 * 2 * kBM * 2 : 4 * 2 * kBM * 4 + 2 * kBM * 2;
  static constexpr int OFF_BAR = (OFF_X + X_BYTES + 7) / 8 * 8;  // 26 mbarrier slots
  static constexpr int OFF_MISC = OFF_BAR + 26 * 8;
  static constexpr int BYTES = OFF_MISC + 64;
  static constexpr int SMEM = BYTES + 1024;                 // base alignment slack
};

// 227 KB of shared memory per block, with the static part (ll_red)
static_assert(Shape<128, true>::SMEM + 8 * kEpiWarps <= 232448, "shared memory");
static_assert(Shape<128, false>::SMEM + 8 * kEpiWarps <= 232448, "shared memory");

// TMEM accumulator buffers of 128 columns (four allocated; the streamed
// mode uses two).
constexpr int kTmemCols = 512;
enum Bar {
  A_FULL = 0, A_EMPTY = 1, B_FULL = 2, B_EMPTY = 4, T_FULL = 6, T_EMPTY = 10, TR_FULL = 14,
  R_FULL = 18, R_FREE = 20, EXG = 22, EX_A = 22, EX_B = 23, EX_C = 24
};

// 8 consecutive stored coordinates as float, from raw 16-byte words.
template <int XT>
__device__ __forceinline__ void raw_to_float8(const uint4* w, float* v) {
  if constexpr (XT == GMM_F32) {
    v[0] = __uint_as_float(w[0].x); v[1] = __uint_as_float(w[0].y);
    v[2] = __uint_as_float(w[0].z); v[3] = __uint_as_float(w[0].w);
    v[4] = __uint_as_float(w[1].x); v[5] = __uint_as_float(w[1].y);
    v[6] = __uint_as_float(w[1].z); v[7] = __uint_as_float(w[1].w);
  } else {
    const uint32_t u[4] = {w[0].x, w[0].y, w[0].z, w[0].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f;
      if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
}

// Raw words of 8 coordinates starting at element `elem` (16-byte aligned).
template <int XT>
__device__ __forceinline__ void load_raw8(const void* X, size_t elem, uint4* w) {
  if constexpr (XT == GMM_F32) {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const float*>(X) + elem);
    w[0] = __ldg(p);
    w[1] = __ldg(p + 1);
  } else {
    w[0] = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(X) + elem));
  }
}

// Bounded wait whose outcome is the same for every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = tc::mbar_wait(bar, parity, kWait);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool warp_aborted(volatile int* flag) {
  return __any_sync(0xffffffffu, *flag != 0);
}

// Keeps lbm[0..m) the m largest values seen (descending); v > lbm[m-1].
__device__ __forceinline__ void insert_lower_bound(float* lbm, int m, float v) {
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    if (t < m && v > lbm[t]) { const float tmp = lbm[t]; lbm[t] = v; v = tmp; }
  }
}

// Four consecutive trailer entries of one field (16-byte aligned): one
// shared load serves four columns.
__device__ __forceinline__ void ld_trail4(const float* p, float* o) {
  const float4 q = *reinterpret_cast<const float4*>(p);
  o[0] = q.x; o[1] = q.y; o[2] = q.z; o[3] = q.w;
}

// Operands of one exact evaluation: row n of X against NC components.
template <int NC>
struct D2Args {
  const void* X;
  int64_t n;
  const float* mu[NC];
  const float* w[NC];   // 1/var (iso: one value)
  float wi[NC];         // iso: the value
  bool iso;
};

// Partial l: sum over dimensions l*D/32 .. (l+1)*D/32 - 1 of w (x - mu)^2,
// sequential fma from 0.
template <int D, int XT, int NC>
__device__ __forceinline__ void d2_leaf(const D2Args<NC>& q, int l, float* out) {
  constexpr int DPL = D / 32;
  float xv[DPL];
  const size_t e0 = (size_t)q.n * D + l * DPL;
  if constexpr (DPL == 4) {
    if constexpr (XT == GMM_F32) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(q.X) + e0));
      xv[0] = v.x; xv[1] = v.y; xv[2] = v.z; xv[3] = v.w;
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(q.X) + e0));
      const uint32_t u[2] = {v.x, v.y};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float2 f;
        if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&u[hh]));
        else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[hh]));
        xv[2 * hh] = f.x; xv[2 * hh + 1] = f.y;
      }
    }
  } else {
    if constexpr (XT == GMM_F32) {
      const float2 v = __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(q.X) + e0));
      xv[0] = v.x; xv[1] = v.y;
    } else {
      const uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(static_cast<const uint16_t*>(q.X) + e0));
      float2 f;
      if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&u));
      else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
      xv[0] = f.x; xv[1] = f.y;
    }
  }
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    float mv[DPL], wv[DPL];
    if constexpr (DPL == 4) {
      const float4 mq = __ldg(reinterpret_cast<const float4*>(q.mu[c] + l * 4));
      mv[0] = mq.x; mv[1] = mq.y; mv[2] = mq.z; mv[3] = mq.w;
      if (q.iso) {
        wv[0] = wv[1] = wv[2] = wv[3] = q.wi[c];
      } else {
        const float4 wq = __ldg(reinterpret_cast<const float4*>(q.w[c] + l * 4));
        wv[0] = wq.x; wv[1] = wq.y; wv[2] = wq.z; wv[3] = wq.w;
      }
    } else {
      const float2 mq = __ldg(reinterpret_cast<const float2*>(q.mu[c] + l * 2));
      mv[0] = mq.x; mv[1] = mq.y;
      if (q.iso) {
        wv[0] = wv[1] = q.wi[c];
      } else {
        const float2 wq = __ldg(reinterpret_cast<const float2*>(q.w[c] + l * 2));
        wv[0] = wq.x; wv[1] = wq.y;
      }
    }
    float part = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const float t = xv[i] - mv[i];
      part = fmaf(t * t, wv[i], part);
    }
    out[c] = part;
  }
}

// Quarter-warp evaluation of one pair: lane q (0..3) of a group of four
// computes the partials q, q+4, ..., q+28 of the 32-partial form (partial l
// = sum over dimensions l*D/32 .. (l+1)*D/32 - 1 of w (x - mu)^2,
// sequential fma from 0) and combines them in the pairwise tree order
// (+16, +8, +4 inside the lane; +2, +1 across the group with xor
// shuffles), so the result has the bits of every other evaluation.
template <int D, int XT>
__device__ __forceinline__ float group_d2(const void* X, int64_t n, const float* mu,
                                          const float* w, bool iso, int q) {
  D2Args<1> a;
  a.X = X; a.n = n; a.iso = iso;
  a.mu[0] = mu;
  a.w[0] = w;
  a.wi[0] = iso ? __ldg(w) : 0.f;
  float p[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) d2_leaf<D, XT, 1>(a, q + 4 * m, &p[m]);
  // +16: p[m] + p[m+4]; +8: + p[m+2]; +4: + p[m+1]
#pragma unroll
  for (int m = 0; m < 4; ++m) p[m] = p[m] + p[m + 4];
#pragma unroll
  for (int m = 0; m < 2; ++m) p[m] = p[m] + p[m + 2];
  float v = p[0] + p[1];
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// lbm[i] for a run-time i < 8 without indexing a local array.
__device__ __forceinline__ float pick8(const float* lbm, int i) {
  float v = lbm[0];
#pragma unroll
  for (int t = 1; t < 8; ++t) v = i == t ? lbm[t] : v;
  return v;
}

// Exact log joints of the warp's candidate lists (same arithmetic as the
// CUDA-core kernels): the warp's (row, candidate) pairs are numbered by an
// exclusive scan of the per-lane counts and taken eight at a time, four lanes
// per pair; cub[e][row] receives l of candidate e.
template <int D, int XT>
__device__ __forceinline__ void refine_lists(const void* X, int64_t tile, int q, int lane,
                                             int mycnt, float* cub, const uint16_t* ck,
                                             const float* g_mu, const float* g_prec,
                                             const float* g_c, bool iso) {
  __syncwarp();  // every lane's list entries are written
  int incl = mycnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - mycnt;
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  const int grp = lane >> 2, gq = lane & 3;
  for (int p0 = 0; p0 < total; p0 += 8) {
    const int pidx = p0 + grp;
    const bool live = pidx < total;
    // owner lane of pair pidx: the last lane whose excl <= pidx
    int owner = 0;
#pragma unroll
    for (int st = 16; st > 0; st >>= 1) {
      const int cand = owner + st;
      const int ev = __shfl_sync(0xffffffffu, excl, cand & 31);
      if (cand < 32 && ev <= pidx) owner = cand;
    }
    const int e = pidx - __shfl_sync(0xffffffffu, excl, owner);
    const int rr = q * 32 + owner;
    const int k = live ? (int)ck[e * kBM + rr] : 0;
    // (idle groups evaluate row 0 of the tile, which always exists)
    const float d2 = group_d2<D, XT>(X, tile * kBM + (live ? rr : 0), g_mu + (size_t)k * D,
                                     iso ? g_prec + k : g_prec + (size_t)k * D, iso, gq);
    if (live && gq == 0) cub[e * kBM + rr] = __ldg(g_c + k) - 0.5f * d2;
  }
  __syncwarp();
}

// Folds this row's cnt exact values into its running log-sum-exp (mx, sum).
__device__ __forceinline__ void fold_lse(const float* cub, int r, int cnt, float* mx, float* sum) {
  float lmx = -INFINITY;
  for (int e = 0; e < cnt; ++e) lmx = fmaxf(lmx, cub[e * kBM + r]);
  if (lmx == -INFINITY) return;
  const float nm = fmaxf(*mx, lmx);
  float s = *mx == -INFINITY ? 0.f : *sum * expf(*mx - nm);
  for (int e = 0; e < cnt; ++e) s += expf(cub[e * kBM + r] - nm);
  *mx = nm;
  *sum = s;
}

// Writes this row's cnt records {(k << 7) | row, l} (single: the flagged
// record of a point's only candidate, no value) to the warp's region of the
// tile's record buffer, after the records the warp wrote before (wpos, the
// same in every lane): the order is a function of the data alone.  Records
// past region_cap are not written; the warp's rows then take the CUDA-core
// path.
__device__ __forceinline__ void emit_records(int lane, int r, int cnt, const float* cub,
                                             const uint16_t* ck, uint32_t* wpos, uint2* region,
                                             int region_cap, bool single) {
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  const uint32_t p0 = *wpos + (uint32_t)(incl - cnt);
  for (int e = 0; e < cnt; ++e) {
    if (p0 + e < (uint32_t)region_cap) {
      const uint32_t key = (single ? kRecSingle : 0u) | ((uint32_t)ck[e * kBM + r] << 7) | (uint32_t)r;
      region[p0 + e] = make_uint2(key, single ? 0u : __float_as_uint(cub[e * kBM + r]));
    }
  }
  *wpos += (uint32_t)total;
}

template <int D, int XT, int MODE, bool GRP>
__global__ void __launch_bounds__(kThreads, 1) tc_screen_kernel(const ScreenArgs a) {
  using S = Shape<D, GRP>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = sm + S::OFF_A;
  unsigned char* sB = sm + S::OFF_B;
  float* sT = (float*)(sm + S::OFF_T);
  float* sRN = (float*)(sm + S::OFF_RN);
  float* sCUB = (float*)(sm + S::OFF_CUB);
  uint16_t* sCK = (uint16_t*)(sm + S::OFF_CK);
  float* xref = (float*)(sm + S::OFF_X);  // [2][128] per half: best lower bound
  float* xlbm = xref + 2 * kBM;           // [2][128] m-th largest lower bound (assign)
  float* xmx = xlbm + 2 * kBM;            // [2][128] max exact log joint
  float* xsum = xmx + 2 * kBM;            // [2][128] sum exp(l - max)
  uint16_t* xcnt = (uint16_t*)(xsum + 2 * kBM);  // [2][128] count, 0xffff: not exact
  uint16_t* xcg = (uint16_t*)(sm + S::OFF_X);    // grouped: [group][tile parity][128] counts
  uint64_t* bar = (uint64_t*)(sm + S::OFF_BAR);
  uint32_t* tmem_slot = (uint32_t*)(sm + S::OFF_MISC);
  volatile int* abort_flag = (volatile int*)(sm + S::OFF_MISC + 4);
  __shared__ double ll_red[kEpiWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t ntiles = (a.N + kBM - 1) / kBM;
  const int my_tiles = blockIdx.x < ntiles ? (int)((ntiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
  const int nch = a.L.tc_chunks;
  const bool resident = GRP;  // parameter chunks loaded once and kept (K <= 256)
  // TMEM buffer (and trailer slot) and its use count for contraction gi
  // (pass gi / nch, chunk gi % nch) of tile it: grouped, chunk j of the
  // group's tiles keeps buffer 2g + j, contracted once and swept by both
  // passes; streamed, each pass contracts again and the contractions
  // alternate over two buffers
  // streamed parameters: each tile contracted twice (bounds, then candidates)
  const int ncontr = GRP ? nch : 2 * nch;  // contractions per tile
  auto tbuf = [&](int it, int gi, int* buf, uint32_t* use) {
    if constexpr (GRP) {
      *buf = 2 * (it & 1) + gi % nch;   // one contraction per chunk, swept twice
      *use = (uint32_t)(it >> 1);
    } else {
      const int64_t gq = (int64_t)it * ncontr + gi;
      *buf = (int)(gq & 1);
      *use = (uint32_t)(gq >> 1);
    }
  };

  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar[A_FULL], 4);
    tc::mbar_init(&bar[A_EMPTY], 1);
    // arrivals per phase from the epilogue: a group (4 warps) or all 8
    const uint32_t epi = GRP ? 4u : (uint32_t)kEpiWarps;
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&bar[B_FULL + i], 1);
      tc::mbar_init(&bar[B_EMPTY + i], 1);
      tc::mbar_init(&bar[R_FULL + i], 4);
      tc::mbar_init(&bar[R_FREE + i], epi);
    }
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&bar[T_FULL + i], 1);
      tc::mbar_init(&bar[T_EMPTY + i], epi);
      tc::mbar_init(&bar[TR_FULL + i], 1);
    }
    if constexpr (GRP) {
      tc::mbar_init(&bar[EXG], 4);
      tc::mbar_init(&bar[EXG + 1], 4);
    } else {
      tc::mbar_init(&bar[EX_A], kEpiWarps);
      tc::mbar_init(&bar[EX_B], kEpiWarps);
      tc::mbar_init(&bar[EX_C], kEpiWarps);
    }
    *abort_flag = 0;
    tc::mbar_fence_init();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&](void) {
    *abort_flag = 1;
    raise_status(a.st, GMM_ERR_TIMEOUT);
  };

  const unsigned char* gB = at<unsigned char>(a.prepared, a.L.off_tcB);
  const float* gT = at<float>(a.prepared, a.L.off_tcT);
  const float* g_mu = at<float>(a.prepared, a.L.off_mu);
  const float* g_prec = at<float>(a.prepared, a.L.off_prec);
  const float* g_c = at<float>(a.prepared, a.L.off_c);
  const bool iso = a.L.cov == GMM_COV_ISO;

  if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issue + loads
    if (lane == 0 && my_tiles > 0) {
      const int64_t total = (int64_t)my_tiles * ncontr;
      auto load_b = [&](int64_t g) {
        const int buf = (int)(g & 1), c = (int)(g % nch);
        tc::mbar_arrive_expect_tx(&bar[B_FULL + buf], S::B_BYTES);
        tc::bulk_g2s(sB + buf * S::B_BYTES, gB + (size_t)c * a.L.tcB_chunk_bytes, S::B_BYTES,
                     &bar[B_FULL + buf]);
      };
      if (resident) {
        for (int c = 0; c < nch; ++c) {
          tc::mbar_arrive_expect_tx(&bar[B_FULL + c], S::B_BYTES);
          tc::bulk_g2s(sB + c * S::B_BYTES, gB + (size_t)c * a.L.tcB_chunk_bytes, S::B_BYTES,
                       &bar[B_FULL + c]);
        }
      } else {
        for (int64_t g = 0; g < 2 && g < total; ++g) load_b(g);
      }
      const uint32_t idesc = tc::idesc_f16_f32(kBM, kBN);
      bool ok = true;
      for (int it = 0; it < my_tiles && ok; ++it) {
        if (!tc::mbar_wait(&bar[A_FULL], it & 1, kWait)) { fail(); ok = false; break; }
        tc::tc_fence_after();
        for (int gi = 0; gi < ncontr; ++gi) {
          const int j = gi % nch;
          const int64_t g = (int64_t)it * ncontr + gi;
          const int sbuf = (int)(g & 1);               // streamed B buffer
          int buf;                                     // TMEM buffer and trailer slot
          uint32_t use;
          tbuf(it, gi, &buf, &use);
          const int bbuf = resident ? j : sbuf;
          if (!tc::mbar_wait(&bar[B_FULL + bbuf], resident ? 0u : (uint32_t)((g >> 1) & 1), kWait) ||
              !tc::mbar_wait(&bar[T_EMPTY + buf], (use & 1) ^ 1, kWait) || *abort_flag) {
            fail(); ok = false; break;
          }
          tc::tc_fence_after();
          if constexpr (!GRP) {
            // the trailer slot of a TMEM buffer is free once the buffer is
            tc::mbar_arrive_expect_tx(&bar[TR_FULL + buf], S::T_BYTES);
            tc::bulk_g2s(sT + buf * (S::T_BYTES / 4), gT + (size_t)j * kTcTrail, S::T_BYTES,
                         &bar[TR_FULL + buf]);
          }
          const uint32_t d_tmem = tmem_base + (uint32_t)(buf * kBN);
          const unsigned char* bb = sB + bbuf * S::B_BYTES;
#pragma unroll
          for (int ks = 0; ks < S::KSTEPS; ++ks) {
            const int atom = ks >> 2, within = (ks & 3) * 32;
            const uint64_t da = tc::sdesc_k128(tc::smem_addr(sA + atom * kBM * 128 + within));
            const uint64_t db = tc::sdesc_k128(tc::smem_addr(bb + atom * kBN * 128 + within));
            tc::mma_f16(d_tmem, da, db, idesc, ks > 0 ? 1u : 0u);
          }
          if constexpr (GRP) {
            // the folded step: bias and margin (unswizzled K = 16 operands)
            tc::mma_f16(d_tmem, tc::sdesc_k16(tc::smem_addr(sm + S::OFF_AX)),
                        tc::sdesc_k16(tc::smem_addr(bb + S::B_MAIN)), idesc, 1u);
          }
          if (!resident) tc::mma_commit(&bar[B_EMPTY + sbuf]);
          tc::mma_commit(&bar[T_FULL + buf]);
          if (gi == ncontr - 1) tc::mma_commit(&bar[A_EMPTY]);
          if (!resident && g + 1 < total && g + 1 >= 2) {
            // refill the other buffer once the MMAs of chunk g-1 are done
            const int pb = (int)((g + 1) & 1);
            const uint32_t puse = (uint32_t)((g + 1) >> 1);
            if (!tc::mbar_wait(&bar[B_EMPTY + pb], (puse - 1) & 1, kWait)) {
              fail(); ok = false; break;
            }
            load_b(g + 1);
          }
        }
      }
      // drain: the last parameter loads must land before the CTA exits
      if (!resident && total >= 1) {
        for (int64_t g = total - 2; g < total; ++g) {
          if (g < 0) continue;
          tc::mbar_wait(&bar[B_EMPTY + (int)(g & 1)], (uint32_t)((g >> 1) & 1), kWait);
        }
      }
    }
  } else if (warp >= kProdWarp0) {
    // ------------------------------------------------------- producers
    constexpr int G = D / 8;                       // 8-coordinate groups per row
    constexpr int WPG = XT == GMM_F32 ? 2 : 1;     // 16-byte words per group
    constexpr int PF = XT == GMM_F32 ? (G > 8 ? 8 : G) : G;  // groups loaded ahead
    const int p = tid - kProdWarp0 * 32;
    for (int it = 0; it < my_tiles; ++it) {
      if (warp_aborted(abort_flag)) break;
      const int64_t tile = blockIdx.x + (int64_t)it * gridDim.x;
      const int64_t n = tile * kBM + p;
      const bool in = n < a.N;
      // this tile's row, requested before the buffers are free
      uint4 pre[PF * WPG];
#pragma unroll
      for (int g = 0; g < PF; ++g) {
        if (in) load_raw8<XT>(a.X, (size_t)n * D + g * 8, pre + g * WPG);
        else
#pragma unroll
          for (int i = 0; i < WPG; ++i) pre[g * WPG + i] = make_uint4(0u, 0u, 0u, 0u);
      }
      float rn2 = 0.f;
      if constexpr (XT == GMM_F16) {
        // fp16 input: the row norm needs only the loaded row, so it is taken
        // before the wait for the operand buffer (while the previous tile's
        // contraction runs)
#pragma unroll
        for (int c8 = 0; c8 < G; ++c8) {
          const uint32_t w4[4] = {pre[c8].x, pre[c8].y, pre[c8].z, pre[c8].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 xx = *reinterpret_cast<const __half2*>(&w4[i]);
            const __half2 qq = __hmul2(xx, xx);
            const float2 xf = __half22float2(xx), qf = __half22float2(qq);
            rn2 += xf.x * xf.x + xf.y * xf.y + qf.x * qf.x + qf.y * qf.y;
          }
        }
      }
      if (it > 0 && !warp_wait(&bar[A_EMPTY], (it - 1) & 1)) { fail(); break; }
      if (it >= 2 && !warp_wait(&bar[R_FREE + (it & 1)], ((it >> 1) - 1) & 1)) {
        fail(); break;
      }
#pragma unroll
      for (int c8 = 0; c8 < G; ++c8) {
        if constexpr (XT == GMM_F16) {
          // fp16 input: x is the operand as stored, and x^2 = RN(x x) is one
          // packed multiply (fp16 multiplication is correctly rounded, the
          // same value as rounding the exact fp32 square)
          const uint32_t w4[4] = {pre[c8].x, pre[c8].y, pre[c8].z, pre[c8].w};
          uint32_t hq[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 qq = __hmul2(*reinterpret_cast<const __half2*>(&w4[i]),
                                       *reinterpret_cast<const __half2*>(&w4[i]));
            hq[i] = *reinterpret_cast<const uint32_t*>(&qq);
          }
          *reinterpret_cast<uint4*>(sA + tc::sw128_offset(p, c8 * 8, kBM)) = pre[c8];
          *reinterpret_cast<uint4*>(sA + tc::sw128_offset(p, D + c8 * 8, kBM)) =
              make_uint4(hq[0], hq[1], hq[2], hq[3]);
          continue;
        }
        float v[8];
        if (c8 < PF) {
          raw_to_float8<XT>(pre + c8 * WPG, v);
        } else {
          uint4 w[WPG];
          if (in) load_raw8<XT>(a.X, (size_t)n * D + c8 * 8, w);
          else
#pragma unroll
            for (int i = 0; i < WPG; ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
          raw_to_float8<XT>(w, v);
        }
        uint32_t hx[4], hq[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 xx = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
          const __half2 qq = __floats2half2_rn(v[2 * i] * v[2 * i], v[2 * i + 1] * v[2 * i + 1]);
          const float2 xf = __half22float2(xx), qf = __half22float2(qq);
          rn2 += xf.x * xf.x + xf.y * xf.y + qf.x * qf.x + qf.y * qf.y;
          hx[i] = *reinterpret_cast<const uint32_t*>(&xx);
          hq[i] = *reinterpret_cast<const uint32_t*>(&qq);
        }
        *reinterpret_cast<uint4*>(sA + tc::sw128_offset(p, c8 * 8, kBM)) =
            make_uint4(hx[0], hx[1], hx[2], hx[3]);
        *reinterpret_cast<uint4*>(sA + tc::sw128_offset(p, D + c8 * 8, kBM)) =
            make_uint4(hq[0], hq[1], hq[2], hq[3]);
      }
      // the norm (its fp32 sum errs by at most (D + 1) 2^-24 relative) with a
      // floor: fp16 subnormal rounding of x^2 (and of bf16 x below fp16's
      // normal range) errs by at most 2^-25 per coordinate, sqrt(2D) 2^-25 |b|
      // in all, below kappa x 1e-3 |b| for D <= 128
      const float rn = sqrtf(rn2) * 1.0001f + 1e-3f;
      sRN[(it & 1) * kBM + p] = rn;
      if constexpr (GRP) {
        // the folded step's row: [2^10, 1, 2^-10, ru(rn / 16), 1, 0 ...]
        const uint32_t h3 = (uint32_t)__half_as_ushort(__float2half_ru(rn * 0.0625f));
        *reinterpret_cast<uint4*>(sm + S::OFF_AX + tc::k16_offset(p, 0)) =
            make_uint4(0x3C006400u, 0x1400u | (h3 << 16), 0x3C00u, 0u);
        *reinterpret_cast<uint4*>(sm + S::OFF_AX + tc::k16_offset(p, 8)) = make_uint4(0u, 0u, 0u, 0u);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&bar[A_FULL]);
        tc::mbar_arrive(&bar[R_FULL + (it & 1)]);
      }
    }
  } else {
    if constexpr (GRP) {
    // ------------------------------------- epilogue (resident parameters)
    // group g (warps 4g .. 4g+3) takes tiles g, g+2, ...; warp q of the group
    // reads TMEM lane quarter q (32 points) over every column
    const int g = warp >> 2, q = warp & 3;
    const int r = q * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float* __restrict__ cub = sCUB + g * kCSG * kBM;     // this group's candidate lists
    uint16_t* __restrict__ ck = sCK + g * kCSG * kBM;
    double ll_acc = 0.0;
    for (int it = g; it < my_tiles; it += 2) {
      if (warp_aborted(abort_flag)) break;
      const int s = it >> 1;  // the group's s-th tile
      const int64_t tile = blockIdx.x + (int64_t)it * gridDim.x;
      const int64_t n = tile * kBM + r;
      const bool valid = n < a.N;
      if (!warp_wait(&bar[R_FULL + g], s & 1)) { fail(); break; }
      const float rn = sRN[g * kBM + r];
      // the slot holds only the row norms: hand it back at once, so that the
      // producers' next write of it never waits for this tile's sweeps
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[R_FREE + g]);
      float ref = -INFINITY;  // lower bound of the best log joint
      float dropped = -INFINITY;
      float lbm[8];           // assign: the m largest lower bounds seen
#pragma unroll
      for (int i = 0; i < 8; ++i) lbm[i] = -INFINITY;
      float lmth = -INFINITY;  // assign: the m-th largest of them
      int cnt = 0;
      bool ok = true;
      float thr = -INFINITY;  // the point's window, fixed after pass 0
      // EM: the point's log-sum-exp over its refined candidates, this warp's
      // region of the tile's records (regions 2q and 2q + 1 of the eight),
      // the point's candidate masks (every chunk, for the dense-row kernels)
      // and whether its list filled (the point then goes to those kernels)
      float mx = -INFINITY, ssum = 0.f;
      bool deferred = false;
      uint32_t wpos = 0;
      const int rcap = a.rec_cap / 4;
      uint2* region = a.recs + (size_t)tile * a.rec_cap + (size_t)q * rcap;
      uint32_t* rmask = MODE == MODE_EM ? a.cmask + (size_t)(tile * kBM + r) * nch * 4 : nullptr;
      // pass 0: lower bounds only; pass 1 (a second sweep of the same
      // accumulators): candidates against the point's final window
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          thr = ref - kT;
          // assign: m components have a lower bound >= the m-th largest, so
          // nothing below it can be in the top m
          if constexpr (MODE == MODE_ASSIGN) thr = fminf(thr, lmth);
        }
        for (int j = 0; j < nch; ++j) {
          int buf;
          uint32_t use;
          tbuf(it, j, &buf, &use);
          if (pass == 0) {
            if (!warp_wait(&bar[T_FULL + buf], use & 1)) { fail(); ok = false; break; }
            tc::tc_fence_after();
          }
          // the chunk's scale and margins (see tc_fold)
          const float* __restrict__ gTj = gT + (size_t)j * kTcTrail;
          const float Sj = __ldg(gTj + kFoldS);
          const uint32_t tcol = tmem_base + lane_base + (uint32_t)(buf * kBN);
          if (pass == 0) {
            // the accumulators hold hi_k / S.  The largest, its column packed
            // into the low seven bits (a change below 2^-16 relative), names
            // a component whose lower bound hi - 2.01 (rn u + d) bounds the
            // best log joint from below
            float pk0 = -INFINITY, pk1 = -INFINITY;  // two chains
            float wmax = 0.f;
            if constexpr (MODE == MODE_ASSIGN)
              wmax = 2.01f * fmaf(rn, __ldg(gTj + kFoldUMax), __ldg(gTj + kFoldDMax));
#pragma unroll
            for (int c0 = 0; c0 < kBN; c0 += 32) {
              uint32_t u[32];
              tc::tmem_ld32_issue(tcol + (uint32_t)c0, u);
              tc::tmem_wait32(u);
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const float pv = __uint_as_float((u[i] & ~0x7Fu) | (uint32_t)(c0 + i));
                if (i & 1) pk1 = fmaxf(pk1, pv);
                else pk0 = fmaxf(pk0, pv);
                if constexpr (MODE == MODE_ASSIGN) {
                  // a lower bound with the chunk's largest margin
                  const float h = Sj * __uint_as_float(u[i]);
                  const float lo = h - wmax - 1e-6f * fabsf(h);
                  if (lo > lmth) {
                    insert_lower_bound(lbm, a.m, lo);
                    lmth = pick8(lbm, a.m - 1);
                  }
                }
              }
            }
            const uint32_t pb = __float_as_uint(fmaxf(pk0, pk1));
            const int kh = (int)(pb & 0x7Fu);
            const float t0 = __uint_as_float(pb & ~0x7Fu);
            const float h = Sj * (t0 - fabsf(t0) * 0x1p-15f);
            const float lo = h - 2.01f * fmaf(rn, __ldg(gTj + kh), __ldg(gTj + kTcChunk + kh)) -
                             1e-6f * fabsf(h);
            ref = fmaxf(ref, lo);
          } else {
            // every component whose upper bound reaches the window,
            // hi_k / S >= thr / S (S a power of two)
            const float tthr = thr * __ldg(gTj + kFoldInvS);
#pragma unroll 1
            for (int c0 = 0; c0 < kBN; c0 += 32) {
              uint32_t u[32];
              tc::tmem_ld32_issue(tcol + (uint32_t)c0, u);
              tc::tmem_wait32(u);
              // a bit per column in the window (no branch in the sweep), then
              // the (rare) appends in column order
              uint32_t pm = 0u;
#pragma unroll
              for (int i = 0; i < 32; ++i) pm |= __uint_as_float(u[i]) >= tthr ? (1u << i) : 0u;
              if (!valid) pm = 0u;
              if constexpr (MODE == MODE_EM) {
                if (!isfinite(rn)) pm = 0u;  // handed over (non-finite input)
                if (valid) rmask[j * 4 + (c0 >> 5)] = pm;
                // append while the list has room; a point with more
                // candidates goes to the dense-row kernels with its masks
                while (pm && cnt < kCSG) {
                  const int kk = c0 + __ffs(pm) - 1;
                  pm &= pm - 1u;
                  ck[cnt * kBM + r] = (uint16_t)(j * kBN + kk);
                  ++cnt;
                }
                if (pm) deferred = true;
              } else {
                while (pm) {
                  const int kk = c0 + __ffs(pm) - 1;
                  pm &= pm - 1u;
                  if (cnt < kCSG) {
                    ck[cnt * kBM + r] = (uint16_t)(j * kBN + kk);
                    ++cnt;
                  } else {
                    dropped = INFINITY;  // list full: the row goes to the CUDA-core path
                  }
                }
              }
            }
          }
          if (pass == 1) {  // the buffer is free after the second sweep
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bar[T_EMPTY + buf]);
          }
        }
      }
      __syncwarp();
      if (!ok) break;
      if constexpr (MODE == MODE_EM) {
        // this warp's record count: past its region's capacity the warp's
        // rows take the CUDA-core path
        int mine = deferred ? 0 : cnt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        const bool overflow = mine > rcap;
        const bool exact = valid && isfinite(rn) && cnt > 0 && !deferred && !overflow;
        // a point with a single candidate has gamma = 1 (every other
        // component lies more than 40 nats below it); unless LSE_n is wanted
        // its exact log joint is not needed here: the statistics give its
        // log-likelihood term
        const bool single = exact && cnt == 1 && !a.want_lse;
        refine_lists<D, XT>(a.X, tile, q, lane, (exact && !single) ? cnt : 0, cub, ck, g_mu,
                            g_prec, g_c, iso);
        if (exact && !single) fold_lse(cub, r, cnt, &mx, &ssum);
        emit_records(lane, r, exact ? cnt : 0, cub, ck, &wpos, region, rcap, single);
        if (exact && !single) {
          const float lse = mx + logf(ssum);
          if (!isfinite(lse)) raise_status(a.st, GMM_ERR_NONFINITE);
          a.lse[n] = lse;
          ll_acc += (double)lse;
        }
        // rows of an overflowing warp, and rows without a candidate
        // (non-finite input), go to the CUDA-core path; rows with a full
        // list to the dense-row kernels
        const bool dense = valid && isfinite(rn) && deferred && !overflow;
        const unsigned fbm = __ballot_sync(0xffffffffu, valid && !exact && !dense);
        const unsigned dbm = __ballot_sync(0xffffffffu, dense);
        if (lane == 0) {
          a.fb_mask[tile * 4 + q] = fbm;
          a.dmask[tile * 4 + q] = dbm;
          a.tile_cnt[tile * 8 + 2 * q] = overflow ? 0u : (uint32_t)mine;
          a.tile_cnt[tile * 8 + 2 * q + 1] = 0u;
        }
      } else {
      const bool exact = valid && isfinite(rn) && !(dropped >= thr) && cnt > 0;
      // a point with a single candidate has gamma = 1 (every other component
      // lies more than 40 nats below it); unless LSE_n is wanted its exact
      // log joint is not needed here (the statistics give its
      // log-likelihood term)
      const bool single = exact && cnt == 1 && a.lse == nullptr;
      // exact log joints of the other points' candidates
      refine_lists<D, XT>(a.X, tile, q, lane, (exact && !single) ? cnt : 0, cub, ck, g_mu, g_prec,
                          g_c, iso);
      float lse = 0.f;
      if (exact && !single) {
        float mx = -INFINITY, sum = 0.f;
        for (int e = 0; e < cnt; ++e) mx = fmaxf(mx, cub[e * kBM + r]);
        for (int e = 0; e < cnt; ++e) sum += expf(cub[e * kBM + r] - mx);
        lse = mx + logf(sum);
      }
        if (single) {
          a.ids[n * a.m] = ck[r];
          a.gamma[n * a.m] = 1.f;
          for (int t = 1; t < a.m; ++t) {
            a.ids[n * a.m + t] = -1;
            a.gamma[n * a.m + t] = 0.f;
          }
        } else if (exact) {
          if (!isfinite(lse)) raise_status(a.st, GMM_ERR_NONFINITE);
          if (a.lse) a.lse[n] = lse;
          // top-m by exact value, ties to the lower component
          uint32_t taken = 0;
          for (int t = 0; t < a.m; ++t) {
            int best = -1, bk = 0x7fffffff;
            float bv = -INFINITY;
            for (int e = 0; e < cnt; ++e) {
              if (taken & (1u << e)) continue;
              const float v = cub[e * kBM + r];
              const int k = ck[e * kBM + r];
              if (best < 0 || v > bv || (v == bv && k < bk)) { best = e; bv = v; bk = k; }
            }
            if (best < 0) {
              a.ids[n * a.m + t] = -1;
              a.gamma[n * a.m + t] = 0.f;
              continue;
            }
            taken |= 1u << best;
            a.ids[n * a.m + t] = bk;
            a.gamma[n * a.m + t] = bv == -INFINITY ? 0.f : expf(bv - lse);
          }
        }
        const unsigned fbm = __ballot_sync(0xffffffffu, valid && !exact);
        if (lane == 0) a.fb_mask[tile * 4 + q] = fbm;
      }
      __syncwarp();
    }
    if constexpr (MODE == MODE_EM) {
      const double sacc = warp_sum(ll_acc);
      if (lane == 0) ll_red[warp] = sacc;
    }
    } else if constexpr (MODE == MODE_EM) {
    // --------------------------- epilogue (streamed parameters, EM mode)
    // warp w reads lane quarter q = w % 4 and column half h = w / 4 of every
    // chunk.  Each tile is contracted twice: pass 0 finds the best lower bound
    // (both halves combined at barrier A), pass 1 collects every column whose
    // upper bound reaches it minus 40 nats, and writes every row's candidate
    // masks.  A row with more candidates than a half's list holds is left to
    // the dense-row kernels, which evaluate its candidates from the masks with
    // the parameters staged in shared memory.  Barrier B: both halves' counts
    // (singles, overflow, left rows); barrier C: both halves' partial
    // log-sum-exp.
    const int q = warp & 3, h = warp >> 2;
    const int r = q * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float* __restrict__ cub = sCUB + h * kCS * kBM;     // this half's candidate list
    uint16_t* __restrict__ ck = sCK + h * kCS * kBM;
    uint32_t* xtot = reinterpret_cast<uint32_t*>(xlbm);  // [2][128] records per row and half
    const int rcap = a.rec_cap / 8;                       // this warp's region of the tile's records
    double ll_acc = 0.0;
    for (int it = 0; it < my_tiles; ++it) {
      if (warp_aborted(abort_flag)) break;
      const int64_t tile = blockIdx.x + (int64_t)it * gridDim.x;
      const int64_t n = tile * kBM + r;
      const bool valid = n < a.N;
      if (!warp_wait(&bar[R_FULL + (it & 1)], (it >> 1) & 1)) { fail(); break; }
      const float rn = sRN[(it & 1) * kBM + r];
      const float rnk = kKappa * rn;
      // the slot holds only the row norms: hand it back at once
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[R_FREE + (it & 1)]);
      const bool rowok = valid && isfinite(rn);
      float ref = -INFINITY, thr = -INFINITY;
      float mx = -INFINITY, ssum = 0.f;
      int cnt = 0;
      bool deferred = false, ok = true;
      uint32_t wpos = 0;
      uint2* region = a.recs + (size_t)tile * a.rec_cap + (size_t)(2 * q + h) * rcap;
      uint32_t* rmask = a.cmask + (size_t)(tile * kBM + r) * nch * 4 + 2 * h;
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          xref[h * kBM + r] = ref;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bar[EX_A]);
          if (!warp_wait(&bar[EX_A], it & 1)) { fail(); ok = false; break; }
          // the window (never reached by an excluded component: its bound is -inf)
          thr = fmaxf(fmaxf(xref[r], xref[kBM + r]) - kT, -FLT_MAX);
        }
        for (int j = 0; j < nch; ++j) {
          const int64_t gq = ((int64_t)it * 2 + pass) * nch + j;
          const int buf = (int)(gq & 1);             // TMEM buffer and trailer slot
          const uint32_t use = (uint32_t)(gq >> 1);
          if (!warp_wait(&bar[T_FULL + buf], use & 1) || !warp_wait(&bar[TR_FULL + buf], use & 1)) {
            fail(); ok = false; break;
          }
          tc::tc_fence_after();
          const float* __restrict__ tsc = sT + buf * (S::T_BYTES / 4) + h * kHalf;
          const float* __restrict__ tcn = tsc + kBN;
          const float* __restrict__ tbl = tsc + 2 * kBN;   // bias - delta
          const float* __restrict__ tbh = tsc + 3 * kBN;   // bias + delta
          const float Sj = tsc[0];  // the chunk's common scale (every slot holds it)
          const uint32_t tcol = tmem_base + lane_base + (uint32_t)(buf * kBN + h * kHalf);
          uint32_t pms[kHalf / 32];
#pragma unroll
          for (int b = 0; b < kHalf / 32; ++b) {
            const int c0 = b * 32;
            uint32_t u[32];
            tc::tmem_ld32_issue(tcol + (uint32_t)c0, u);
            tc::tmem_wait32(u);
            uint32_t pm = 0u;
            if (pass == 0) {
              // lower bounds lo = s v + (bias - delta) - rnk |b|
              float best0 = -INFINITY, best1 = -INFINITY;
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                float nb[4], bb[4];
                ld_trail4(tcn + c0 + i, nb);
                ld_trail4(tbl + c0 + i, bb);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const float lo = fmaf(__uint_as_float(u[i + t]), Sj, fmaf(-rnk, nb[t], bb[t]));
                  if (t & 1) best1 = fmaxf(best1, lo);
                  else best0 = fmaxf(best0, lo);
                }
              }
              ref = fmaxf(ref, fmaxf(best0, best1));
            } else {
              // every column whose upper bound hi = s v + (bias + delta) + rnk |b|
              // reaches the window
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                float nb[4], bb[4];
                ld_trail4(tcn + c0 + i, nb);
                ld_trail4(tbh + c0 + i, bb);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const float hi = fmaf(__uint_as_float(u[i + t]), Sj, fmaf(rnk, nb[t], bb[t]));
                  pm |= hi >= thr ? (1u << (i + t)) : 0u;
                }
              }
            }
            pms[b] = rowok ? pm : 0u;
          }
          // the accumulators and the trailer slot are read: hand them back
          // before the (possibly long) appends and flushes
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bar[T_EMPTY + buf]);
          if (pass == 1) {
            // the row's masks (read back only for rows left to the dense-row kernels)
            if (valid) *reinterpret_cast<uint2*>(rmask + j * 4) = make_uint2(pms[0], pms[1]);
#pragma unroll
            for (int b = 0; b < kHalf / 32; ++b) {
              uint32_t pm = deferred ? 0u : pms[b];
              const int kb = j * kBN + h * kHalf + b * 32;
              while (pm) {
                const int kk = __ffs(pm) - 1;
                pm &= pm - 1u;
                if (cnt < kCS) {
                  ck[cnt * kBM + r] = (uint16_t)(kb + kk);
                  ++cnt;
                } else {
                  deferred = true;  // the list is full: the row goes to the dense-row kernels
                  pm = 0u;
                }
              }
            }
          }
        }
      }
      if (!ok) break;
      // barrier B: candidates per row and half (bit 31: the half's list was
      // full, the row is left to the dense-row kernels)
      xtot[h * kBM + r] = (uint32_t)cnt | (deferred ? 0x80000000u : 0u);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[EX_B]);
      if (!warp_wait(&bar[EX_B], it & 1)) { fail(); break; }
      const uint32_t t0 = xtot[r], t1 = xtot[kBM + r];
      const bool left = ((t0 | t1) >> 31) != 0u;
      // this quarter's two regions: past either one's capacity, the
      // quarter's rows take the CUDA-core path
      uint32_t w0 = left ? 0u : (t0 & 0x7fffffffu), w1 = left ? 0u : (t1 & 0x7fffffffu);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        w0 += __shfl_xor_sync(0xffffffffu, w0, o);
        w1 += __shfl_xor_sync(0xffffffffu, w1, o);
      }
      const bool overflow = w0 > (uint32_t)rcap || w1 > (uint32_t)rcap;
      const uint32_t both = (t0 & 0x7fffffffu) + (t1 & 0x7fffffffu);
      const bool exact = rowok && !left && both > 0 && !overflow;
      const bool single = exact && both == 1 && !a.want_lse;
      refine_lists<D, XT>(a.X, tile, q, lane, (exact && !single) ? cnt : 0, cub, ck, g_mu, g_prec,
                          g_c, iso);
      if (exact && !single) fold_lse(cub, r, cnt, &mx, &ssum);
      emit_records(lane, r, exact ? cnt : 0, cub, ck, &wpos, region, rcap, single);
      // barrier C: both halves' partial log-sum-exp
      xmx[h * kBM + r] = mx;
      xsum[h * kBM + r] = ssum;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[EX_C]);
      if (!warp_wait(&bar[EX_C], it & 1)) { fail(); break; }
      if (h == 0) {
        if (exact && !single) {
          const float m0 = xmx[r], m1 = xmx[kBM + r];
          const float M = fmaxf(m0, m1);
          float sum = 0.f;
          if (m0 > -INFINITY) sum += xsum[r] * expf(m0 - M);
          if (m1 > -INFINITY) sum += xsum[kBM + r] * expf(m1 - M);
          const float lse = M + logf(sum);
          if (!isfinite(lse)) raise_status(a.st, GMM_ERR_NONFINITE);
          a.lse[n] = lse;
          ll_acc += (double)lse;
        }
        // rows of an overflowing quarter, and rows without a candidate
        // (non-finite input), go to the CUDA-core path; rows with a full list
        // to the dense-row kernels
        const bool dense = rowok && left && !overflow;
        const unsigned fbm = __ballot_sync(0xffffffffu, valid && !exact && !dense);
        const unsigned dbm = __ballot_sync(0xffffffffu, dense);
        if (lane == 0) {
          a.fb_mask[tile * 4 + q] = fbm;
          a.dmask[tile * 4 + q] = dbm;
        }
      }
      if (lane == 0) a.tile_cnt[tile * 8 + 2 * q + h] = overflow ? 0u : (h == 0 ? w0 : w1);
      __syncwarp();
    }
    {
      const double sacc = warp_sum(ll_acc);
      if (lane == 0) ll_red[warp] = sacc;
    }
    } else {
    // ------------------------- epilogue (streamed parameters, assignment)
    const int q = warp & 3, h = warp >> 2;
    const int r = q * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float* __restrict__ cub = sCUB + h * kCS * kBM;     // this half's candidate list
    uint16_t* __restrict__ ck = sCK + h * kCS * kBM;
    double ll_acc = 0.0;
    for (int it = 0; it < my_tiles; ++it) {
      if (warp_aborted(abort_flag)) break;
      const int64_t tile = blockIdx.x + (int64_t)it * gridDim.x;
      const int64_t n = tile * kBM + r;
      const bool valid = n < a.N;
      if (!warp_wait(&bar[R_FULL + (it & 1)], (it >> 1) & 1)) { fail(); break; }
      const float rn = sRN[(it & 1) * kBM + r];
      const float rnk = kKappa * rn;
      float ref = -INFINITY;  // lower bound of the best log joint (this half)
      float dropped = -INFINITY;
      float lbm[8];           // assign: the m largest lower bounds seen
#pragma unroll
      for (int i = 0; i < 8; ++i) lbm[i] = -INFINITY;
      float lmth = -INFINITY;  // assign: the m-th largest of them
      int cnt = 0;
      bool ok = true;
      float thr = -INFINITY;  // the point's window, fixed after pass 0
      // pass 0: lower bounds only; pass 1 (a second contraction of the same
      // tile): candidates against the point's final window
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) {
          // exchange A: the best lower bound (assign: the m-th largest) of
          // both column halves
          xref[h * kBM + r] = ref;
          if constexpr (MODE == MODE_ASSIGN) xlbm[h * kBM + r] = lmth;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bar[EX_A]);
          if (!warp_wait(&bar[EX_A], it & 1)) { fail(); ok = false; break; }
          thr = fmaxf(xref[r], xref[kBM + r]) - kT;
          // assign: at least m components have a lower bound >= the larger
          // of the two halves' m-th largest, so nothing below it can be in
          // the top m
          if constexpr (MODE == MODE_ASSIGN) thr = fminf(thr, fmaxf(xlbm[r], xlbm[kBM + r]));
        }
        for (int j = 0; j < nch; ++j) {
          const int64_t g = ((int64_t)it * 2 + pass) * nch + j;
          const int buf = (int)(g & 1);             // TMEM buffer and trailer slot
          const uint32_t use = (uint32_t)(g >> 1);
          const int tb = buf;
          if (!warp_wait(&bar[T_FULL + buf], use & 1) ||
              !warp_wait(&bar[TR_FULL + tb], use & 1)) {
            fail(); ok = false; break;
          }
          tc::tc_fence_after();
          // (the trailer and the candidate lists never overlap)
          const float* __restrict__ tsc = sT + tb * (S::T_BYTES / 4) + h * kHalf;
          const float* __restrict__ tcn = tsc + kBN;
          const float* __restrict__ tbl = tsc + 2 * kBN;   // bias - delta
          const float* __restrict__ tbh = tsc + 3 * kBN;   // bias + delta
          const float Sj = tsc[0];  // the chunk's common scale (every slot holds it)
          const uint32_t tcol = tmem_base + lane_base + (uint32_t)(buf * kBN + h * kHalf);
          if (pass == 0) {
            // the best lower bound of the half-chunk,
            //   lo = s v + (bias - delta) - rnk |b|
            float best0 = -INFINITY, best1 = -INFINITY;  // two chains
#pragma unroll 1
            for (int c0 = 0; c0 < kHalf; c0 += 32) {
              uint32_t u[32];
              tc::tmem_ld32_issue(tcol + (uint32_t)c0, u);
              tc::tmem_wait32(u);
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                float nb[4], bb[4];
                ld_trail4(tcn + c0 + i, nb);
                ld_trail4(tbl + c0 + i, bb);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const float v = __uint_as_float(u[i + t]);
                  const float lo = fmaf(v, Sj, fmaf(-rnk, nb[t], bb[t]));
                  if (t & 1) best1 = fmaxf(best1, lo);
                  else best0 = fmaxf(best0, lo);
                  if constexpr (MODE == MODE_ASSIGN) {
                    if (lo > lmth) {
                      insert_lower_bound(lbm, a.m, lo);
                      lmth = pick8(lbm, a.m - 1);
                    }
                  }
                }
              }
            }
            ref = fmaxf(ref, fmaxf(best0, best1));
          } else {
            // every component whose upper bound
            //   hi = s v + (bias + delta) + rnk |b|
            // reaches the window
#pragma unroll 1
            for (int c0 = 0; c0 < kHalf; c0 += 32) {
              uint32_t u[32];
              tc::tmem_ld32_issue(tcol + (uint32_t)c0, u);
              tc::tmem_wait32(u);
              // a bit per column in the window (no branch in the sweep), then
              // the (rare) appends in column order
              uint32_t pm = 0u;
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                float nb[4], bb[4];
                ld_trail4(tcn + c0 + i, nb);
                ld_trail4(tbh + c0 + i, bb);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                  const float v = __uint_as_float(u[i + t]);
                  const float hi = fmaf(v, Sj, fmaf(rnk, nb[t], bb[t]));
                  pm |= hi >= thr ? (1u << (i + t)) : 0u;
                }
              }
              if (!valid) pm = 0u;
              while (pm) {
                const int kk = c0 + __ffs(pm) - 1;
                pm &= pm - 1u;
                if (cnt < kCS) {
                  ck[cnt * kBM + r] = (uint16_t)(j * kBN + h * kHalf + kk);
                  ++cnt;
                } else {
                  dropped = INFINITY;  // list full: the row goes to the CUDA-core path
                }
              }
            }
          }
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&bar[T_EMPTY + buf]);
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[R_FREE + (it & 1)]);
      if (!ok) break;
      const bool mine = valid && isfinite(rn) && !(dropped >= thr);
      // exact log joints of this half's candidates (same arithmetic as the
      // CUDA-core kernels): the warp's (row, candidate) pairs are numbered by
      // an exclusive scan of the counts and taken eight at a time
      {
        const int mycnt = mine ? cnt : 0;
        int incl = mycnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const int excl = incl - mycnt;
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        // eight pairs per round, one per group of four lanes
        const int grp = lane >> 2, gq = lane & 3;
        for (int p0 = 0; p0 < total; p0 += 8) {
          const int pidx = p0 + grp;
          const bool live = pidx < total;
          // owner lane of pair pidx: the last lane whose excl <= pidx
          int owner = 0;
#pragma unroll
          for (int st = 16; st > 0; st >>= 1) {
            const int cand = owner + st;
            const int ev = __shfl_sync(0xffffffffu, excl, cand & 31);
            if (cand < 32 && ev <= pidx) owner = cand;
          }
          const int e = pidx - __shfl_sync(0xffffffffu, excl, owner);
          const int rr = q * 32 + owner;
          const int k = live ? (int)ck[e * kBM + rr] : 0;
          // (idle groups evaluate row 0 of the tile, which always exists)
          const float d2 = group_d2<D, XT>(a.X, tile * kBM + (live ? rr : 0), g_mu + (size_t)k * D,
                                           iso ? g_prec + k : g_prec + (size_t)k * D, iso, gq);
          if (live && gq == 0) cub[e * kBM + rr] = __ldg(g_c + k) - 0.5f * d2;
        }
        __syncwarp();
      }
      float mx = -INFINITY, ssum = 0.f;
      if (mine && cnt > 0) {
        for (int e = 0; e < cnt; ++e) mx = fmaxf(mx, cub[e * kBM + r]);
        for (int e = 0; e < cnt; ++e) ssum += expf(cub[e * kBM + r] - mx);
      }
      // exchange B: both halves' partial log-sum-exp
      xmx[h * kBM + r] = mx;
      xsum[h * kBM + r] = ssum;
      xcnt[h * kBM + r] = mine ? (uint16_t)cnt : (uint16_t)0xffff;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar[EX_B]);
      if (!warp_wait(&bar[EX_B], it & 1)) { fail(); break; }
      const int c0 = xcnt[r], c1 = xcnt[kBM + r];
      const bool exact = c0 != 0xffff && c1 != 0xffff && c0 + c1 > 0;
      float lse = 0.f;
      if (exact) {
        const float m0 = xmx[r], m1 = xmx[kBM + r];
        const float M = fmaxf(m0, m1);
        float sum = 0.f;
        if (c0 > 0 && m0 > -INFINITY) sum += xsum[r] * expf(m0 - M);
        if (c1 > 0 && m1 > -INFINITY) sum += xsum[kBM + r] * expf(m1 - M);
        lse = M + logf(sum);
      }
      if constexpr (MODE == MODE_EM) {
        // responsibility records of this tile, in row order (half 0's
        // components, then half 1's): an exclusive prefix sum of the rows'
        // counts over the 128 rows.  Rows past the capacity go to the row list.
        const int my = exact ? c0 + c1 : 0;
        // every warp reads all 128 rows' counts (lane: rows 4 lane .. 4 lane + 3)
        int rc[4], tsum = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int rr = lane * 4 + t;
          const int a0 = xcnt[rr], a1 = xcnt[kBM + rr];
          rc[t] = (a0 != 0xffff && a1 != 0xffff) ? a0 + a1 : 0;
          tsum += rc[t];
        }
        int incl = tsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const int all = __shfl_sync(0xffffffffu, incl, 31);
        // exclusive offset of row r = prefix of its group of four + earlier rows in it
        const int grp = r >> 2;
        int off = __shfl_sync(0xffffffffu, incl - tsum, grp);
        const int r0c = __shfl_sync(0xffffffffu, rc[0], grp);
        const int r1c = __shfl_sync(0xffffffffu, rc[1], grp);
        const int r2c = __shfl_sync(0xffffffffu, rc[2], grp);
        const int within = r & 3;
        off += (within > 0 ? r0c : 0) + (within > 1 ? r1c : 0) + (within > 2 ? r2c : 0);
        const bool fits = exact && off + my <= a.rec_cap;
        if (h == 0) {
          if (exact && off <= a.rec_cap && off + my > a.rec_cap) a.tile_cnt[tile] = (uint32_t)off;
          if (r == kBM - 1 && all <= a.rec_cap) a.tile_cnt[tile] = (uint32_t)all;
          if (fits) {
            if (!isfinite(lse)) raise_status(a.st, GMM_ERR_NONFINITE);
            if (a.lse) a.lse[n] = lse;
            ll_acc += (double)lse;
          }
          const unsigned fbm = __ballot_sync(0xffffffffu, valid && !fits);
          if (lane == 0) a.fb_mask[tile * 4 + q] = fbm;
        }
        if (fits) {
          const int mc = h == 0 ? c0 : c1;
          uint2* out = a.recs + (size_t)tile * a.rec_cap + off + (h == 0 ? 0 : c0);
          for (int e = 0; e < mc; ++e) {
            const uint32_t k = ck[e * kBM + r];
            const float gm = expf(cub[e * kBM + r] - lse);
            out[e] = make_uint2((k << 7) | (uint32_t)r, __float_as_uint(gm));
          }
        }
      } else {
        if (h == 0) {
          if (exact) {
            if (!isfinite(lse)) raise_status(a.st, GMM_ERR_NONFINITE);
            if (a.lse) a.lse[n] = lse;
            // top-m over both halves' exact values, ties to the lower component
            uint32_t taken = 0;
            for (int t = 0; t < a.m; ++t) {
              int best = -1, bk = 0x7fffffff;
              float bv = -INFINITY;
              for (int e = 0; e < c0 + c1; ++e) {
                if (taken & (1u << e)) continue;
                const int hh = e < c0 ? 0 : kCS;
                const int ee = e < c0 ? e : e - c0;
                const float v = sCUB[(hh + ee) * kBM + r];
                const int k = sCK[(hh + ee) * kBM + r];
                if (best < 0 || v > bv || (v == bv && k < bk)) { best = e; bv = v; bk = k; }
              }
              if (best < 0) {
                a.ids[n * a.m + t] = -1;
                a.gamma[n * a.m + t] = 0.f;
                continue;
              }
              taken |= 1u << best;
              a.ids[n * a.m + t] = bk;
              a.gamma[n * a.m + t] = bv == -INFINITY ? 0.f : expf(bv - lse);
            }
          }
          const unsigned fbm = __ballot_sync(0xffffffffu, valid && !exact);
          if (lane == 0) a.fb_mask[tile * 4 + q] = fbm;
        }
        // half 1's list stays untouched until half 0 has read it
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar[EX_C]);
        if (!warp_wait(&bar[EX_C], it & 1)) { fail(); break; }
      }
      __syncwarp();
    }
    if constexpr (MODE == MODE_EM) {
      const double s = warp_sum(ll_acc);
      if (lane == 0) ll_red[warp] = s;
    }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if constexpr (MODE == MODE_EM) {
    if (tid == 0 && a.ll_part) {
      double t = 0.0;
      for (int w = 0; w < kEpiWarps; ++w) t += ll_red[w];
      a.ll_part[blockIdx.x] = t;
    }
  }
  if (warp == kMmaWarp) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Ascending list of the rows whose bit is set in the hand-over bitmap (word
// w covers rows 32w .. 32w + 31), in two passes over segments of kSegWords
// words: count per segment, then each segment's block takes its offset (the
// sum of the earlier segments' counts), scans its threads' counts (8
// consecutive words each) and writes its rows in order.
constexpr int kSegThreads = 256;
constexpr int kSegWords = kSegThreads * 8;

__device__ __forceinline__ uint32_t fb_word(const uint32_t* mask, int64_t N, int64_t w) {
  uint32_t m = mask[w];
  const int64_t left = N - w * 32;
  if (left < 32) m &= (1u << left) - 1u;
  return m;
}

__global__ void __launch_bounds__(kSegThreads)
fb_count_kernel(const uint32_t* __restrict__ mask, int64_t N, uint32_t* __restrict__ segcnt) {
  __shared__ uint32_t wsum[kSegThreads / 32];
  const int64_t nwords = (N + 31) / 32;
  const int64_t w0 = (int64_t)blockIdx.x * kSegWords + threadIdx.x * 8;
  uint32_t c = 0;
  for (int i = 0; i < 8; ++i)
    if (w0 + i < nwords) c += __popc(fb_word(mask, N, w0 + i));
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int i = 0; i < kSegThreads / 32; ++i) t += wsum[i];
    segcnt[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(kSegThreads)
fb_write_kernel(const uint32_t* __restrict__ mask, int64_t N, const uint32_t* __restrict__ segcnt,
                uint32_t* __restrict__ rows, uint32_t* __restrict__ count) {
  __shared__ uint32_t wsum[kSegThreads / 32];
  __shared__ uint32_t base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    uint32_t b = 0;
    for (unsigned i = 0; i < blockIdx.x; ++i) b += segcnt[i];
    base = b;
  }
  const int64_t nwords = (N + 31) / 32;
  const int64_t w0 = (int64_t)blockIdx.x * kSegWords + tid * 8;
  uint32_t words[8], mine = 0;
  for (int i = 0; i < 8; ++i) {
    words[i] = w0 + i < nwords ? fb_word(mask, N, w0 + i) : 0u;
    mine += __popc(words[i]);
  }
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t before = base;
  for (int i = 0; i < warp; ++i) before += wsum[i];
  uint32_t pos = before + incl - mine;
  for (int i = 0; i < 8; ++i) {
    uint32_t m = words[i];
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1u;
      rows[pos++] = (uint32_t)((w0 + i) * 32 + b);
    }
  }
  if (blockIdx.x == gridDim.x - 1 && tid == kSegThreads - 1) *count = pos;
}

template <int D, int XT, int MODE>
cudaError_t run_screen(const ScreenArgs& args, int grid, cudaStream_t s) {
  // resident, folded parameters (at most two chunks): the grouped epilogue
  const bool grp = tc_fold(args.L.tc_chunks);
  // the chunk images in global memory must match the shared-memory layout
  if ((size_t)(grp ? Shape<D, true>::B_BYTES : Shape<D, false>::B_BYTES) !=
      args.L.tcB_chunk_bytes)
    return cudaErrorInvalidValue;
  auto kern = grp ? tc_screen_kernel<D, XT, MODE, true> : tc_screen_kernel<D, XT, MODE, false>;
  const int smem = grp ? Shape<D, true>::SMEM : Shape<D, false>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, s>>>(args);
  return cudaGetLastError();
}

}  // namespace

// Grid of the screening kernel: one persistent CTA per SM (capped by tiles).
int tc_screen_grid(int64_t N) {
  static int sms = 0;
  if (!sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  const int64_t tiles = (N + kBM - 1) / kBM;
  return (int)(tiles < sms ? tiles : sms);
}

// mode 0: EM (lse, ll_part, records; streamed parameters also the candidate
// masks and the rows left to the dense-row kernels); mode 1: assign (top-m).
// EM mode: lse (every point's LSE_n, written for all points but those with a
// single candidate unless want_lse) and the records are required.
cudaError_t tc_screen(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                      const void* prepared, int mode, float* lse, int want_lse, double* ll_part,
                      int m, int32_t* ids, float* gamma, uint32_t* fb_mask, uint32_t* cmask,
                      uint32_t* dmask, uint2* recs, uint32_t* tile_cnt, int rec_cap,
                      DeviceStatus* st, cudaStream_t s) {
  ScreenArgs a;
  a.cmask = cmask; a.dmask = dmask;
  a.X = X; a.N = N; a.K = K; a.m = m; a.prepared = prepared;
  a.L = PreparedLayout::make(D, K, cov);
  a.lse = lse; a.want_lse = want_lse; a.ll_part = ll_part; a.ids = ids; a.gamma = gamma;
  a.fb_mask = fb_mask; a.st = st;
  a.recs = recs; a.tile_cnt = tile_cnt; a.rec_cap = rec_cap;
  if (!a.L.tc_chunks || N < 1) return cudaErrorInvalidValue;
  if (mode == MODE_EM && (!recs || !tile_cnt || !lse || rec_cap < kBM)) return cudaErrorInvalidValue;
  if (mode == MODE_EM && (!cmask || !dmask)) return cudaErrorInvalidValue;
  const int grid = tc_screen_grid(N);
#define GMM_SCREEN(DD, XX)                                                              \
  return mode == MODE_EM ? run_screen<DD, XX, MODE_EM>(a, grid, s)                      \
                         : run_screen<DD, XX, MODE_ASSIGN>(a, grid, s)
  if (D == 128) {
    if (xdtype == GMM_F16) { GMM_SCREEN(128, GMM_F16); }
    if (xdtype == GMM_BF16) { GMM_SCREEN(128, GMM_BF16); }
    GMM_SCREEN(128, GMM_F32);
  } else {
    if (xdtype == GMM_F16) { GMM_SCREEN(64, GMM_F16); }
    if (xdtype == GMM_BF16) { GMM_SCREEN(64, GMM_BF16); }
    GMM_SCREEN(64, GMM_F32);
  }
#undef GMM_SCREEN
}

// Rows handed over by the screening launch over N rows -> rows[0 .. *count).
// segcnt: fb_compact_segments(N) words of scratch.
int fb_compact_segments(int64_t N) { return (int)(((N + 31) / 32 + kSegWords - 1) / kSegWords); }

cudaError_t fb_compact(const uint32_t* fb_mask, int64_t N, uint32_t* rows, uint32_t* count,
                       uint32_t* segcnt, cudaStream_t s) {
  const int nseg = fb_compact_segments(N);
  fb_count_kernel<<<nseg, kSegThreads, 0, s>>>(fb_mask, N, segcnt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fb_write_kernel<<<nseg, kSegThreads, 0, s>>>(fb_mask, N, segcnt, rows, count);
  return cudaGetLastError();
}

}  // namespace gmm
