// sparse_stats.cu - sufficient statistics from the tensor-core E-step's
// responsibility records (Flash-GMM summary, Method: online s0, s1, s2).
//
// The screening kernel writes, per 128-point tile, in eight regions (one or
// two per epilogue warp, each in the warp's own order), the (component,
// point, exact log joint l) of every pair it evaluated exactly; the
// responsibility is g = exp(l - LSE_n), or 1 for a record flagged as a
// point's only candidate.  All other pairs carry less than 4.3e-18 of their
// point's responsibility.  The statistics come from the records without an
// N x K matrix, in five steps:
//   count    records per (component, block of kTPB tiles), in shared memory
//   scan     per component (a warp each): its total and the exclusive offsets
//            of its blocks; then one block: the start of each component's
//            records and of its chunks of kCH records
//   scatter  each record to its component's list with its responsibility
//            (a warp per tile, or per block of tiles for large K, walks the
//            tile's regions in order, 32 records at a time; __match_any_sync
//            ranks records of the same component, so the order is fixed)
//   reduce   one warp per chunk: gathers the chunk's rows of X into shared
//            memory by bulk copies (a batch in flight while the previous
//            one is added up), accumulates g, g y, g y^2 with y = x - c_k about the
//            component's input mean c_k (lane l: dimensions l*D/32 ..
//            (l+1)*D/32 - 1), and for the flagged records of points with a
//            single candidate (g = 1) their count and sum of y^2, and writes
//            the chunk's fp32 sums
//   merge    one block per component: adds its chunks in fp64 in order and
//            writes [S0 | S1 about c | M2 about the mean], the partial the
//            M-step merges (continuing the partial of an earlier call when
//            accumulating over slabs or chunks of host data); and the
//            log-likelihood of its single-candidate points,
//            n1 c_k - 1/2 sum_d w_kd Q_d (their LSE is their log joint).
// Every sum is taken in a fixed order, so results are the same on every run.
#include <math.h>

#include "gmm_internal.cuh"
#include "tc_ptx.cuh"

namespace gmm {

cudaError_t launch_ll_finalize(const double* ll_part, int64_t n, double* out, int accumulate,
                               cudaStream_t s);

namespace {

constexpr int kTile = 128;       // points per record tile
constexpr int kTPB = 8;          // tiles per counting / scattering block
constexpr int kCH = 512;         // records per reduction chunk
constexpr int kScanThreads = 1024;

// Shared-memory counters limit the component count of this path.
constexpr int kMaxSparseK = 16384;

struct SparseLayout {
  int64_t ntiles, nb, max_recs, max_chunks;
  size_t off_counts, off_ktot, off_cstart, off_kstart, off_sorted, off_cpart, bytes;
  static SparseLayout make(int64_t rows, int D, int K, int rec_cap) {
    SparseLayout S;
    S.ntiles = (rows + kTile - 1) / kTile;
    S.nb = (S.ntiles + kTPB - 1) / kTPB;
    S.max_recs = S.ntiles * rec_cap;
    S.max_chunks = (S.max_recs + kCH - 1) / kCH + K;
    size_t o = 0;
    S.off_counts = o; o = align_up(o + sizeof(uint32_t) * (size_t)K * S.nb);
    S.off_ktot = o;   o = align_up(o + sizeof(uint32_t) * (size_t)K);
    S.off_cstart = o; o = align_up(o + sizeof(uint32_t) * (size_t)(K + 1));
    S.off_kstart = o; o = align_up(o + sizeof(uint32_t) * (size_t)(K + 1));
    S.off_sorted = o; o = align_up(o + sizeof(uint2) * (size_t)S.max_recs);
    S.off_cpart = o;  o = align_up(o + sizeof(float) * (size_t)S.max_chunks * (2 + 3 * D));
    S.bytes = o;
    return S;
  }
};

// Records of tile t: eight regions of rec_cap / 8, region w holding
// tile_cnt[8 t + w] records.  rec_pos maps the tile's i-th record (regions in
// order) to its position in the buffer.
constexpr int kRegions = 8;
__device__ __forceinline__ uint32_t tile_records(const uint32_t* __restrict__ tile_cnt, int64_t t,
                                                 uint32_t* cnt) {
  uint32_t tot = 0;
#pragma unroll
  for (int w = 0; w < kRegions; ++w) {
    cnt[w] = tile_cnt[t * kRegions + w];
    tot += cnt[w];
  }
  return tot;
}
__device__ __forceinline__ size_t rec_pos(const uint32_t* cnt, int64_t t, int rec_cap, uint32_t i) {
  int w = 0;
  while (w < kRegions - 1 && i >= cnt[w]) { i -= cnt[w]; ++w; }
  return (size_t)t * rec_cap + (size_t)w * (rec_cap / kRegions) + i;
}

// count: block b walks tiles [b kTPB, (b+1) kTPB) and counts its records per
// component in shared memory; column b of counts[k][nb].
__global__ void __launch_bounds__(256)
rec_count_kernel(const uint32_t* __restrict__ tile_cnt, const uint2* __restrict__ recs,
                 int rec_cap, int64_t ntiles, int K, int64_t nb, uint32_t* __restrict__ counts) {
  extern __shared__ uint32_t hist[];
  const int64_t b = blockIdx.x;
  for (int k = threadIdx.x; k < K; k += blockDim.x) hist[k] = 0u;
  __syncthreads();
  const int64_t t1 = min(ntiles, (b + 1) * kTPB);
  for (int64_t t = b * kTPB; t < t1; ++t) {
    uint32_t rc[kRegions];
    const uint32_t cnt = tile_records(tile_cnt, t, rc);
    for (uint32_t i = threadIdx.x; i < cnt; i += blockDim.x) {
      const uint32_t k = (recs[rec_pos(rc, t, rec_cap, i)].x >> 7) & kRecKMask;
      if (k < (uint32_t)K) atomicAdd(&hist[k], 1u);
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += blockDim.x) counts[(size_t)k * nb + b] = hist[k];
}

// Exclusive block-wide prefix of one value per thread (kScanThreads).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t t = wsum[lane];
    uint32_t ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += u;
    }
    wsum[lane] = ti - t;
    if (lane == 31) *total = ti;
  }
  __syncthreads();
  const uint32_t r = wsum[warp] + incl - v;
  __syncthreads();
  return r;
}

// scan, part 1 (one block of kScanThreads per component): counts[k][b] ->
// offsets of block b within component k (in place, exclusive), ktot[k] =
// the component's total.
__global__ void __launch_bounds__(kScanThreads)
rec_scan_blocks_kernel(uint32_t* __restrict__ counts, int K, int64_t nb,
                       uint32_t* __restrict__ ktot) {
  __shared__ uint32_t wsum[kScanThreads / 32];
  __shared__ uint32_t total;
  const int k = blockIdx.x;
  uint32_t* c = counts + (size_t)k * nb;
  uint32_t carry = 0;
  for (int64_t base = 0; base < nb; base += kScanThreads) {
    const int64_t i = base + threadIdx.x;
    const uint32_t v = i < nb ? c[i] : 0u;
    const uint32_t ex = block_excl_scan(v, wsum, &total);
    if (i < nb) c[i] = carry + ex;
    carry += total;
    __syncthreads();  // total is rewritten by the next round
  }
  if (threadIdx.x == 0) ktot[k] = carry;
}

// scan, part 2 (one block): cstart[k] = first record of component k
// (cstart[K] = total); kstart[k] = first chunk of component k (kstart[K] =
// chunk count).
__global__ void __launch_bounds__(kScanThreads)
rec_scan_comps_kernel(const uint32_t* __restrict__ ktot, int K, uint32_t* __restrict__ cstart,
                      uint32_t* __restrict__ kstart) {
  __shared__ uint32_t wsum[kScanThreads / 32];
  __shared__ uint32_t total;
  const int kper = (K + kScanThreads - 1) / kScanThreads;
  const int k0 = min(K, (int)threadIdx.x * kper), k1 = min(K, k0 + kper);
  uint32_t mine = 0, nch = 0;
  for (int k = k0; k < k1; ++k) {
    mine += ktot[k];
    nch += (ktot[k] + kCH - 1) / kCH;
  }
  uint32_t run = block_excl_scan(mine, wsum, &total);
  for (int k = k0; k < k1; ++k) {
    cstart[k] = run;
    run += ktot[k];
  }
  if (threadIdx.x == 0) cstart[K] = total;
  uint32_t krun = block_excl_scan(nch, wsum, &total);
  for (int k = k0; k < k1; ++k) {
    kstart[k] = krun;
    krun += (ktot[k] + kCH - 1) / kCH;
  }
  if (threadIdx.x == 0) kstart[K] = total;
}

// Responsibility of a record: 1 for a point's only candidate, else
// exp(l - LSE_n).
__device__ __forceinline__ float rec_gamma(uint2 rec, int64_t t, const float* __restrict__ lse) {
  if (rec.x & kRecSingle) return 1.f;
  return expf(__uint_as_float(rec.y) - lse[t * kTile + (rec.x & 127)]);
}

// scatter: the warp of block b places the block's records, tile by tile and
// region by region, at their component's offsets: sorted[] = {single flag |
// point index in this call, gamma}.
__global__ void __launch_bounds__(32)
rec_scatter_kernel(const uint32_t* __restrict__ tile_cnt, const uint2* __restrict__ recs,
                   int rec_cap, int64_t ntiles, int K, int64_t nb,
                   const uint32_t* __restrict__ offsets, const uint32_t* __restrict__ cstart,
                   const float* __restrict__ lse, uint2* __restrict__ sorted) {
  extern __shared__ uint32_t cursor[];
  const int64_t b = blockIdx.x;
  const int lane = threadIdx.x;
  for (int k = lane; k < K; k += 32) cursor[k] = cstart[k] + offsets[(size_t)k * nb + b];
  __syncwarp();
  const int64_t t1 = min(ntiles, (b + 1) * kTPB);
  for (int64_t t = b * kTPB; t < t1; ++t) {
    uint32_t rc[kRegions];
    const uint32_t cnt = tile_records(tile_cnt, t, rc);
    for (uint32_t base = 0; base < cnt; base += 32) {
      const uint32_t i = base + lane;
      const bool live = i < cnt;
      uint2 rec = make_uint2(0xffffffffu, 0u);
      if (live) rec = recs[rec_pos(rc, t, rec_cap, i)];
      const uint32_t k = (rec.x >> 7) & kRecKMask;
      const bool ok = live && k < (uint32_t)K;
      const unsigned grp = __match_any_sync(0xffffffffu, ok ? k : 0xffffffffu);
      if (ok) {
        const uint32_t pos = cursor[k] + __popc(grp & ((1u << lane) - 1u));
        sorted[pos] = make_uint2((uint32_t)(t * kTile + (rec.x & 127)) | (rec.x & kRecSingle),
                                 __float_as_uint(rec_gamma(rec, t, lse)));
      }
      __syncwarp();
      if (ok && lane == 31 - __clz(grp)) cursor[k] += __popc(grp);
      __syncwarp();
    }
  }
}

// DPL consecutive coordinates of one row staged in shared memory, as float.
// scatter with a warp per tile (K <= kScatterWideK): the block's eight
// warps first count their tiles' records per component (cnt[w][k]), turn
// the counts into each tile's starting positions (the block's offset plus
// the earlier tiles' counts), then place their records as the one-warp
// kernel does.  The positions are the same as that kernel's.
constexpr int kScatterWideK = 1024;
__global__ void __launch_bounds__(32 * kTPB)
rec_scatter_wide_kernel(const uint32_t* __restrict__ tile_cnt, const uint2* __restrict__ recs,
                        int rec_cap, int64_t ntiles, int K, int64_t nb,
                        const uint32_t* __restrict__ offsets, const uint32_t* __restrict__ cstart,
                        const float* __restrict__ lse, uint2* __restrict__ sorted) {
  extern __shared__ uint32_t pos[];  // [kTPB][K]
  const int64_t b = blockIdx.x;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kTPB * K; i += blockDim.x) pos[i] = 0u;
  __syncthreads();
  const int64_t t = b * kTPB + w;
  uint32_t cnt = 0;
  uint32_t rc[kRegions];
  if (t < ntiles) {
    cnt = tile_records(tile_cnt, t, rc);
    for (uint32_t i = lane; i < cnt; i += 32) {
      const uint32_t k = (recs[rec_pos(rc, t, rec_cap, i)].x >> 7) & kRecKMask;
      if (k < (uint32_t)K) atomicAdd(&pos[w * K + k], 1u);
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    uint32_t run = cstart[k] + offsets[(size_t)k * nb + b];
#pragma unroll
    for (int v = 0; v < kTPB; ++v) {
      const uint32_t n = pos[v * K + k];
      pos[v * K + k] = run;
      run += n;
    }
  }
  __syncthreads();
  uint32_t* cursor = pos + w * K;
  for (uint32_t base = 0; base < cnt; base += 32) {
    const uint32_t i = base + lane;
    const bool live = i < cnt;
    uint2 rec = make_uint2(0xffffffffu, 0u);
    if (live) rec = recs[rec_pos(rc, t, rec_cap, i)];
    const uint32_t k = (rec.x >> 7) & kRecKMask;
    const bool ok = live && k < (uint32_t)K;
    const unsigned grp = __match_any_sync(0xffffffffu, ok ? k : 0xffffffffu);
    if (ok) {
      const uint32_t at_ = cursor[k] + __popc(grp & ((1u << lane) - 1u));
      sorted[at_] = make_uint2((uint32_t)(t * kTile + (rec.x & 127)) | (rec.x & kRecSingle),
                               __float_as_uint(rec_gamma(rec, t, lse)));
    }
    __syncwarp();
    if (ok && lane == 31 - __clz(grp)) cursor[k] += __popc(grp);
    __syncwarp();
  }
}

template <int XT, int DPL>
__device__ __forceinline__ void staged_row(const unsigned char* row, int d0, float* v) {
  if constexpr (XT == GMM_F32) {
    const float* p = reinterpret_cast<const float*>(row) + d0;
    if constexpr (DPL == 4) {
      const float4 q = *reinterpret_cast<const float4*>(p);
      v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
      const float2 q = *reinterpret_cast<const float2*>(p);
      v[0] = q.x; v[1] = q.y;
    }
  } else {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(row) + d0;
    uint32_t u[DPL / 2];
    if constexpr (DPL == 4) {
      const uint2 q = *reinterpret_cast<const uint2*>(p);
      u[0] = q.x; u[1] = q.y;
    } else {
      u[0] = *reinterpret_cast<const uint32_t*>(p);
    }
#pragma unroll
    for (int i = 0; i < DPL / 2; ++i) {
      float2 f;
      if constexpr (XT == GMM_F16) f = __half22float2(*reinterpret_cast<const __half2*>(&u[i]));
      else f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
}

constexpr int kReduceThreads = 256;
constexpr uint32_t kReduceWait = 1u << 22;

// Rows of X per batch and warp (staged twice: this batch and the next).
template <int XT>
__host__ __device__ constexpr int reduce_batch() { return XT == GMM_F32 ? 8 : 16; }

template <int D, int XT>
constexpr size_t reduce_smem() {
  return (size_t)(kReduceThreads / 32) * 2 * reduce_batch<XT>() * D * (XT == GMM_F32 ? 4 : 2) +
         (size_t)(kReduceThreads / 32) * 2 * sizeof(uint64_t);
}

// reduce: warp-per-chunk, grid-stride over the chunks.  Each batch's rows
// of X arrive in the warp's shared-memory stage by one bulk copy per row
// (lane u copies row u), double buffered, so the next batch is in flight
// while this one is accumulated.  Chunk sums cpart[c] = [s0 | s1 (D) | s2 (D)
// | n1 | q1 (D)] in fp32 (n1, q1: count and sum of y^2 of the flagged
// single-candidate records).
template <int D, int XT>
__global__ void __launch_bounds__(kReduceThreads)
rec_reduce_kernel(const void* __restrict__ X, int K, const float* __restrict__ mu,
                  const uint32_t* __restrict__ cstart, const uint32_t* __restrict__ kstart,
                  const uint2* __restrict__ sorted, float* __restrict__ cpart, DeviceStatus* st) {
  constexpr int DPL = D / 32, F = 2 + 3 * D, B = reduce_batch<XT>();
  constexpr int ROWB = D * (XT == GMM_F32 ? 4 : 2);
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  unsigned char* stage = smem + (size_t)wib * 2 * B * ROWB;  // [2][B][ROWB]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (size_t)(kReduceThreads / 32) * 2 * B * ROWB) +
                  2 * wib;
  if (lane == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_fence_init();
  }
  __syncwarp();
  uint32_t ph = 0u;  // bit b: parity of the next phase of stage buffer b
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const uint32_t nchunks = kstart[K];
  bool ok = true;
  for (int64_t c = gw; c < nchunks && ok; c += nw) {
    // component of chunk c: the last k with kstart[k] <= c
    int lo = 0, hi = K - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (kstart[mid] <= (uint32_t)c) lo = mid; else hi = mid - 1;
    }
    const int k = lo;
    const uint32_t r0 = cstart[k] + (uint32_t)(c - kstart[k]) * kCH;
    const uint32_t r1 = min(cstart[k + 1], r0 + kCH);
    float cen[DPL], s1[DPL], s2[DPL], q1[DPL], s0 = 0.f, n1 = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      cen[i] = __ldg(mu + (size_t)k * D + lane * DPL + i);
      s1[i] = s2[i] = q1[i] = 0.f;
    }
    // lanes 0 .. B-1 hold the records of the batch at r; lane u copies row u
    auto issue = [&](uint32_t r, int b, uint2* rec) {
      const int nb = (int)min((uint32_t)B, r1 - r);
      *rec = lane < nb ? sorted[r + lane] : make_uint2(0u, 0u);
      if (lane == 0) tc::mbar_arrive_expect_tx(&bar[b], (uint32_t)(nb * ROWB));
      __syncwarp();
      if (lane < nb)
        tc::bulk_g2s(stage + ((size_t)b * B + lane) * ROWB,
                     static_cast<const unsigned char*>(X) + (size_t)(rec->x & ~kRecSingle) * ROWB,
                     ROWB, &bar[b]);
    };
    uint2 cur, nxt = make_uint2(0u, 0u);
    int b = 0;
    issue(r0, 0, &cur);
    for (uint32_t r = r0; r < r1; r += B) {
      // the next batch goes to the other buffer, read in the previous round
      if (r + B < r1) issue(r + B, b ^ 1, &nxt);
      const bool got = tc::mbar_wait(&bar[b], (ph >> b) & 1u, kReduceWait);
      ph ^= 1u << b;
      if (!__all_sync(0xffffffffu, got)) {
        // wait (bounded) for the copies still in flight, then stop
        if (!got) tc::mbar_wait(&bar[b], ((ph >> b) & 1u) ^ 1u, kReduceWait);
        if (r + B < r1) tc::mbar_wait(&bar[b ^ 1], (ph >> (b ^ 1)) & 1u, kReduceWait);
        if (lane == 0) raise_status(st, GMM_ERR_TIMEOUT);
        ok = false;
        break;
      }
      const int nb = (int)min((uint32_t)B, r1 - r);
      for (int u = 0; u < nb; ++u) {
        const uint32_t key = __shfl_sync(0xffffffffu, cur.x, u);
        const float g = __uint_as_float(__shfl_sync(0xffffffffu, cur.y, u));
        const bool single = (key & kRecSingle) != 0u;
        float x[DPL];
        staged_row<XT, DPL>(stage + ((size_t)b * B + u) * ROWB, lane * DPL, x);
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          const float y = x[i] - cen[i];
          const float gy = g * y;
          s1[i] += gy;
          s2[i] = fmaf(gy, y, s2[i]);
          if (single) q1[i] = fmaf(y, y, q1[i]);
        }
        s0 += g;
        if (single) n1 += 1.f;
      }
      __syncwarp();  // every lane has read buffer b before it is refilled
      cur = nxt;
      b ^= 1;
    }
    if (!ok) break;
    float* o = cpart + (size_t)c * F;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      o[1 + lane * DPL + i] = s1[i];
      o[1 + D + lane * DPL + i] = s2[i];
      o[2 + 2 * D + lane * DPL + i] = q1[i];
    }
    if (lane == 0) {
      o[0] = s0;
      o[1 + 2 * D] = n1;
    }
  }
}

// merge: one block of D threads per component (thread d: dimension d);
// partial [S0 | S1 about c | M2 about the mean], and llk[k] = n1 c_k - 1/2
// sum_d w_kd Q_d, the log-likelihood of the component's single-candidate
// points (each one's LSE is its log joint c_k - 1/2 sum_d w_kd (x_d -
// c_kd)^2, the centre c_k being the input mean).
template <int D>
__global__ void __launch_bounds__(D)
rec_merge_kernel(int K, const uint32_t* __restrict__ kstart, const float* __restrict__ cpart,
                 const float* __restrict__ bias_c, const float* __restrict__ prec, bool iso,
                 double* __restrict__ part, double* __restrict__ llk, int accumulate) {
  constexpr int F = 1 + 2 * D, FC = 2 + 3 * D;
  __shared__ double red[D / 32];
  const int k = blockIdx.x, d = threadIdx.x, lane = d & 31;
  double* o = part + (size_t)k * F;
  const uint32_t c0 = kstart[k], c1 = kstart[k + 1];
  // the chunk sums are fp32 sums of up to kCH records; adding them up in
  // fp32 (even and odd chunks apart, then together) keeps their accuracy,
  // and the FP64 pipe is left for the second moment below
  float a0[2] = {0.f, 0.f}, an[2] = {0.f, 0.f}, a1[2] = {0.f, 0.f}, a2[2] = {0.f, 0.f},
        aq[2] = {0.f, 0.f};
#pragma unroll 4
  for (uint32_t c = c0; c < c1; ++c) {
    const float* cp = cpart + (size_t)c * FC;
    const int h = (int)((c - c0) & 1u);
    a0[h] += cp[0];
    an[h] += cp[1 + 2 * D];
    a1[h] += cp[1 + d];
    a2[h] += cp[1 + D + d];
    aq[h] += cp[2 + 2 * D + d];
  }
  const double s0 = (double)a0[0] + (double)a0[1], n1 = (double)an[0] + (double)an[1];
  double S1 = (double)a1[0] + (double)a1[1], S2c = (double)a2[0] + (double)a2[1];
  const double Q = (double)aq[0] + (double)aq[1];
  const double S0o = accumulate ? o[0] : 0.0;
  const double S0 = S0o + s0;
  if (accumulate) {
    // continue the earlier partial: its second moment back about c
    const double o1 = o[1 + d];
    S2c += o[1 + D + d] + (S0o > 0.0 ? o1 * o1 / S0o : 0.0);
    S1 += o1;
  }
  const double wq = warp_sum((double)(iso ? prec[k] : prec[(size_t)k * D + d]) * Q);
  if (lane == 0) red[d >> 5] = wq;
  __syncthreads();  // every thread has read o[0] (S0o) before it is rewritten
  o[1 + d] = S1;
  o[1 + D + d] = S0 > 0.0 ? S2c - S1 * S1 / S0 : 0.0;
  if (d == 0) {
    double t = 0.0;
    for (int w = 0; w < D / 32; ++w) t += red[w];
    o[0] = S0;
    llk[k] = n1 > 0.0 ? n1 * (double)bias_c[k] - 0.5 * t : 0.0;
  }
}

int g_sms = 0;

}  // namespace

// Workspace of sparse_stats for calls of up to `rows` points.
size_t sparse_stats_ws_bytes(int64_t rows, int D, int K, int rec_cap) {
  return SparseLayout::make(rows, D, K, rec_cap).bytes;
}

bool sparse_stats_supported(int K) { return K <= kMaxSparseK; }

// Diagonal / isotropic statistics (the partial layout is the same for both;
// the isotropic M-step averages the diagonal) into ONE partial slot, part;
// llk[k] (K doubles) receives the log-likelihood of component k's
// single-candidate points.
// prepared: the block written for this call's parameters (its mean array is
// the centre c).  accumulate: continue the partial of an earlier call.
// sws: sparse_stats_ws_bytes(N, D, K, rec_cap) bytes, 256-byte aligned.
cudaError_t sparse_stats(const void* X, int xdtype, int64_t N, int D, int K, const void* prepared,
                         int cov, const float* lse, const uint32_t* tile_cnt, const uint2* recs,
                         int rec_cap, void* sws, double* part, int accumulate, double* llk,
                         DeviceStatus* st, cudaStream_t s) {
  if (K > kMaxSparseK || (D != 64 && D != 128)) return cudaErrorInvalidValue;
  const SparseLayout S = SparseLayout::make(N, D, K, rec_cap);
  const PreparedLayout L = PreparedLayout::make(D, K, cov);
  uint32_t* counts = at<uint32_t>(sws, S.off_counts);
  uint32_t* ktot = at<uint32_t>(sws, S.off_ktot);
  uint32_t* cstart = at<uint32_t>(sws, S.off_cstart);
  uint32_t* kstart = at<uint32_t>(sws, S.off_kstart);
  uint2* sorted = at<uint2>(sws, S.off_sorted);
  float* cpart = at<float>(sws, S.off_cpart);
  const size_t hsm = sizeof(uint32_t) * (size_t)K;
  cudaError_t e;
  if (hsm > 48 * 1024) {
    e = cudaFuncSetAttribute(rec_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsm);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(rec_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsm);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope p("rec_count_kernel", s);
    rec_count_kernel<<<(unsigned)S.nb, 256, hsm, s>>>(tile_cnt, recs, rec_cap, S.ntiles, K, S.nb,
                                                      counts);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope p("rec_scan_kernels", s, 2);
    rec_scan_blocks_kernel<<<(unsigned)K, kScanThreads, 0, s>>>(counts, K, S.nb, ktot);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    rec_scan_comps_kernel<<<1, kScanThreads, 0, s>>>(ktot, K, cstart, kstart);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    ProfScope p("rec_scatter_kernel", s);
    if (K <= kScatterWideK) {
      const size_t wsm = sizeof(uint32_t) * (size_t)kTPB * K;
      if (wsm > 48 * 1024) {
        e = cudaFuncSetAttribute(rec_scatter_wide_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsm);
        if (e != cudaSuccess) return e;
      }
      rec_scatter_wide_kernel<<<(unsigned)S.nb, 32 * kTPB, wsm, s>>>(
          tile_cnt, recs, rec_cap, S.ntiles, K, S.nb, counts, cstart, lse, sorted);
    } else {
      rec_scatter_kernel<<<(unsigned)S.nb, 32, hsm, s>>>(tile_cnt, recs, rec_cap, S.ntiles, K,
                                                         S.nb, counts, cstart, lse, sorted);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (!g_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_sms <= 0) g_sms = 1;
  }
  const float* mu = at<float>(prepared, L.off_mu);
  const unsigned rblocks = (unsigned)g_sms * 8;
#define GMM_REDUCE(DD, XX)                                                                    \
  do {                                                                                        \
    constexpr size_t sm = reduce_smem<DD, XX>();                                              \
    e = cudaFuncSetAttribute(rec_reduce_kernel<DD, XX>,                                       \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);           \
    if (e != cudaSuccess) return e;                                                           \
    rec_reduce_kernel<DD, XX><<<rblocks, kReduceThreads, sm, s>>>(X, K, mu, cstart, kstart,   \
                                                                  sorted, cpart, st);         \
  } while (0)
  {
    ProfScope prof_reduce("rec_reduce_kernel", s);
    if (D == 128) {
      if (xdtype == GMM_F16) GMM_REDUCE(128, GMM_F16);
      else if (xdtype == GMM_BF16) GMM_REDUCE(128, GMM_BF16);
      else GMM_REDUCE(128, GMM_F32);
    } else {
      if (xdtype == GMM_F16) GMM_REDUCE(64, GMM_F16);
      else if (xdtype == GMM_BF16) GMM_REDUCE(64, GMM_BF16);
      else GMM_REDUCE(64, GMM_F32);
    }
#undef GMM_REDUCE
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  const float* bias_c = at<float>(prepared, L.off_c);
  const float* prec = at<float>(prepared, L.off_prec);
  const bool iso = cov == GMM_COV_ISO;
  {
    ProfScope prof_merge("rec_merge_kernel", s);
    if (D == 128)
      rec_merge_kernel<128><<<K, 128, 0, s>>>(K, kstart, cpart, bias_c, prec, iso, part, llk,
                                              accumulate);
    else
      rec_merge_kernel<64><<<K, 64, 0, s>>>(K, kstart, cpart, bias_c, prec, iso, part, llk,
                                            accumulate);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace gmm
