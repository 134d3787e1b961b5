// gmm_api.cu - the C ABI declared in include/gmm.h: argument checks,
// workspace layout and the order of kernel launches for one EM iteration.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "gmm_internal.cuh"

namespace gmm {

cudaError_t launch_prepare(const gmm_params* p, int D, int K, int cov, float ridge_rel,
                           void* prepared, DeviceStatus* st, cudaStream_t s);
cudaError_t simt_lse(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                     const void* prepared, float* lse, double* ll_part, int m, int32_t* ids,
                     float* gamma, DeviceStatus* st, cudaStream_t s);
cudaError_t simt_lse_rows(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                          const void* prepared, float* lse, double* ll_part, int m, int32_t* ids,
                          float* gamma, DeviceStatus* st, const uint32_t* rows,
                          const uint32_t* row_count, int grid, cudaStream_t s);
cudaError_t tc_screen(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                      const void* prepared, int mode, float* lse, int want_lse, double* ll_part,
                      int m, int32_t* ids, float* gamma, uint32_t* fb_mask, uint32_t* cmask,
                      uint32_t* dmask, uint2* recs, uint32_t* tile_cnt, int rec_cap,
                      DeviceStatus* st, cudaStream_t s);
int dense_ll_parts();
int dense_stat_parts(int D, int K);
cudaError_t dense_rows(const void* X, int xdtype, int D, int K, int cov, const void* prepared,
                       const uint32_t* rows, const uint32_t* count, const uint32_t* cmask,
                       float2* part, float* lse, double* ll_part, double* stat, int accumulate,
                       DeviceStatus* st, cudaStream_t s);
int tc_screen_grid(int64_t N);
cudaError_t fb_compact(const uint32_t* fb_mask, int64_t N, uint32_t* rows, uint32_t* count,
                       uint32_t* segcnt, cudaStream_t s);
int fb_compact_segments(int64_t N);
cudaError_t simt_stats(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                       const void* prepared, const float* lse, int parts, double* part,
                       int accumulate, cudaStream_t s);
cudaError_t simt_stats_rows(const void* X, int xdtype, int64_t N, int D, int K, int cov,
                            const void* prepared, const float* lse, int parts, double* part,
                            int accumulate, const uint32_t* rows, const uint32_t* row_count,
                            cudaStream_t s);
size_t sparse_stats_ws_bytes(int64_t rows, int D, int K, int rec_cap);
bool sparse_stats_supported(int K);
cudaError_t sparse_stats(const void* X, int xdtype, int64_t N, int D, int K, const void* prepared,
                         int cov, const float* lse, const uint32_t* tile_cnt, const uint2* recs,
                         int rec_cap, void* sws, double* part, int accumulate, double* ll,
                         DeviceStatus* st, cudaStream_t s);
int simt_stat_chunk(int D, int cov);
cudaError_t launch_mstep(const double* part, int parts, int64_t N, int D, int K, int cov,
                         const float* centre, const int32_t* prep_flags, float var_floor,
                         float min_s0, gmm_params* p, int32_t* flags_out, cudaStream_t s);
cudaError_t launch_ll_finalize(const double* ll_part, int64_t n, double* out, int accumulate,
                               cudaStream_t s);
bool fc_eligible(int D, int K, int cov);
int fc_ll_parts(int64_t N);
cudaError_t fc_estep(const void* X, int xdtype, int64_t N, int D, int K, const void* prepared,
                     uint32_t* mask, bool screen, float* lse, double* ll_part, double* stat,
                     int parts, int accumulate, DeviceStatus* st, cudaStream_t s);

namespace {

constexpr int kTargetCtas = 608;   // 4 x 152 SMs: statistics blocks per launch
constexpr int kListGrid = 304;     // blocks of the CUDA-core pass over handed-over rows
constexpr int kMaxScreenGrid = 1024;  // upper bound of tc_screen_grid (SM count)
// Tensor-core path: records {key, exact log joint} per 128-point tile, in
// eight regions (one per epilogue warp and column half), and rows per slab
// (one screening launch; its records are consumed before the next slab).  A
// point keeps at most 13 (folded parameters) or 2 x 15 (streamed) candidates
// in its lists, and a point with more goes to the dense-row kernels, so a
// region of 32 points never needs more than 32 x 15 = 480 records: 32 records
// a point per tile.
int rec_cap_for(int K) {
  (void)K;
  return 128 * 32;
}
int64_t slab_rows_for(int K) {
  (void)K;
  return (int64_t)1 << 21;
}

bool valid_d(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }
size_t esize(int xdtype) { return xdtype == GMM_F32 ? 4 : 2; }

// Point partitions of the statistics kernel: enough blocks to fill the GPU,
// fixed by the sizes alone so the reduction order never depends on the device.
int stat_parts(int64_t N, int D, int K, int cov) {
  const int kc = simt_stat_chunk(D, cov);
  const int64_t chunks = (K + kc - 1) / kc;
  int64_t p = (kTargetCtas + chunks - 1) / chunks;
  const int64_t tiles = (N + 63) / 64;
  if (p > tiles) p = tiles;
  if (p < 1) p = 1;
  return (int)p;
}

struct WsLayout {
  size_t off_status, off_prep, off_lse, off_llpart, off_ll, off_part, off_flags, off_fb,
      off_fbm, off_fbseg, off_rec, off_tcnt, off_sws, off_cmask, off_dmask, off_drows, off_dpart,
      off_stage, bytes;
  int parts;          // statistics partials of the CUDA-core path
  int sp_parts;       // tensor-core path: the records' partial (1) ...
  int lp_parts;       // ... followed by those of the row-list pass ...
  int dp_parts;       // ... and those of the dense-row kernels
  int64_t lse_rows;
};

// The tensor-core E-step of an EM iteration (screening + statistics from
// its records).
bool use_tc(int D, int K, int cov, const gmm_opts& o) {
  return tc_eligible(D, cov) && sparse_stats_supported(K) && !(o.flags & GMM_OPT_CUDA_CORES);
}

// The full-covariance path for few components (candidate masks, exact
// log joints and statistics with every W in shared memory).
bool use_fc(int D, int K, int cov, const gmm_opts& o) {
  return fc_eligible(D, K, cov) && !(o.flags & GMM_OPT_CUDA_CORES);
}

// rows: rows processed per launch (N, or the chunk size of the host path);
// stage_bytes: host path staging buffers (0 otherwise).
WsLayout ws_layout(int64_t N, int64_t rows, int D, int K, int cov, size_t stage_bytes) {
  WsLayout W;
  size_t o = 0;
  W.off_status = o; o = align_up(o + sizeof(DeviceStatus));
  W.off_prep = o;   o = align_up(o + PreparedLayout::make(D, K, cov).bytes);
  W.lse_rows = rows;
  W.off_lse = o;    o = align_up(o + sizeof(float) * (size_t)rows);
  const bool tc = tc_eligible(D, cov);
  {
    // dense LSE blocks, or per slab the tensor-core CTAs and the components
    // (single-candidate points), then the list blocks
    const size_t dense = (size_t)((rows + kLseRows - 1) / kLseRows);
    const size_t nslabs = (size_t)((rows + slab_rows_for(K) - 1) / slab_rows_for(K));
    const size_t tcl =
        tc ? nslabs * (size_t)(kMaxScreenGrid + K + dense_ll_parts()) + kListGrid : 0;
    W.off_llpart = o; o = align_up(o + sizeof(double) * (dense > tcl ? dense : tcl));
  }
  W.off_ll = o;     o = align_up(o + sizeof(double));
  W.parts = stat_parts(rows, D, K, cov);
  W.sp_parts = W.lp_parts = W.dp_parts = 0;
  int slots = W.parts;
  const bool dense_rows_on = tc;  // rows whose candidate lists fill go to the dense-row kernels
  if (tc) {
    W.sp_parts = 1;
    const int kc = simt_stat_chunk(D, cov);
    const int chunks = (K + kc - 1) / kc;
    W.lp_parts = (kListGrid + chunks - 1) / chunks;
    W.dp_parts = dense_rows_on ? dense_stat_parts(D, K) : 0;
    if (W.sp_parts + W.lp_parts + W.dp_parts > slots) slots = W.sp_parts + W.lp_parts + W.dp_parts;
  }
  W.off_part = o;   o = align_up(o + sizeof(double) * (size_t)slots * K * stat_width(D, cov));
  W.off_flags = o;  o = align_up(o + sizeof(int32_t) * K);
  const int64_t slab_max = slab_rows_for(K);
  const int64_t slab = rows < slab_max ? rows : slab_max;
  // hand-over bitmap and row list: for all rows of the call (handled once, after the slabs)
  W.off_fb = o;     o = align_up(o + sizeof(uint32_t) * (size_t)rows);
  const size_t slab_tiles = tc ? (size_t)((slab + 127) / 128) : 0;
  W.off_fbm = o;    o = align_up(o + sizeof(uint32_t) * 4 * (size_t)((rows + 127) / 128));
  W.off_fbseg = o;  o = align_up(o + sizeof(uint32_t) * (tc ? fb_compact_segments(rows) : 0));
  W.off_rec = o;    o = align_up(o + sizeof(uint2) * slab_tiles * (size_t)rec_cap_for(K));
  W.off_tcnt = o;   o = align_up(o + sizeof(uint32_t) * 8 * slab_tiles);
  W.off_sws = o;
  o = align_up(o + (tc ? sparse_stats_ws_bytes(slab, D, K, rec_cap_for(K)) : 0));
  // every row's candidate masks, the rows left to the
  // dense-row kernels (bitmap, list) and their per-chunk log-sum-exp
  const size_t nch = (size_t)((K + kTcChunk - 1) / kTcChunk);
  W.off_cmask = o;  o = align_up(o + (dense_rows_on ? sizeof(uint32_t) * 4 * nch * (size_t)slab : 0));
  W.off_dmask = o;  o = align_up(o + (dense_rows_on ? sizeof(uint32_t) * 4 * slab_tiles : 0));
  W.off_drows = o;  o = align_up(o + (dense_rows_on ? sizeof(uint32_t) * (size_t)slab : 0));
  W.off_dpart = o;  o = align_up(o + (dense_rows_on ? sizeof(float2) * 2 * nch * (size_t)slab : 0));
  W.off_stage = o;  o = align_up(o + stage_bytes);
  W.bytes = o;
  (void)N;
  return W;
}

gmm_status check_common(const void* X, gmm_dtype xdtype, int64_t N, int D, int K, int cov) {
  if (!X || N < 1 || K < 1 || K > kMaxK) return GMM_ERR_INVALID_ARG;
  if (xdtype < GMM_F32 || xdtype > GMM_BF16) return GMM_ERR_INVALID_ARG;
  if (cov < GMM_COV_FULL || cov > GMM_COV_ISO) return GMM_ERR_INVALID_ARG;
  if (!valid_d(D)) return D > 0 ? GMM_ERR_UNSUPPORTED : GMM_ERR_INVALID_ARG;
  return GMM_OK;
}

gmm_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return GMM_OK;
  fprintf(stderr, "libgmm: CUDA error %s\n", cudaGetErrorString(e));
  return GMM_ERR_CUDA;
}

#define GMM_TRY(expr)                                  \
  do {                                                 \
    gmm_status _s = cuda_status(expr);                 \
    if (_s != GMM_OK) return _s;                       \
  } while (0)

// ---------------------------------------------------------------- profiler
// When enabled, every kernel launch of the library is bracketed by two CUDA
// events recorded on the launching stream; gmm_profile_read sums them per
// kernel.  Off by default (no events recorded).
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
  int kernels;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;
struct ProfSum { const char* name; double ms; long launches; };
std::vector<ProfSum> g_prof_sum;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) { cudaEvent_t e = g_prof_pool.back(); g_prof_pool.pop_back(); return e; }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}


#define GMM_PROF(name) ProfScope _prof_scope(name, s)
#define GMM_PROFN(name, n) ProfScope _prof_scope(name, s, n)

// The E-step and statistics for one block of rows, accumulating into the
// workspace partials (accumulate = 0 for the first block of an iteration).
// lse: LSE_n of the rows (the caller's array, or workspace); want_lse: the
// caller asked for it (otherwise the screen skips the exact log joint of
// points with a single candidate).
gmm_status estep_rows(const void* X, gmm_dtype xdtype, int64_t rows, int D, int K, int cov,
                      const WsLayout& W, void* ws, float* lse, bool want_lse, int accumulate,
                      bool tc, bool fc, cudaStream_t s) {
  DeviceStatus* st = at<DeviceStatus>(ws, W.off_status);
  const void* prep = at<char>(ws, W.off_prep);
  double* llp = at<double>(ws, W.off_llpart);
  if (fc) {
    // candidate masks (in the hand-over bitmap's space: one word a row),
    // exact LSE_n and statistics of the candidates, the log-likelihood
    GMM_TRY(fc_estep(X, xdtype, rows, D, K, prep, at<uint32_t>(ws, W.off_fb), true, lse, llp,
                     at<double>(ws, W.off_part), W.parts, accumulate, st, s));
    {
      GMM_PROF("ll_finalize_kernel");
      GMM_TRY(launch_ll_finalize(llp, fc_ll_parts(rows), at<double>(ws, W.off_ll), accumulate, s));
    }
    return GMM_OK;
  }
  if (tc) {
    // Slabs of rows.  Per slab: screen on the tensor cores (exact LSE_n of
    // the points and records of their candidates) and statistics from the
    // records.  Then, once for all rows: the CUDA-core passes over the rows
    // handed over (a warp's records past its region, non-finite input) and
    // the log-likelihood from every partial (zeroed first, so unused slots
    // count nothing).
    uint32_t* fb = at<uint32_t>(ws, W.off_fb);
    uint32_t* fbm = at<uint32_t>(ws, W.off_fbm);
    uint2* recs = at<uint2>(ws, W.off_rec);
    uint32_t* tcnt = at<uint32_t>(ws, W.off_tcnt);
    double* part = at<double>(ws, W.off_part);
    double* lpart = part + (size_t)W.sp_parts * K * stat_width(D, cov);
    const int64_t slab_rows = slab_rows_for(K);
    const int rec_cap = rec_cap_for(K);
    const int64_t nslabs = (rows + slab_rows - 1) / slab_rows;
    // log-likelihood partials per slab: screening blocks, components
    // (single-candidate points), dense-row blocks
    const size_t lls = (size_t)kMaxScreenGrid + (size_t)K + (size_t)dense_ll_parts();
    const size_t nll = (size_t)nslabs * lls + kListGrid;
    const bool dense_on = W.dp_parts > 0;
    double* dpart = lpart + (size_t)W.lp_parts * K * stat_width(D, cov);
    GMM_TRY(cudaMemsetAsync(llp, 0, sizeof(double) * nll, s));
    for (int64_t si = 0; si < nslabs; ++si) {
      const int64_t r0 = si * slab_rows;
      const int64_t sn = (rows - r0) < slab_rows ? (rows - r0) : slab_rows;
      const void* Xs = (const char*)X + (size_t)r0 * D * esize(xdtype);
      float* ls = lse + r0;
      const int acc = accumulate || r0 > 0;
      double* llp_s = llp + (size_t)si * lls;
      uint32_t* dmask = dense_on ? at<uint32_t>(ws, W.off_dmask) : nullptr;
      uint32_t* cmask = dense_on ? at<uint32_t>(ws, W.off_cmask) : nullptr;
      {
        GMM_PROF("tc_screen_kernel");
        GMM_TRY(tc_screen(Xs, xdtype, sn, D, K, cov, prep, 0, ls, want_lse ? 1 : 0, llp_s, 0,
                          nullptr, nullptr, fbm + (size_t)(r0 / 128) * 4, cmask, dmask, recs,
                          tcnt, rec_cap, st, s));
      }
      GMM_TRY(sparse_stats(Xs, xdtype, sn, D, K, prep, cov, ls, tcnt, recs, rec_cap,
                           at<char>(ws, W.off_sws), part, acc, llp_s + kMaxScreenGrid, st, s));
      if (dense_on) {
        uint32_t* drows = at<uint32_t>(ws, W.off_drows);
        {
          GMM_PROFN("fb_compact_kernel", 2);
          GMM_TRY(fb_compact(dmask, sn, drows, &st->dense_count, at<uint32_t>(ws, W.off_fbseg), s));
        }
        GMM_TRY(dense_rows(Xs, xdtype, D, K, cov, prep, drows, &st->dense_count, cmask,
                           at<float2>(ws, W.off_dpart), ls, llp_s + kMaxScreenGrid + K, dpart, acc,
                           st, s));
      }
    }
    {
      GMM_PROFN("fb_compact_kernel", 2);
      GMM_TRY(fb_compact(fbm, rows, fb, &st->fb_count, at<uint32_t>(ws, W.off_fbseg), s));
    }
    {
      GMM_PROF("lse_rows_kernel");
      GMM_TRY(simt_lse_rows(X, xdtype, rows, D, K, cov, prep, lse, llp + (size_t)nslabs * lls, 0,
                            nullptr, nullptr, st, fb, &st->fb_count, kListGrid, s));
    }
    {
      GMM_PROF("stats_rows_kernel");
      GMM_TRY(simt_stats_rows(X, xdtype, rows, D, K, cov, prep, lse, W.lp_parts, lpart,
                              accumulate, fb, &st->fb_count, s));
    }
    {
      GMM_PROF("ll_finalize_kernel");
      GMM_TRY(launch_ll_finalize(llp, (int64_t)nll, at<double>(ws, W.off_ll), accumulate, s));
    }
    return GMM_OK;
  }
  {
    GMM_PROF("lse_kernel");
    GMM_TRY(simt_lse(X, xdtype, rows, D, K, cov, prep, lse, llp, 0, nullptr, nullptr, st, s));
  }
  {
    GMM_PROF("ll_finalize_kernel");
    GMM_TRY(launch_ll_finalize(llp, (rows + kLseRows - 1) / kLseRows, at<double>(ws, W.off_ll),
                               accumulate, s));
  }
  {
    GMM_PROF("stats_kernel");
    GMM_TRY(simt_stats(X, xdtype, rows, D, K, cov, prep, lse, W.parts,
                       at<double>(ws, W.off_part), accumulate, s));
  }
  return GMM_OK;
}

// Partials the M-step merges for the path taken.
int mstep_parts(const WsLayout& W, bool tc) {
  return tc ? W.sp_parts + W.lp_parts + W.dp_parts : W.parts;
}

// Library-owned copy stream and events of the host path (one set per device).
struct HostPathRes {
  cudaStream_t copy = nullptr;
  cudaEvent_t copied[2] = {nullptr, nullptr};
  cudaEvent_t consumed[2] = {nullptr, nullptr};
};
std::mutex g_res_mu;
HostPathRes g_res[64];

gmm_status host_res(HostPathRes** out) {
  int dev = 0;
  GMM_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return GMM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_res_mu);
  HostPathRes& r = g_res[dev];
  if (!r.copy) {
    GMM_TRY(cudaStreamCreateWithFlags(&r.copy, cudaStreamNonBlocking));
    for (int i = 0; i < 2; ++i) {
      GMM_TRY(cudaEventCreateWithFlags(&r.copied[i], cudaEventDisableTiming));
      GMM_TRY(cudaEventCreateWithFlags(&r.consumed[i], cudaEventDisableTiming));
    }
  }
  *out = &r;
  return GMM_OK;
}

}  // namespace

ProfScope::ProfScope(const char* n, cudaStream_t st, int nkernels)
    : name(n), s(st), kernels(nkernels) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof_on) { a = prof_event(); cudaEventRecord(a, s); }
}

ProfScope::~ProfScope() {
  if (!a) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  cudaEvent_t b = prof_event();
  cudaEventRecord(b, s);
  g_prof_pending.push_back({name, a, b, kernels});
}

// The statistics partition count the entry points above use, for other
// translation units that launch the same kernels.
int stat_parts_for(int64_t N, int D, int K, int cov) { return stat_parts(N, D, K, cov); }

}  // namespace gmm

using namespace gmm;

extern "C" {

gmm_opts gmm_default_opts(void) {
  gmm_opts o;
  o.ridge_rel = 0.0f;
  o.var_floor = 0.0f;
  o.min_s0 = 0.5f;
  o.flags = 0;
  return o;
}

const char* gmm_status_string(gmm_status s) {
  switch (s) {
    case GMM_OK: return "GMM_OK";
    case GMM_ERR_INVALID_ARG: return "GMM_ERR_INVALID_ARG";
    case GMM_ERR_UNSUPPORTED: return "GMM_ERR_UNSUPPORTED";
    case GMM_ERR_NOT_PD: return "GMM_ERR_NOT_PD";
    case GMM_ERR_NONFINITE: return "GMM_ERR_NONFINITE";
    case GMM_ERR_WORKSPACE: return "GMM_ERR_WORKSPACE";
    case GMM_ERR_TIMEOUT: return "GMM_ERR_TIMEOUT";
    case GMM_ERR_CUDA: return "GMM_ERR_CUDA";
  }
  return "unknown gmm_status";
}

size_t gmm_prepared_bytes(int D, int K, gmm_cov_type cov) {
  if (!valid_d(D) || K < 1 || K > kMaxK || cov < GMM_COV_FULL || cov > GMM_COV_ISO) return 0;
  return PreparedLayout::make(D, K, cov).bytes;
}

size_t gmm_workspace_bytes(int64_t N, int D, int K, gmm_cov_type cov, gmm_dtype xdtype) {
  if (N < 1 || !valid_d(D) || K < 1 || K > kMaxK || cov < GMM_COV_FULL || cov > GMM_COV_ISO ||
      xdtype < GMM_F32 || xdtype > GMM_BF16)
    return 0;
  return ws_layout(N, N, D, K, cov, 0).bytes;
}

size_t gmm_workspace_bytes_host(int64_t N, int D, int K, gmm_cov_type cov, gmm_dtype xdtype,
                                int64_t chunk_rows) {
  if (chunk_rows < 1 || gmm_workspace_bytes(N, D, K, cov, xdtype) == 0) return 0;
  int64_t rows = chunk_rows < N ? chunk_rows : N;
  size_t stage = 2 * align_up((size_t)rows * D * esize(xdtype));
  return ws_layout(N, rows, D, K, cov, stage).bytes;
}

gmm_status gmm_prepare(const gmm_params* p, int D, int K, gmm_cov_type cov, const gmm_opts* opts,
                       void* prepared, int32_t* flags_dev, void* stream) {
  if (!p || !p->pi || !p->mu || !p->cov || !prepared || K < 1 || K > kMaxK) return GMM_ERR_INVALID_ARG;
  if (cov < GMM_COV_FULL || cov > GMM_COV_ISO) return GMM_ERR_INVALID_ARG;
  if (!valid_d(D)) return D > 0 ? GMM_ERR_UNSUPPORTED : GMM_ERR_INVALID_ARG;
  gmm_opts o = opts ? *opts : gmm_default_opts();
  cudaStream_t s = (cudaStream_t)stream;
  {
    GMM_PROFN("prepare_kernel", 1 + (tc_eligible(D, cov) ? 3 : 0));
    GMM_TRY(launch_prepare(p, D, K, cov, o.ridge_rel, prepared, nullptr, s));
  }
  if (flags_dev) {
    PreparedLayout L = PreparedLayout::make(D, K, cov);
    GMM_TRY(cudaMemcpyAsync(flags_dev, at<char>(prepared, L.off_flags), sizeof(int32_t) * K,
                            cudaMemcpyDeviceToDevice, s));
  }
  return GMM_OK;
}

gmm_status gmm_em_step(const void* X, gmm_dtype xdtype, int64_t N, int D, int K,
                       gmm_params* params, gmm_cov_type cov, const gmm_opts* opts, void* ws,
                       size_t ws_bytes, double* loglik_dev, float* lse_dev, int32_t* flags_dev,
                       void* stream) {
  gmm_status c = check_common(X, xdtype, N, D, K, cov);
  if (c != GMM_OK) return c;
  if (!params || !params->pi || !params->mu || !params->cov || !ws || !loglik_dev)
    return GMM_ERR_INVALID_ARG;
  if (((uintptr_t)X & 15) || ((uintptr_t)ws & 255)) return GMM_ERR_INVALID_ARG;
  WsLayout W = ws_layout(N, N, D, K, cov, 0);
  if (ws_bytes < W.bytes) return GMM_ERR_WORKSPACE;
  gmm_opts o = opts ? *opts : gmm_default_opts();
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus* st = at<DeviceStatus>(ws, W.off_status);
  void* prep = at<char>(ws, W.off_prep);
  PreparedLayout PL = PreparedLayout::make(D, K, cov);
  GMM_TRY(cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s));
  {
    GMM_PROFN("prepare_kernel", 1 + (tc_eligible(D, cov) ? 3 : 0));
    GMM_TRY(launch_prepare(params, D, K, cov, o.ridge_rel, prep, st, s));
  }
  float* lse = lse_dev ? lse_dev : at<float>(ws, W.off_lse);
  gmm_status r = estep_rows(X, xdtype, N, D, K, cov, W, ws, lse, lse_dev != nullptr, 0,
                            use_tc(D, K, cov, o), use_fc(D, K, cov, o), s);
  if (r != GMM_OK) return r;
  {
    GMM_PROF("mstep_kernel");
    GMM_TRY(launch_mstep(at<double>(ws, W.off_part), mstep_parts(W, use_tc(D, K, cov, o)), N, D, K, cov,
                         at<float>(prep, PL.off_mu), at<int32_t>(prep, PL.off_flags), o.var_floor,
                         o.min_s0, params, flags_dev ? flags_dev : at<int32_t>(ws, W.off_flags),
                         s));
  }
  GMM_TRY(cudaMemcpyAsync(loglik_dev, at<double>(ws, W.off_ll), sizeof(double),
                          cudaMemcpyDeviceToDevice, s));
  return GMM_OK;
}

gmm_status gmm_em_step_host(const void* X_host, gmm_dtype xdtype, int64_t N, int D, int K,
                            gmm_params* params, gmm_cov_type cov, const gmm_opts* opts, void* ws,
                            size_t ws_bytes, int64_t chunk_rows, double* loglik_dev,
                            double* loglik_host, int32_t* flags_dev, void* stream) {
  gmm_status c = check_common(X_host, xdtype, N, D, K, cov);
  if (c != GMM_OK) return c;
  if (!params || !params->pi || !params->mu || !params->cov || !ws || !loglik_dev ||
      chunk_rows < 1 || ((uintptr_t)ws & 255))
    return GMM_ERR_INVALID_ARG;
  const int64_t rows = chunk_rows < N ? chunk_rows : N;
  const size_t stage_one = align_up((size_t)rows * D * esize(xdtype));
  WsLayout W = ws_layout(N, rows, D, K, cov, 2 * stage_one);
  if (ws_bytes < W.bytes) return GMM_ERR_WORKSPACE;
  HostPathRes* res = nullptr;
  gmm_status rr = host_res(&res);
  if (rr != GMM_OK) return rr;
  gmm_opts o = opts ? *opts : gmm_default_opts();
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus* st = at<DeviceStatus>(ws, W.off_status);
  void* prep = at<char>(ws, W.off_prep);
  PreparedLayout PL = PreparedLayout::make(D, K, cov);
  char* stage[2] = {at<char>(ws, W.off_stage), at<char>(ws, W.off_stage + stage_one)};
  GMM_TRY(cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s));
  {
    GMM_PROFN("prepare_kernel", 1 + (tc_eligible(D, cov) ? 3 : 0));
    GMM_TRY(launch_prepare(params, D, K, cov, o.ridge_rel, prep, st, s));
  }
  // The copy stream may start only after earlier work on `s` that used the
  // staging buffers is done.
  GMM_TRY(cudaEventRecord(res->consumed[0], s));
  GMM_TRY(cudaEventRecord(res->consumed[1], s));
  const int64_t nchunks = (N + rows - 1) / rows;
  const size_t esz = esize(xdtype);
  for (int64_t ci = 0; ci < nchunks; ++ci) {
    const int b = (int)(ci & 1);
    const int64_t r0 = ci * rows;
    const int64_t rn = (N - r0) < rows ? (N - r0) : rows;
    GMM_TRY(cudaStreamWaitEvent(res->copy, res->consumed[b], 0));
    GMM_TRY(cudaMemcpyAsync(stage[b], (const char*)X_host + (size_t)r0 * D * esz,
                            (size_t)rn * D * esz, cudaMemcpyHostToDevice, res->copy));
    GMM_TRY(cudaEventRecord(res->copied[b], res->copy));
    GMM_TRY(cudaStreamWaitEvent(s, res->copied[b], 0));
    gmm_status r = estep_rows(stage[b], xdtype, rn, D, K, cov, W, ws, at<float>(ws, W.off_lse),
                              false, ci > 0, use_tc(D, K, cov, o), use_fc(D, K, cov, o), s);
    if (r != GMM_OK) return r;
    GMM_TRY(cudaEventRecord(res->consumed[b], s));
  }
  {
    GMM_PROF("mstep_kernel");
    GMM_TRY(launch_mstep(at<double>(ws, W.off_part), mstep_parts(W, use_tc(D, K, cov, o)), N, D, K, cov,
                         at<float>(prep, PL.off_mu), at<int32_t>(prep, PL.off_flags), o.var_floor,
                         o.min_s0, params, flags_dev ? flags_dev : at<int32_t>(ws, W.off_flags),
                         s));
  }
  GMM_TRY(cudaMemcpyAsync(loglik_dev, at<double>(ws, W.off_ll), sizeof(double),
                          cudaMemcpyDeviceToDevice, s));
  if (loglik_host)
    GMM_TRY(cudaMemcpyAsync(loglik_host, at<double>(ws, W.off_ll), sizeof(double),
                            cudaMemcpyDeviceToHost, s));
  GMM_TRY(cudaStreamSynchronize(s));
  return GMM_OK;
}

gmm_status gmm_assign_topm(const void* X, gmm_dtype xdtype, int64_t N, int D, int K,
                           const void* prepared, gmm_cov_type cov, int m, int32_t* ids,
                           float* gamma, float* lse, void* ws, size_t ws_bytes, void* stream) {
  gmm_status c = check_common(X, xdtype, N, D, K, cov);
  if (c != GMM_OK) return c;
  if (!prepared || !ids || !gamma || !ws || m < 1 || m > 8 || m > K) return GMM_ERR_INVALID_ARG;
  if (((uintptr_t)X & 15) || ((uintptr_t)ws & 255)) return GMM_ERR_INVALID_ARG;
  const WsLayout W = ws_layout(N, N, D, K, cov, 0);
  const bool tc = tc_eligible(D, cov);
  if (ws_bytes < (tc ? W.bytes : sizeof(DeviceStatus))) return GMM_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus* st = static_cast<DeviceStatus*>(ws);
  GMM_TRY(cudaMemsetAsync(st, 0, sizeof(DeviceStatus), s));
  if (tc) {
    // slabs of rows on the tensor cores, each marking the rows it hands over
    // in the bitmap of all rows; then one CUDA-core pass over those rows
    uint32_t* fb = at<uint32_t>(ws, W.off_fb);
    uint32_t* fbm = at<uint32_t>(ws, W.off_fbm);
    const int64_t slab_rows = slab_rows_for(K);
    for (int64_t r0 = 0; r0 < N; r0 += slab_rows) {
      const int64_t sn = (N - r0) < slab_rows ? (N - r0) : slab_rows;
      const void* Xs = (const char*)X + (size_t)r0 * D * esize(xdtype);
      float* ls = lse ? lse + r0 : nullptr;
      int32_t* is = ids + (size_t)r0 * m;
      float* gs = gamma + (size_t)r0 * m;
      GMM_PROF("tc_screen_kernel");
      GMM_TRY(tc_screen(Xs, xdtype, sn, D, K, cov, prepared, 1, ls, 0, nullptr, m, is, gs,
                        fbm + (size_t)(r0 / 128) * 4, nullptr, nullptr, nullptr, nullptr, 0, st, s));
    }
    {
      GMM_PROFN("fb_compact_kernel", 2);
      GMM_TRY(fb_compact(fbm, N, fb, &st->fb_count, at<uint32_t>(ws, W.off_fbseg), s));
    }
    GMM_PROF("lse_rows_kernel");
    GMM_TRY(simt_lse_rows(X, xdtype, N, D, K, cov, prepared, lse, nullptr, m, ids, gamma, st, fb,
                          &st->fb_count, kListGrid, s));
    return GMM_OK;
  }
  GMM_PROF("lse_topm_kernel");
  GMM_TRY(simt_lse(X, xdtype, N, D, K, cov, prepared, lse, nullptr, m, ids, gamma, st, s));
  return GMM_OK;
}

void gmm_profile_enable(int on) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = on != 0;
}

int gmm_profile_read(const char** names, double* ms_total, long* launches, int max_kernels) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  for (ProfRec& r : g_prof_pending) {
    float ms = 0.f;
    cudaEventSynchronize(r.b);
    cudaEventElapsedTime(&ms, r.a, r.b);
    size_t i = 0;
    for (; i < g_prof_sum.size(); ++i)
      if (strcmp(g_prof_sum[i].name, r.name) == 0) break;
    if (i == g_prof_sum.size()) g_prof_sum.push_back({r.name, 0.0, 0});
    g_prof_sum[i].ms += ms;
    g_prof_sum[i].launches += r.kernels;
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_pending.clear();
  int n = (int)g_prof_sum.size();
  for (int i = 0; i < n && i < max_kernels; ++i) {
    if (names) names[i] = g_prof_sum[i].name;
    if (ms_total) ms_total[i] = g_prof_sum[i].ms;
    if (launches) launches[i] = g_prof_sum[i].launches;
  }
  return n;
}

void gmm_profile_reset(void) {
  const char* dummy[1];
  gmm_profile_read(dummy, nullptr, nullptr, 0);
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_sum.clear();
}

gmm_status gmm_last_device_status(void* ws, void* stream) {
  if (!ws) return GMM_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  DeviceStatus h;
  GMM_TRY(cudaStreamSynchronize(s));
  GMM_TRY(cudaMemcpy(&h, ws, sizeof(DeviceStatus), cudaMemcpyDeviceToHost));
  return (gmm_status)h.code;
}

}  // extern "C"
