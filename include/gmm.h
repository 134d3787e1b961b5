/*
 * gmm.h - C ABI of libgmm: one fused EM iteration of a Gaussian mixture
 * model, and top-m soft assignment, on one GB300 (sm_103a).
 *
 * Sources (page titles as given):
 *  [LP]  design notes for a low-precision GMM operator (hotelren.com news 5857197)
 *  [FG]  "Flash-GMM: a memory-efficient kernel for scalable soft clustering"
 *        (summary at ai-feeds.com paper 2606.10896)
 *
 * Conventions shared by every entry point
 *  - All array arguments are DEVICE pointers unless named *_host, owned by the
 *    caller, and must stay valid until the work queued on `stream` is done.
 *    The library allocates no device memory: scratch space is the caller's
 *    workspace `ws` (size from gmm_workspace_bytes).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every entry point is asynchronous on that stream unless stated.
 *  - X is row-major N x D (point n at X + n*D elements), element type `xdtype`,
 *    16-byte aligned.  D must be 16, 32, 64 or 128; K >= 1; N >= 1.
 *  - Parameters are fp32: pi[K]; mu[K*D] row-major; cov is K*D*D row-major
 *    symmetric (GMM_COV_FULL), K*D variances (GMM_COV_DIAG) or K variances
 *    (GMM_COV_ISO).
 *  - Argument errors are reported synchronously by the return value; nothing
 *    is queued then.  Conditions found on the device (a covariance that is
 *    not positive definite even after the ridge retry, a non-finite
 *    log-likelihood) set bits of a status word inside `ws`, read back by
 *    gmm_last_device_status.
 *  - The N x K responsibility matrix is never stored: the workspace is
 *    O(N + K*D*D) bytes ([FG] "Core insight": O(NK) memory becomes O(N+K)).
 */
#ifndef GMM_H
#define GMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GMM_COV_FULL = 0, GMM_COV_DIAG = 1, GMM_COV_ISO = 2 } gmm_cov_type;
typedef enum { GMM_F32 = 0, GMM_F16 = 1, GMM_BF16 = 2 } gmm_dtype;

typedef enum {
  GMM_OK = 0,
  GMM_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned X */
  GMM_ERR_UNSUPPORTED = 2,  /* valid but not built (e.g. D not in {16,32,64,128}) */
  GMM_ERR_NOT_PD = 3,       /* device: a covariance failed the ridge retry */
  GMM_ERR_NONFINITE = 4,    /* device: a log-likelihood term is not finite */
  GMM_ERR_WORKSPACE = 5,    /* ws_bytes smaller than gmm_workspace_bytes */
  GMM_ERR_TIMEOUT = 6,      /* device: a bounded wait gave up */
  GMM_ERR_CUDA = 7          /* a CUDA launch or runtime call failed */
} gmm_status;

/* Per-component flag bits (flags_dev outputs). */
enum {
  GMM_FLAG_RIDGE = 1,   /* the ridge retry was needed ([LP] sec. 3.3, 4.1) */
  GMM_FLAG_NOT_PD = 2,  /* still not positive definite; component excluded */
  GMM_FLAG_FLOOR = 4,   /* a variance was raised to var_floor */
  GMM_FLAG_EMPTY = 8    /* s0 < min_s0: mean and covariance kept */
};

/* gmm_opts.flags bits. */
enum { GMM_OPT_CUDA_CORES = 1 };

/* Model parameters, fp32 device arrays (layout above). */
typedef struct {
  float* pi;
  float* mu;
  float* cov;
} gmm_params;

/* Options.  ridge_rel: ridge_rel * tr(Sigma)/D is added to every covariance
 * before factorisation (default 0; [LP] sec. 4.1 gives 1e-3 as the rule and
 * 5e-4 as a tried value).  If the factorisation still fails, 1e-3*tr/D more
 * is added and it is retried once ([LP] sec. 3.3: flag and correct in the
 * preprocessing step, never branch in the distance kernel).
 * var_floor: lower bound applied to updated variances (and the diagonal of a
 * full covariance).  min_s0: a component whose responsibility sum s0 is
 * below it keeps its mean and covariance (its weight becomes s0/N).
 * flags: GMM_OPT_CUDA_CORES (bit 0) computes every log-density on CUDA cores
 * even where a tensor-core screening path applies (diagonal / isotropic
 * covariance with D = 64 or 128; full covariance with D = 32 or 64, K <= 32,
 * K D <= 1024, fp16 X); other bits reserved, 0. */
typedef struct {
  float ridge_rel;
  float var_floor;
  float min_s0;
  int flags;
} gmm_opts;

/* Defaults: ridge_rel 0, var_floor 0, min_s0 0.5, flags 0.  (Below s0 = 1/2
 * every point's responsibility for the component is below 1/2 - each point
 * belongs more to the rest of the mixture - so the updated mean would be an
 * average of other components' tail points.) */
gmm_opts gmm_default_opts(void);

/* Human-readable name of a status code (static string). */
const char* gmm_status_string(gmm_status s);

/* Workspace bytes gmm_em_step / gmm_assign_topm need for these sizes.
 * Returns 0 for unsupported arguments. */
size_t gmm_workspace_bytes(int64_t N, int D, int K, gmm_cov_type cov, gmm_dtype xdtype);

/* Bytes of the prepared-parameter block gmm_prepare writes. */
size_t gmm_prepared_bytes(int D, int K, gmm_cov_type cov);

/*
 * gmm_prepare - per-component preprocessing, once per EM iteration, all K
 * components in parallel ([LP] sec. 3.1, "Preprocess kernel": factorise the
 * covariance, compute log|Sigma| and the constant -(D/2) log 2 pi, store the
 * factor for the distance step).
 *   full: Sigma_k = L L^T (fp64 Cholesky, [LP] sec. 1.2), W_k = L^-1 stored
 *         fp32, log|Sigma_k| = 2 sum log L_ii;
 *   diag / iso: inverse variances 1/sigma^2 and sum log sigma^2.
 *   All: bias c_k = log pi_k - log|Sigma_k|/2 - (D/2) log 2 pi, the mean, and
 *   the fp16 operand blocks the tensor-core screens read (diagonal: the
 *   scaled [mu / var, -1 / (2 var)] chunks; full covariance with D = 32 / 64
 *   and K D <= 1024: fp16(W_k / s_k) and the screen's bound coefficients).
 * p:         input parameters (device, fp32).  A model stored in fp16 (the
 *            pages' IVF setting) is passed widened to fp32: every fp16 value
 *            is an fp32 value, so the preprocessing sees exactly the stored
 *            model.
 * prepared:  device buffer of gmm_prepared_bytes(D, K, cov) bytes, written.
 * flags_dev: K int32 flag words (GMM_FLAG_RIDGE / GMM_FLAG_NOT_PD), written;
 *            may be NULL.
 * A component that is not positive definite after the retry gets bias -inf
 * (no responsibility) and sets GMM_ERR_NOT_PD in the status word of `ws`
 * when called through gmm_em_step.
 */
gmm_status gmm_prepare(const gmm_params* p, int D, int K, gmm_cov_type cov, const gmm_opts* opts,
                       void* prepared, int32_t* flags_dev, void* stream);

/*
 * gmm_em_step - one fused EM iteration ([FG] "Method: fused E-M step"):
 *   E: l_nk = log pi_k + log N(x_n | mu_k, Sigma_k); LSE_n = log sum_k exp(l_nk)
 *      taken in fp32 with the running maximum subtracted ([LP] sec. 3.2, 4.2);
 *      g_nk = exp(l_nk - LSE_n) ([LP] sec. 1.1) - never written to memory.
 *   statistics: s0_k = sum_n g_nk, the first moment about the input mean
 *      c_k = mu_k, and the second moment M2_k = sum_n g_nk (x_n - mu'_k)
 *      (x_n - mu'_k)^T about the updated mean (diagonal only for diag / iso)
 *      ([FG] Method: online s0, s1, s2), accumulated in fp32 per block of
 *      points and merged in a fixed order in fp64 with the pairwise update of
 *      Chan, Golub and LeVeque ([LP] sec. 3.1, "M-step kernel": block
 *      partials, then a global reduction).
 *   M: pi' = s0/N, mu' = c + s1/s0, Sigma' = M2/s0 (the same value as
 *      s2/s0 - mu' mu'^T without its cancellation; iso: mean of the
 *      diagonal), floored at var_floor; empty rule with min_s0.
 *   Where a tensor-core path applies (diagonal / isotropic covariance with
 *   D = 64 or 128: the contraction [x, x^2] . [mu / var, -1 / (2 var)]; full
 *   covariance with D = 32 or 64, K <= 32, K D <= 1024 and fp16 X: the
 *   product W_k x, W = L^-1 ([LP] sec. 1.2)), every pair is screened with a
 *   rigorous error bound and the pairs within 40 nats of the point's best
 *   log joint are evaluated exactly in fp32; LSE_n and the statistics use
 *   those, and every other pair carries less than 4.3e-18 of its point's
 *   responsibility.  Diagonal points with more candidates than the screen's
 *   lists hold are evaluated, with their candidate masks, by CUDA-core
 *   kernels that stage the parameters in shared memory; points with a
 *   non-finite coordinate take the CUDA-core path, which uses all K.  Full
 *   covariance outside those shapes (and bf16 / fp32 X, without the screen:
 *   every component a candidate) uses the same exact kernels or the
 *   CUDA-core path.
 * params:     in: the current parameters; out: updated in place (stream order).
 * loglik_dev: one double, written with sum_n LSE_n at the INPUT parameters.
 * lse_dev:    optional N floats, LSE_n at the input parameters (NULL: skipped).
 * flags_dev:  optional K int32 flag words (NULL: skipped).
 * ws:         workspace of at least gmm_workspace_bytes(N, D, K, cov, xdtype).
 */
gmm_status gmm_em_step(const void* X, gmm_dtype xdtype, int64_t N, int D, int K,
                       gmm_params* params, gmm_cov_type cov, const gmm_opts* opts, void* ws,
                       size_t ws_bytes, double* loglik_dev, float* lse_dev, int32_t* flags_dev,
                       void* stream);

/*
 * gmm_em_step_host - gmm_em_step with X in HOST memory: X_host is copied to
 * the device through the workspace in chunks, overlapped with the E-step of
 * the previous chunk, so the data set need not fit in device memory
 * ([FG]: data sets far larger than one GPU's memory).  X_host should be
 * page-locked for the copies to overlap.  params, loglik_dev, flags_dev are
 * device pointers as in gmm_em_step; loglik_host (optional) receives the
 * log-likelihood after the call completes.  This call synchronises `stream`
 * before returning.  ws must hold gmm_workspace_bytes_host(...) bytes.
 */
size_t gmm_workspace_bytes_host(int64_t N, int D, int K, gmm_cov_type cov, gmm_dtype xdtype,
                                int64_t chunk_rows);
gmm_status gmm_em_step_host(const void* X_host, gmm_dtype xdtype, int64_t N, int D, int K,
                            gmm_params* params, gmm_cov_type cov, const gmm_opts* opts, void* ws,
                            size_t ws_bytes, int64_t chunk_rows, double* loglik_dev,
                            double* loglik_host, int32_t* flags_dev, void* stream);

/*
 * gmm_assign_topm - top-m soft assignment for IVF multi-assignment ([FG]
 * "Core insight" and "Key findings": boundary vectors are assigned to several
 * high-responsibility clusters).  For each point: the m components with the
 * largest l_nk (ties to the lower k), sorted descending, and their full-K
 * responsibilities g_nk = exp(l_nk - LSE_n).
 * prepared: output of gmm_prepare for the same D, K, cov.
 * ids:      N*m int32 (device), gamma: N*m float (device), lse: N floats or NULL.
 * m:        1..8, m <= K.
 * ws:       gmm_workspace_bytes(N, D, K, cov, xdtype) bytes (status word and the
 *           list of points handed from the tensor-core to the CUDA-core path).
 */
gmm_status gmm_assign_topm(const void* X, gmm_dtype xdtype, int64_t N, int D, int K,
                           const void* prepared, gmm_cov_type cov, int m, int32_t* ids,
                           float* gamma, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * gmm_ivf_lists - inverted lists of an IVF index with soft multi-assignment,
 * from the output of gmm_assign_topm ([FG] "Core insight", second point, and
 * "Experiments / key findings": a vector near a cluster boundary is stored in
 * the lists of several high-responsibility clusters).  Entry t of point n
 * (component ids[n*m + t], responsibility gamma[n*m + t]) joins that
 * component's list when t == 0 (the point's best component; every point is
 * indexed at least once) or gamma >= gamma_min.  Entries with an id outside
 * [0, K) are skipped.  Within each list the points are in ascending order;
 * the lists are bit-for-bit the same on every run.
 * ids, gamma:  N*m (device), as gmm_assign_topm writes them.
 * offsets:     K+1 int64 (device, written): list k is entries
 *              offsets[k] .. offsets[k+1]-1; offsets[K] = entries in all.
 * list_pts:    point indices (int32, device, written), list_gamma: their
 *              gamma (device, written); room for N*m entries each.
 * ws:          gmm_ivf_lists_ws_bytes(N, m, K) bytes (about 4*K*N/8192).
 * N <= 2^31 - 1, 1 <= m <= 8, 1 <= K <= 65536; gamma_min not NaN.
 */
size_t gmm_ivf_lists_ws_bytes(int64_t N, int m, int K);
gmm_status gmm_ivf_lists(const int32_t* ids, const float* gamma, int64_t N, int m, int K,
                         float gamma_min, int64_t* offsets, int32_t* list_pts, float* list_gamma,
                         void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream` and returns the device status word of `ws`: the
 * first device-side failure of the most recent gmm_em_step, gmm_em_step_host
 * or gmm_assign_topm call on that workspace (each call resets the word), or
 * GMM_OK. */
gmm_status gmm_last_device_status(void* ws, void* stream);

/*
 * gmm_em_step_noalloc - gmm_em_step for callers that cannot allocate device
 * memory.  The source pages have no counterpart: this entry point exists for
 * callers that are handed only their input and output buffers - plugins
 * running inside another framework's memory budget, code that must not call
 * cudaMalloc after start-up - and so cannot provide the `ws` workspace that
 * gmm_em_step needs.
 *
 * It always takes the CUDA-core kernels (the path gmm_em_step takes with
 * GMM_OPT_CUDA_CORES), whatever the shape, and ignores opts->flags: its
 * results match gmm_em_step's within the parity tolerances of this library,
 * not bit for bit where gmm_em_step takes the tensor-core path, and it runs
 * at the CUDA-core path's speed (on 10M x 128 points with K = 256 about 170
 * times slower than gmm_em_step's tensor-core path).  X, params,
 * loglik_dev, lse_dev (N floats, required here) and flags_dev (optional) are
 * the caller's device buffers.  All other scratch lives in one 64 MiB array
 * built into the library's device image: every GPU that loads the library
 * holds it until the process exits, and nothing is allocated by this call.
 * The scratch needed is about N/16 + 8*P*K*F + 4*K*(D+2) + prepared-parameter
 * bytes (P statistics blocks, F = 1+2D, or 1+D+D(D+1)/2 for full
 * covariance); sizes that need more than 64 MiB are rejected with
 * GMM_ERR_WORKSPACE (and a message on stderr) before anything is queued.
 *
 * Every call looks up the array's device address in the current context
 * (cudaGetSymbolAddress).  Every call shares the one array, so calls that
 * overlap on the GPU (other streams, other host threads) race: serialise
 * them.  The call synchronises `stream` before it returns (it reads the
 * device status into host memory), so it cannot be used under stream
 * capture, and returns the first device-side condition of this call
 * (GMM_ERR_NOT_PD, GMM_ERR_NONFINITE) or GMM_OK.
 */
gmm_status gmm_em_step_noalloc(const void* X, gmm_dtype xdtype, int64_t N, int D, int K,
                               gmm_params* params, gmm_cov_type cov, const gmm_opts* opts,
                               double* loglik_dev, float* lse_dev, int32_t* flags_dev,
                               void* stream);

/*
 * Per-kernel timing ("launch / device / sync" breakdown of the ops-debug
 * page, sec. 4.2).  gmm_profile_enable(1): every kernel the library launches
 * is bracketed by two CUDA events recorded on its own stream (adds two event
 * records per launch; off by default).  gmm_profile_read synchronises the
 * recorded events and returns the number of distinct kernels seen so far;
 * for i < min(that, max_kernels) it fills names[i] (static strings),
 * ms_total[i] (summed device time) and launches[i].  gmm_profile_reset
 * clears the sums.  Host-thread safe; not meant for use during capture.
 */
void gmm_profile_enable(int on);
int gmm_profile_read(const char** names, double* ms_total, long* launches, int max_kernels);
void gmm_profile_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* GMM_H */
