// gmm_internal.cuh - layouts and helpers shared by the libgmm kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gmm.h"

namespace gmm {

constexpr size_t kAlign = 256;
// Rows per block of the CUDA-core log-sum-exp kernel (one log-likelihood
// partial each) and the largest component count the entry points accept;
// every translation unit that sizes scratch for those kernels uses these.
constexpr int kLseRows = 128;
constexpr int kMaxK = 1 << 16;
__host__ __device__ inline size_t align_up(size_t v, size_t a = kAlign) {
  return (v + a - 1) / a * a;
}

// Profiler scope: when profiling is on (gmm_profile_enable), the launches in
// its lifetime (`kernels` of them) are bracketed by two CUDA events on `s`
// and summed under `name` (defined in gmm_api.cu).
struct ProfScope {
  const char* name;
  cudaStream_t s;
  int kernels;
  cudaEvent_t a = nullptr;
  ProfScope(const char* n, cudaStream_t st, int nkernels = 1);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;
};

// Status-word bits (first failing condition recorded as a gmm_status value;
// later conditions only OR into the detail word).
struct DeviceStatus {
  int32_t code;        // gmm_status of the first device-side failure (0 = none)
  int32_t detail;      // OR of (1 << gmm_status) for every failure seen
  uint32_t fb_count;   // rows the tensor-core kernel handed to the CUDA-core path
  uint32_t dense_count;  // rows whose candidates went to the dense-row kernels (last slab)
  unsigned long long cand_pairs;  // (point, candidate) pairs the dense-row or full-covariance
                                  // log-sum-exp kernels evaluated in this call
  int32_t pad[58];
};

__device__ inline void raise_status(DeviceStatus* st, int code) {
  atomicCAS(&st->code, 0, code);
  atomicOr(&st->detail, 1 << code);
}

// Number of values per component of the accumulated statistics:
//   diag/iso: [s0 | s1 (D) | s2 diagonal (D)]
//   full:     [s0 | s1 (D) | s2 lower triangle (D(D+1)/2)]
__host__ __device__ inline int stat_width(int D, int cov) {
  return cov == GMM_COV_FULL ? 1 + D + D * (D + 1) / 2 : 1 + 2 * D;
}

// Entries of the per-component precision block of the prepared buffer.
__host__ __device__ inline int prec_width(int D, int cov) {
  return cov == GMM_COV_FULL ? D * D : (cov == GMM_COV_DIAG ? D : 1);
}

// Tensor-core screening applies to diagonal / isotropic covariance with
// D = 64 or 128: the log-density is screened as [x, x^2] . [b1, b2] with
// b1 = mu / var, b2 = -1 / (2 var) on fp16 tensor cores.
constexpr int kTcChunk = 128;  // components per screening chunk (MMA N)
// Per-chunk trailer of the screening operands: scale [128], |(b1, b2)|_2
// [128], then the bias with its absolute and relative fp32 margin
// (delta_k = 1e-3 + 1e-6 |bias_k|) taken off [128] and added on [128].
constexpr int kTcTrail = 4 * kTcChunk;
__host__ __device__ inline bool tc_eligible(int D, int cov) {
  return (cov == GMM_COV_DIAG || cov == GMM_COV_ISO) && (D == 64 || D == 128);
}

// Folded screening operands (up to two chunks, the parameters resident in
// shared memory): every component of a chunk shares one power-of-two scale
// S, and one more K = 16 step of the contraction adds the bias and the
// rigorous error margin, so the accumulator is directly the upper bound
// hi_k / S.  The extra step's operands:
//   A row n: [2^10, 1, 2^-10, ru(rn_n 2^-4), 1, 0 ...]
//   B row k: [b1, b2, b3, ru(u_k 2^4 / S), ru(d_k / S), 0 ...]
// with bias_k / S = 2^10 b1 + b2 + 2^-10 b3 (fp16 parts), rn_n >= |[x, x^2]|
// the row norm, u_k = kappa |(b1, b2)_k| + 2^-20 S the margin per unit of
// row norm and d_k the absolute margin.  Trailer of a folded chunk:
// u_k [128], d_k [128], then S, 1/S, max u_k, max d_k.
constexpr int kTcFoldChunks = 2;
constexpr int kTcExtraK = 16;
constexpr int kTcExtraBytes = kTcChunk * kTcExtraK * 2;  // one chunk's extra B rows
enum { kFoldS = 2 * kTcChunk, kFoldInvS, kFoldUMax, kFoldDMax };
__host__ __device__ inline bool tc_fold(int chunks) { return chunks <= kTcFoldChunks; }

// Records of the tensor-core E-step: uint2 {key, bits of the exact fp32 log
// joint}, key = flag | (component << 7) | row in the 128-point tile.  The
// flag marks a point's only candidate (gamma 1, its log joint not evaluated).
constexpr uint32_t kRecSingle = 1u << 31;
constexpr uint32_t kRecKMask = 0xffffffu;  // component = (key >> 7) & kRecKMask

// Full covariance with few components: the tensor-core screen of
// z = W_k (x - mu_k) (fc_screen.cu) takes D = 32 or 64 and K D <= 1024.  Its
// operands, written by gmm_prepare: the B image [K D rows][128 bytes] of
// fp16(W_k / s_k) as 128-byte swizzled K-major rows (the contraction
// dimension padded with zeros to 64), and fp32 [s_k (32) | bias_k (32) |
// ex_k (32) | em_k (32) | b_k = W_k mu_k (K D)].
constexpr int kFcMaxK = 32;
__host__ __device__ inline bool fc_tc_shape(int D, int K, int cov) {
  return cov == GMM_COV_FULL && (D == 32 || D == 64) && K >= 1 && K <= kFcMaxK && K * D <= 1024;
}

// Prepared-parameter block written by gmm_prepare.
struct PreparedLayout {
  int D, K, cov;
  size_t off_flags;  // int32 [K]
  size_t off_c;      // float [K]    log pi - log|S|/2 - (D/2) log 2pi  (-inf: excluded)
  size_t off_mu;     // float [K*D]  means
  size_t off_prec;   // float [K*P]  diag: 1/var; iso: 1/var; full: W = L^-1 (lower)
  // tensor-core screening operands (tc_eligible shapes only):
  int tc_chunks;     // ceil(K / 128)
  size_t off_tcB;    // fp16 [chunks][2D/64][128 rows][64]: (b1, b2)/scale as 128-byte
                     // swizzled K-major tiles, one contiguous image per chunk; folded:
                     // followed in each image by the chunk's unswizzled K = 16 extra rows
  size_t tcB_chunk_bytes;
  size_t off_tcT;    // float [chunks][kTcTrail]: scale (power of 2) [128], |(b1,b2)|_2 [128],
                     // bias - delta [128], bias + delta [128] (the scale is the chunk's, common to its
                     // components); folded: see tc_fold
  size_t tc_bytes;
  size_t off_fcB;    // full covariance (fc_tc_shape): the screen's B image
  size_t off_fcT;    // ... and its fp32 constants
  size_t bytes;

  __host__ __device__ static PreparedLayout make(int D, int K, int cov) {
    PreparedLayout L;
    L.D = D; L.K = K; L.cov = cov;
    size_t o = 0;
    L.off_flags = o; o = align_up(o + sizeof(int32_t) * K);
    L.off_c = o;     o = align_up(o + sizeof(float) * K);
    L.off_mu = o;    o = align_up(o + sizeof(float) * (size_t)K * D);
    L.off_prec = o;  o = align_up(o + sizeof(float) * (size_t)K * prec_width(D, cov));
    L.tc_chunks = 0;
    L.off_tcB = L.off_tcT = o;
    L.tcB_chunk_bytes = 0;
    L.tc_bytes = 0;
    if (tc_eligible(D, cov)) {
      L.tc_chunks = (K + kTcChunk - 1) / kTcChunk;
      o = align_up(o, 1024);
      L.off_tcB = o;
      L.tcB_chunk_bytes = (size_t)kTcChunk * 2 * D * 2 + (tc_fold(L.tc_chunks) ? kTcExtraBytes : 0);
      o = align_up(o + L.tcB_chunk_bytes * L.tc_chunks);
      L.off_tcT = o;
      o = align_up(o + sizeof(float) * kTcTrail * L.tc_chunks);
      L.tc_bytes = o - L.off_tcB;
    }
    L.off_fcB = L.off_fcT = o;
    if (fc_tc_shape(D, K, cov)) {
      o = align_up(o, 1024);
      L.off_fcB = o;
      o = align_up(o + (size_t)K * D * 128);
      L.off_fcT = o;
      o = align_up(o + sizeof(float) * (4 * kFcMaxK + (size_t)K * D));
    }
    L.bytes = align_up(o);
    return L;
  }
};

template <typename T>
__host__ __device__ inline T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}
template <typename T>
__host__ __device__ inline const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const char*>(base) + off);
}

// Load one stored coordinate as float.
template <int XT>
__device__ __forceinline__ float load_x(const void* X, size_t i) {
  if constexpr (XT == GMM_F32) return __ldg(static_cast<const float*>(X) + i);
  else if constexpr (XT == GMM_F16) return __half2float(static_cast<const __half*>(X)[i]);
  else return __bfloat162float(static_cast<const __nv_bfloat16*>(X)[i]);
}

// Pairs of fp32 operations issued as one packed instruction (each half an
// IEEE fp32 operation rounded to nearest, as the scalar forms).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ double warp_sum(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace gmm
