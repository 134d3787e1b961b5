// gmm_internal.cuh - layouts and helpers shared by the libgmm kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gmm.h"

namespace gmm {

constexpr size_t kAlign = 256;
__host__ __device__ inline size_t align_up(size_t v, size_t a = kAlign) {
  return (v + a - 1) / a * a;
}

// Status-word bits (first failing condition recorded as a gmm_status value;
// later conditions only OR into the detail word).
struct DeviceStatus {
  int32_t code;     // gmm_status of the first device-side failure (0 = none)
  int32_t detail;   // OR of (1 << gmm_status) for every failure seen
  int32_t pad[62];
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

// Prepared-parameter block written by gmm_prepare.
struct PreparedLayout {
  int D, K, cov;
  size_t off_flags;  // int32 [K]
  size_t off_c;      // float [K]    log pi - log|S|/2 - (D/2) log 2pi  (-inf: excluded)
  size_t off_mu;     // float [K*D]  means
  size_t off_prec;   // float [K*P]  diag: 1/var; iso: 1/var; full: W = L^-1 (lower)
  size_t off_tc;     // tensor-core operand blocks (see tc kernels); 0 bytes if none
  size_t tc_bytes;
  size_t bytes;

  __host__ __device__ static PreparedLayout make(int D, int K, int cov) {
    PreparedLayout L;
    L.D = D; L.K = K; L.cov = cov;
    size_t o = 0;
    L.off_flags = o; o = align_up(o + sizeof(int32_t) * K);
    L.off_c = o;     o = align_up(o + sizeof(float) * K);
    L.off_mu = o;    o = align_up(o + sizeof(float) * (size_t)K * D);
    L.off_prec = o;  o = align_up(o + sizeof(float) * (size_t)K * prec_width(D, cov));
    L.off_tc = o;
    L.tc_bytes = 0;
    o = align_up(o + L.tc_bytes);
    L.bytes = o;
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

__device__ __forceinline__ double warp_sum(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace gmm
