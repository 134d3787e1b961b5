// tc_debug.cu - a minimal tcgen05 GEMM used only to check the tensor-core
// building blocks (operand layout and descriptors, TMEM allocation and
// loads, MMA completion through an mbarrier) against a host reference.
#include <stdint.h>

#include "gmm_internal.cuh"
#include "tc_ptx.cuh"

namespace gmm {
namespace {

// C[128][n] = A[128][kdim] * B[n][kdim]^T, fp16 in, fp32 out; kdim in
// {64, 128, 256}, or one of them + 16, the last 16 columns then held in the
// unswizzled K = 16 layout and contracted by one more MMA; n in {64, 128}.
// One CTA of 128 threads.
__global__ void __launch_bounds__(128) tc_gemm_check_kernel(const uint16_t* __restrict__ A,
                                                            const uint16_t* __restrict__ B,
                                                            float* __restrict__ C, int kdim,
                                                            int n, int32_t* status) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment of the operand tiles (128-byte swizzle atoms)
  unsigned char* base = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int kmain = kdim & ~63, ktail = kdim & 63;  // ktail: 0 or 16
  unsigned char* sA = base;                       // 128 x kmain fp16
  unsigned char* sB = base + 128 * kmain * 2;     // n x kmain fp16
  unsigned char* sAt = sB + n * kmain * 2;        // 128 x 16 fp16, unswizzled
  unsigned char* sBt = sAt + 128 * 16 * 2;        // n x 16 fp16, unswizzled
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 128);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  for (int i = tid; i < 128 * kdim; i += 128) {
    const int r = i / kdim, k = i % kdim;
    if (k < kmain) *(uint16_t*)(sA + tc::sw128_offset(r, k, 128)) = A[i];
    else *(uint16_t*)(sAt + tc::k16_offset(r, k - kmain)) = A[i];
  }
  for (int i = tid; i < n * kdim; i += 128) {
    const int r = i / kdim, k = i % kdim;
    if (k < kmain) *(uint16_t*)(sB + tc::sw128_offset(r, k, n)) = B[i];
    else *(uint16_t*)(sBt + tc::k16_offset(r, k - kmain)) = B[i];
  }
  tc::fence_proxy_async_smem();
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_f16_f32(128, n);
    for (int ks = 0; ks < kmain / 16; ++ks) {
      const int atom = ks >> 2, within = (ks & 3) * 32;
      const uint64_t da = tc::sdesc_k128(tc::smem_addr(sA + atom * 128 * 128 + within));
      const uint64_t db = tc::sdesc_k128(tc::smem_addr(sB + atom * n * 128 + within));
      tc::mma_f16(tmem, da, db, idesc, ks > 0 ? 1u : 0u);
    }
    if (ktail)
      tc::mma_f16(tmem, tc::sdesc_k16(tc::smem_addr(sAt)), tc::sdesc_k16(tc::smem_addr(sBt)),
                  idesc, 1u);
    tc::mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = tc::mbar_wait(&bar, 0, 1u << 22);
  if (!ok && (tid & 31) == 0) atomicCAS(status, 0, (int)GMM_ERR_TIMEOUT);
  tc::tc_fence_after();
  if (ok) {
    const int row = warp * 32 + (tid & 31);
    for (int c0 = 0; c0 < n; c0 += 32) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      for (int j = 0; j < 32; ++j) C[row * n + c0 + j] = v[j];
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

}  // namespace
}  // namespace gmm

// Test-only check of the tensor-core building blocks (declared in
// include/gmm_debug.h).  Returns 0 on launch success; *status_dev (device
// int32, zeroed by the caller) receives GMM_ERR_TIMEOUT if the MMA never
// completed.
extern "C" int gmm_debug_tc_gemm(const void* A, const void* B, float* C, int kdim, int n,
                                 int32_t* status_dev, void* stream) {
  if (!A || !B || !C || !status_dev) return GMM_ERR_INVALID_ARG;
  const int kmain = kdim & ~63, ktail = kdim & 63;
  if (!(kmain == 64 || kmain == 128 || kmain == 256) || !(ktail == 0 || ktail == 16) ||
      !(n == 64 || n == 128))
    return GMM_ERR_INVALID_ARG;
  const size_t smem = 1024 + (size_t)(128 + n) * (kmain + 16) * 2;
  cudaError_t e = cudaFuncSetAttribute(gmm::tc_gemm_check_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return GMM_ERR_CUDA;
  gmm::tc_gemm_check_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
      (const uint16_t*)A, (const uint16_t*)B, C, kdim, n, status_dev);
  return cudaGetLastError() == cudaSuccess ? GMM_OK : GMM_ERR_CUDA;
}
