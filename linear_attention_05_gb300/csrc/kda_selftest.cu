// Tensor-core layout self-test: one CTA computes D = A * B with tcgen05.mma
// from 128-byte-swizzled shared-memory tiles in a chosen operand layout
// (K-major or MN-major for A and for B) and writes D (fp32) back. The
// chunked kernels use exactly these tile conventions, so a host-side
// comparison with a plain matrix product validates the descriptor encoding
// on the device at hand.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda_selftest.h"
#include "kda_common.cuh"
#include "tc_common.cuh"

namespace {

using namespace kda::tc;

__device__ unsigned g_selftest_err;
// error word of the bounded-wait self-test, read and cleared by kda_get_error()
__device__ unsigned g_wait_test_err;

// A: [M x K] row-major bf16; B: [K x N] row-major bf16; D: [M x N] fp32.
__global__ void __launch_bounds__(128) umma_selftest_kernel(const __nv_bfloat16 *A,
                                                            const __nv_bfloat16 *B, float *D,
                                                            int M, int N, int K, int a_mn,
                                                            int b_mn) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sA = base;
  uint8_t *sB = base + ((M * K * 2 + 1023) & ~1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int e = tid; e < M * K; e += 128) {
    const int m = e / K, k = e % K;
    const uint32_t off = a_mn ? sw128_off(k, m, K) : sw128_off(m, k, M);
    *reinterpret_cast<__nv_bfloat16 *>(sA + off) = A[e];
  }
  for (int e = tid; e < K * N; e += 128) {
    const int k = e / N, n = e % N;
    const uint32_t off = b_mn ? sw128_off(k, n, K) : sw128_off(n, k, N);
    *reinterpret_cast<__nv_bfloat16 *>(sB + off) = B[e];
  }
  fence_async_smem();
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  if (tid == 0) {
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    const uint32_t idesc = idesc_bf16(M, N, a_mn, b_mn);
    for (int kk = 0; kk < K / 16; ++kk) {
      uint64_t ad, bd;
      // MN-major: K rows of 128 bytes, MN atom columns K * 128 bytes apart
      ad = a_mn ? desc_mnmajor(a0, K, kk) : desc_kmajor(a0, M, kk);
      bd = b_mn ? desc_mnmajor(b0, K, kk) : desc_kmajor(b0, N, kk);
      mma_bf16(tb, ad, bd, idesc, kk > 0 ? 1u : 0u);
    }
    mma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0);
  if (!ok && lane == 0) atomicOr(&g_selftest_err, 1u);
  tc_fence_after();
  if (ok && warp * 32 < M) {
    for (int c = 0; c < N; c += 32) {
      float v[32];
      tmem_ld32(tmem_addr(tb, warp * 32, c), v);
      tmem_wait_ld();
      const int row = warp * 32 + lane;
#pragma unroll
      for (int i = 0; i < 32; ++i) D[(size_t)row * N + c + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}

// Bounded-wait self-test: one CTA of 128 threads waits on an mbarrier that nothing will ever
// arrive on (no bulk copy and no MMA is issued against it), for at most limit_ns on every
// thread, exactly as the chunked kernels wait on their copies and MMAs. The threads then vote
// with a barrier that ANDs their results, as the state pass does, so that every warp leaves
// by the same branch; on a timeout one thread records it in the error word, and the kernel
// returns normally.
__global__ void __launch_bounds__(128) wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = named_bar_and(1, 128, mbar_wait(&bar, 0, limit_ns));
  if (!ok && threadIdx.x == 0) atomicOr(&g_wait_test_err, kda::kErrTimeout);
}

}  // namespace

namespace kda {
cudaError_t selftest_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_wait_test_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_wait_test_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}
}  // namespace kda

extern "C" int kda_selftest_wait_timeout(unsigned limit_us, kda_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return KDA_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 128, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000ull);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" int kda_selftest_umma(const void *A, const void *B, float *D, int M, int N, int K,
                                 int a_mn_major, int b_mn_major, kda_stream_t stream) {
  if (M != 128 || N < 16 || N > 256 || N % 32 != 0 || K < 16 || K > 128 || K % 64 != 0)
    return KDA_ERR_UNSUPPORTED;
  if (!A || !B || !D) return KDA_ERR_INVALID_ARG;
  const int smem = ((M * K * 2 + 1023) & ~1023) + K * N * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(umma_selftest_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  unsigned z = 0;
  cudaMemcpyToSymbolAsync(g_selftest_err, &z, sizeof(z), 0, cudaMemcpyHostToDevice,
                          (cudaStream_t)stream);
  umma_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
      (const __nv_bfloat16 *)A, (const __nv_bfloat16 *)B, D, M, N, K, a_mn_major, b_mn_major);
  e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  unsigned v = 0;
  cudaMemcpyFromSymbol(&v, g_selftest_err, sizeof(v));
  return v ? KDA_ERR_TIMEOUT : KDA_OK;
}
