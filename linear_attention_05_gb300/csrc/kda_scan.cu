// Ordered prefix scan of per-segment affine state maps (fp32).
//
// K3 training overview (zuoshipin.com/article/18261), section 3 "KDA context
// parallel": every segment emits how it rewrites the memory it is handed (X)
// and the state it builds from empty memory (Z); merging them in order
// recovers the exact state entering each segment:
//   E_0 = S_init,  E_s = X_{s-1} E_{s-1} + Z_{s-1},  S_final = X_{n-1} E_{n-1} + Z_{n-1}.
// Value columns of E are independent, so each block owns (head, 32 columns)
// and runs the n_seg dependent dk x dk by dk x 32 products in order, with its
// slice of E in shared memory.
#include <cuda_runtime.h>

#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int BV = 32;

template <int DK, int DV>
__global__ void __launch_bounds__(256) kda_scan_kernel(const float *__restrict__ X,
                                                       const float *__restrict__ Z, int n_seg,
                                                       int H, const float *__restrict__ S_init,
                                                       float *__restrict__ E_out,
                                                       float *__restrict__ S_final) {
  constexpr int LS = BV + 1, LX = DK + 1;
  __shared__ float sE[DK * LS];
  extern __shared__ float sX[];  // [DK][LX]
  const int h = blockIdx.x, j0 = blockIdx.y * BV, tid = threadIdx.x;
  const int jt = tid & 31, rt = tid >> 5;
  for (int c = rt; c < DK; c += 8)
    sE[c * LS + jt] = S_init ? S_init[((size_t)h * DK + c) * DV + j0 + jt] : 0.f;
  __syncthreads();
  for (int s = 0; s < n_seg; ++s) {
    const float *Xs = X + ((size_t)s * H + h) * DK * DK;
    const float *Zs = Z + ((size_t)s * H + h) * DK * DV;
    for (int e = tid; e < DK * DK; e += 256) sX[(e / DK) * LX + e % DK] = Xs[e];
    if (E_out)
      for (int c = rt; c < DK; c += 8)
        E_out[(((size_t)s * H + h) * DK + c) * DV + j0 + jt] = sE[c * LS + jt];
    __syncthreads();
    float acc[DK / 8];
#pragma unroll
    for (int m = 0; m < DK / 8; ++m) acc[m] = Zs[(size_t)(rt + 8 * m) * DV + j0 + jt];
    for (int l = 0; l < DK; ++l) {
      const float e = sE[l * LS + jt];
#pragma unroll
      for (int m = 0; m < DK / 8; ++m) acc[m] = fmaf(sX[(rt + 8 * m) * LX + l], e, acc[m]);
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < DK / 8; ++m) sE[(rt + 8 * m) * LS + jt] = acc[m];
    __syncthreads();
  }
  if (S_final)
    for (int c = rt; c < DK; c += 8) S_final[((size_t)h * DK + c) * DV + j0 + jt] = sE[c * LS + jt];
}

template <int DK, int DV>
cudaError_t launch_t(const float *X, const float *Z, int n_seg, int H, const float *S_init,
                     float *E_out, float *S_final, cudaStream_t st) {
  const size_t sm = sizeof(float) * DK * (DK + 1);
  cudaError_t e = cudaFuncSetAttribute(kda_scan_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  kda_scan_kernel<DK, DV><<<dim3(H, DV / BV), 256, sm, st>>>(X, Z, n_seg, H, S_init, E_out,
                                                              S_final);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scan_combine(const float *X, const float *Z, int n_seg, int H, int dk, int dv,
                                const float *S_init, float *E_out, float *S_final,
                                cudaStream_t st) {
  if (dk == 128 && dv == 128) return launch_t<128, 128>(X, Z, n_seg, H, S_init, E_out, S_final, st);
  if (dk == 64 && dv == 64) return launch_t<64, 64>(X, Z, n_seg, H, S_init, E_out, S_final, st);
  if (dk == 128 && dv == 64) return launch_t<128, 64>(X, Z, n_seg, H, S_init, E_out, S_final, st);
  if (dk == 64 && dv == 128) return launch_t<64, 128>(X, Z, n_seg, H, S_init, E_out, S_final, st);
  return cudaErrorInvalidValue;
}

}  // namespace kda
