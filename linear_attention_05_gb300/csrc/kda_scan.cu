// Ordered prefix scan of per-segment affine state maps (fp32).
//
// K3 training overview (zuoshipin.com/article/18261), section 3 "KDA context
// parallel": every segment emits how it rewrites the memory it is handed (X)
// and the state it builds from empty memory (Z); merging them in order
// recovers the exact state entering each segment:
//   E_0 = S_init,  E_s = X_{s-1} E_{s-1} + Z_{s-1},  S_final = X_{n-1} E_{n-1} + Z_{n-1}.
// Value columns of E are independent, so each block owns (head, 16 value
// columns) and runs the n_seg dependent dk x dk by dk x 16 products in order
// with its slice of E in shared memory, 256 threads x (8 rows, 1 column) each. X_{s+1} arrives
// by 16-byte asynchronous copies of all threads (into a padded double buffer) while step s
// computes.
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_common.cuh"

namespace kda {

__device__ unsigned g_scan_err;

namespace {

using namespace tc;

constexpr int BV = 16;   // value columns per block
constexpr int XP = 132;  // row pitch of X in shared memory (floats): 16-byte rows, no conflicts

template <int DK, int DV>
__global__ void __launch_bounds__(256) kda_scan_kernel(const float *__restrict__ X,
                                                       const float *__restrict__ Z, int n_seg,
                                                       int H, const float *__restrict__ S_init,
                                                       float *__restrict__ E_out,
                                                       float *__restrict__ S_final) {
  constexpr int RPT = DK / 16;  // rows per thread
  extern __shared__ __align__(16) float smem[];
  float *sX = smem;                 // [2][DK][XP]
  float *sE = smem + 2 * DK * XP;   // [DK][BV]
  const int h = blockIdx.x, j0 = blockIdx.y * BV, tid = threadIdx.x;
  const int jj = tid & 15, rg = tid >> 4;  // column, row group (rows rg + 16 m)
  for (int e = tid; e < DK * BV; e += 256) {
    const int c = e / BV, j = e % BV;
    sE[e] = S_init ? S_init[((size_t)h * DK + c) * DV + j0 + j] : 0.f;
  }
  __syncthreads();
  // X_s into buffer s % 2: 16-byte asynchronous copies spread over all threads (the load path;
  // one commit group per step, also when there is no such step)
  auto load_x = [&](int s) {
    if (s < n_seg) {
      const float *src = X + ((size_t)s * H + h) * DK * DK;
      const uint32_t dst = smem_u32(sX + (s & 1) * DK * XP);
      for (int e = tid; e < DK * DK / 4; e += 256) {
        const int c = e / (DK / 4), q4 = e % (DK / 4);
        cp_async16(dst + (c * XP + 4 * q4) * 4, src + (size_t)c * DK + 4 * q4);
      }
    }
    cp_async_commit();
  };
  load_x(0);
  for (int s = 0; s < n_seg; ++s) {
    const int b = s & 1;
    load_x(s + 1);  // the other buffer was read in step s - 1
    const float *Zs = Z + ((size_t)s * H + h) * DK * DV;
    float acc[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) acc[m] = Zs[(size_t)(rg + 16 * m) * DV + j0 + jj];
    if (E_out)
#pragma unroll
      for (int m = 0; m < RPT; ++m)
        E_out[(((size_t)s * H + h) * DK + rg + 16 * m) * DV + j0 + jj] = sE[(rg + 16 * m) * BV + jj];
    cp_async_wait_group<1>();  // X_s has landed (only X_{s+1} may be pending)
    __syncthreads();           // ... for every thread's part of it
    const float *xb = sX + b * DK * XP;
    for (int l = 0; l < DK; l += 4) {
      const float e0 = sE[(l + 0) * BV + jj], e1 = sE[(l + 1) * BV + jj];
      const float e2 = sE[(l + 2) * BV + jj], e3 = sE[(l + 3) * BV + jj];
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const float4 x = *reinterpret_cast<const float4 *>(xb + (rg + 16 * m) * XP + l);
        acc[m] = fmaf(x.x, e0, fmaf(x.y, e1, fmaf(x.z, e2, fmaf(x.w, e3, acc[m]))));
      }
    }
    __syncthreads();  // everyone is done reading sE and this X buffer
#pragma unroll
    for (int m = 0; m < RPT; ++m) sE[(rg + 16 * m) * BV + jj] = acc[m];
    __syncthreads();
  }
  cp_async_wait_group<0>();  // nothing left in flight
  if (S_final)
#pragma unroll
    for (int m = 0; m < RPT; ++m)
      S_final[((size_t)h * DK + rg + 16 * m) * DV + j0 + jj] = sE[(rg + 16 * m) * BV + jj];
}

template <int DK, int DV>
cudaError_t launch_t(const float *X, const float *Z, int n_seg, int H, const float *S_init,
                     float *E_out, float *S_final, cudaStream_t st) {
  const size_t sm = sizeof(float) * (2 * DK * XP + DK * BV);
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

cudaError_t scan_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_scan_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_scan_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

}  // namespace kda
