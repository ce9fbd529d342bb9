// Ordered prefix scan of per-segment affine state maps (fp32).
//
// K3 training overview (zuoshipin.com/article/18261), section 3 "KDA context
// parallel": every segment emits how it rewrites the memory it is handed (X)
// and the state it builds from empty memory (Z); merging them in order
// recovers the exact state entering each segment:
//   E_0 = S_init,  E_s = X_{s-1} E_{s-1} + Z_{s-1},  S_final = X_{n-1} E_{n-1} + Z_{n-1}.
// Value columns of E are independent, so each block owns (head, 16 value
// columns) and runs the n_seg dependent dk x dk by dk x 16 products in order
// with its slice of E double-buffered (transposed) in shared memory, 256 threads x
// (dk / 32 rows, 2 columns) each, one barrier per step. X_{s+1} arrives by 16-byte asynchronous copies of all threads
// (into a padded double buffer) and Z_{s+1} into registers while step s computes.
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_common.cuh"

namespace kda {

__device__ unsigned g_scan_err;

namespace {

using namespace tc;

constexpr int BV = 16;   // value columns per block
constexpr int NT = 256;   // threads per block
constexpr int XP = 132;  // row pitch of X in shared memory (floats): 16-byte rows, no conflicts

template <int DK, int DV>
__global__ void __launch_bounds__(NT, 1) kda_scan_kernel(const float *__restrict__ X,
                                                      const float *__restrict__ Z, int n_seg,
                                                      int H, const float *__restrict__ S_init,
                                                      float *__restrict__ E_out,
                                                      float *__restrict__ S_final) {
  constexpr int RG = NT / 8;    // row groups: rows rg + RG m
  constexpr int RPT = DK / RG;  // rows per thread
  constexpr int EP = DK + 4;    // row pitch of the transposed E slice (floats)
  extern __shared__ __align__(16) float smem[];
  float *sX = smem;                 // [2][DK][XP]: X_s in buffer s % 2
  float *sE = smem + 2 * DK * XP;   // [2][BV][EP]: E_s^T (column j of the slice = row j) in buffer s % 2
  const int h = blockIdx.x, j0 = blockIdx.y * BV, tid = threadIdx.x;
  // columns jc and jc + 8 (their E^T rows sit 4 banks apart for neighbouring jc), rows
  // rg + RG m: each 16-byte load of X or E feeds 8 or 4 of this thread's FMAs
  const int jc = tid & 7, rg = tid >> 3;
  auto load_x = [&](int s) {  // X_s into buffer s % 2, one commit group per call
    if (s < n_seg) {
      const float *src = X + ((size_t)s * H + h) * DK * DK;
      const uint32_t dst = smem_u32(sX + (s & 1) * DK * XP);
      for (int e = tid; e < DK * DK / 4; e += NT) {
        const int c = e / (DK / 4), q4 = e % (DK / 4);
        cp_async16(dst + (c * XP + 4 * q4) * 4, src + (size_t)c * DK + 4 * q4);
      }
    }
    cp_async_commit();
  };
  auto gidx = [&](int c, int q) { return (size_t)c * DV + j0 + jc + 8 * q; };  // within [DK, DV]
  auto load_z = [&](int s, float (*z)[2]) {
#pragma unroll
    for (int m = 0; m < RPT; ++m)
#pragma unroll
      for (int q = 0; q < 2; ++q)
        z[m][q] = s < n_seg ? Z[((size_t)s * H + h) * DK * DV + gidx(rg + RG * m, q)] : 0.f;
  };
  load_x(0);
  load_x(1);
  for (int e = tid; e < DK * BV; e += NT) {
    const int c = e / BV, j = e % BV;
    sE[j * EP + c] = S_init ? S_init[((size_t)h * DK + c) * DV + j0 + j] : 0.f;
  }
  float zn[RPT][2];
  load_z(0, zn);
  cp_async_wait_group<1>();  // X_0 has landed (X_1 may be pending)
  __syncthreads();           // ... for every thread's part of it, and E_0
  // Step s reads X_s and E_s and writes E_{s+1} into the other E buffer, so one barrier per
  // step suffices: after it E_{s+1} and X_{s+1} are complete and buffer s % 2 of X is free
  // for X_{s+2}. Z_{s+1} is loaded into registers while step s computes.
  for (int s = 0; s < n_seg; ++s) {
    const float *xb = sX + (s & 1) * DK * XP;
    const float *eb = sE + (s & 1) * BV * EP;
    float acc[RPT][2];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
      acc[m][0] = zn[m][0];
      acc[m][1] = zn[m][1];
    }
    load_z(s + 1, zn);
    if (E_out)
#pragma unroll
      for (int m = 0; m < RPT; ++m)
#pragma unroll
        for (int q = 0; q < 2; ++q)
          E_out[((size_t)s * H + h) * DK * DV + gidx(rg + RG * m, q)] =
              eb[(jc + 8 * q) * EP + rg + RG * m];
#pragma unroll
    for (int l = 0; l < DK; l += 4) {
      const float4 e0 = *reinterpret_cast<const float4 *>(eb + jc * EP + l);
      const float4 e1 = *reinterpret_cast<const float4 *>(eb + (jc + 8) * EP + l);
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const float4 x = *reinterpret_cast<const float4 *>(xb + (rg + RG * m) * XP + l);
        acc[m][0] = fmaf(x.x, e0.x, fmaf(x.y, e0.y, fmaf(x.z, e0.z, fmaf(x.w, e0.w, acc[m][0]))));
        acc[m][1] = fmaf(x.x, e1.x, fmaf(x.y, e1.y, fmaf(x.z, e1.z, fmaf(x.w, e1.w, acc[m][1]))));
      }
    }
    float *en = sE + ((s + 1) & 1) * BV * EP;
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
      en[jc * EP + rg + RG * m] = acc[m][0];
      en[(jc + 8) * EP + rg + RG * m] = acc[m][1];
    }
    cp_async_wait_group<0>();  // X_{s+1} (the only group in flight) has landed
    __syncthreads();
    load_x(s + 2);             // into the buffer step s read
  }
  cp_async_wait_group<0>();  // nothing left in flight
  if (S_final) {
    const float *eb = sE + (n_seg & 1) * BV * EP;
#pragma unroll
    for (int m = 0; m < RPT; ++m)
#pragma unroll
      for (int q = 0; q < 2; ++q)
        S_final[(size_t)h * DK * DV + gidx(rg + RG * m, q)] = eb[(jc + 8 * q) * EP + rg + RG * m];
  }
}

template <int DK, int DV>
cudaError_t launch_t(const float *X, const float *Z, int n_seg, int H, const float *S_init,
                     float *E_out, float *S_final, cudaStream_t st) {
  const size_t sm = sizeof(float) * (2 * DK * XP + 2 * BV * (DK + 4));
  cudaError_t e = cudaFuncSetAttribute(kda_scan_kernel<DK, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  kda_scan_kernel<DK, DV><<<dim3(H, DV / BV), NT, sm, st>>>(X, Z, n_seg, H, S_init, E_out,
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
