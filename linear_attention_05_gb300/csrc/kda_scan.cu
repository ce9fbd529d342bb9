// Ordered prefix scan of per-segment affine state maps (fp32).
//
// K3 training overview (zuoshipin.com/article/18261), section 3 "KDA context
// parallel": every segment emits how it rewrites the memory it is handed (X)
// and the state it builds from empty memory (Z); merging them in order
// recovers the exact state entering each segment:
//   E_0 = S_init,  E_s = X_{s-1} E_{s-1} + Z_{s-1},  S_final = X_{n-1} E_{n-1} + Z_{n-1}.
// Value columns of E are independent, so each block owns (head, 16 value
// columns) and runs the n_seg dependent dk x dk by dk x 16 products in order
// with its slice of E in shared memory, 256 threads x (8 rows, 1 column) each. X_s arrives by bulk copies (one per
// row, into a padded double buffer) while step s - 1 computes.
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
  __shared__ uint64_t bar[2];
  const int h = blockIdx.x, j0 = blockIdx.y * BV, tid = threadIdx.x;
  const int jj = tid & 15, rg = tid >> 4;  // column, row group (rows rg + 16 m)
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  for (int e = tid; e < DK * BV; e += 256) {
    const int c = e / BV, j = e % BV;
    sE[e] = S_init ? S_init[((size_t)h * DK + c) * DV + j0 + j] : 0.f;
  }
  __syncthreads();
  auto load_x = [&](int s) {  // warp 0: one bulk copy per row of X_s
    const int b = s & 1;
    if (tid == 0) mbar_arrive_expect_tx(&bar[b], DK * DK * 4);
    __syncwarp();
    const float *src = X + ((size_t)s * H + h) * DK * DK;
    for (int c = tid; c < DK; c += 32) bulk_g2s(sX + (b * DK + c) * XP, src + (size_t)c * DK, DK * 4, &bar[b]);
  };
  if (tid < 32 && n_seg > 0) load_x(0);
  uint32_t phase[2] = {0u, 0u};
  bool ok = true;
  for (int s = 0; s < n_seg && ok; ++s) {
    const int b = s & 1;
    if (tid < 32 && s + 1 < n_seg) load_x(s + 1);  // the other buffer was read in step s - 1
    const float *Zs = Z + ((size_t)s * H + h) * DK * DV;
    float acc[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) acc[m] = Zs[(size_t)(rg + 16 * m) * DV + j0 + jj];
    if (E_out)
#pragma unroll
      for (int m = 0; m < RPT; ++m)
        E_out[(((size_t)s * H + h) * DK + rg + 16 * m) * DV + j0 + jj] = sE[(rg + 16 * m) * BV + jj];
    // every thread takes the same branch, so a timeout cannot strand others at a barrier
    if (!__syncthreads_and(mbar_wait(&bar[b], phase[b]))) {
      ok = false;
      break;
    }
    phase[b] ^= 1u;
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
  if (!ok) {
    if (tid == 0) {
      atomicOr(&g_scan_err, kErrTimeout);
      // let a copy still in flight land (bounded) before shared memory is released
      for (int b = 0; b < 2; ++b) mbar_wait(&bar[b], phase[b], 100000000ull);
    }
    return;
  }
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
