// Ordered prefix scan of per-segment affine state maps (fp32 in and out). dk = dv = 128 runs
// on the tensor cores (kda_scan_tc, below); the other shapes on the CUDA cores (kda_scan_kernel).
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

#include <cstring>

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

// ---------------------------------------------------------------- tensor cores, dk = dv = 128
// The same recurrence on the tensor cores at fp32-level accuracy. Every fp32 operand v is
// written as three bf16 terms, v0 = bf16(v), v1 = bf16(v - v0), v2 = bf16(v - v0 - v1) (the
// differences are exact in fp32; what the three leave is below 2^-27 |v|), and X E is the sum
// of the six products X_a E_b with a + b <= 2, accumulated in fp32 by tcgen05.mma (the three
// dropped products are below 2^-24 |X||E|). One CTA per (head, SN = 16 value columns). Three
// MMA chains, one per term of X, each into its own accumulator in tensor memory (lane = row c
// of E) and issued interleaved, so that no instruction waits for the one before it:
//   P_0 = X_0 [E_0 | E_1 | E_2]     P_1 = X_1 [E_0 | E_1]     P_2 = X_2 E_0
//   E_{s+1} = Z_s + sum over a + b <= 2 of the block b of P_a.
// Two groups of eight warps:
//  - the X group has X loaded two steps ahead by tensor-map loads (one thread issues them),
//    splits it and writes the three terms into tensor memory, where the MMAs read their A
//    operand (two buffers, so that X_{s+1} and X_{s+2} are prepared while step s runs);
//  - the E group (whose thread 0 issues the MMAs) turns the accumulators into E_{s+1}: it adds
//    Z_s, writes E_out and puts the terms of E_{s+1} into the MMAs' B tile in shared memory,
//    MN-major (row c, value columns along the row: [E_0 | E_1 | E_2] in one 128-byte atom
//    column).
// Without S_init, E_1 = Z_0 needs no product and the chain starts at step 1.
namespace sct {
constexpr int SN = 16;                  // value columns per CTA
constexpr int CPT = SN / 2;             // value columns per E-group thread
constexpr int NT = 512;                 // threads per CTA: E group warps 0-7, X group 8-15
constexpr int PF = 4;                   // steps of X and Z prefetched into L2 ahead
constexpr uint32_t BT = 128 * 128;      // B tile: one atom column of 128 rows ([E_0|E_1|E_2])
constexpr uint32_t XS = 4 * 128 * 128;  // one staging slot: fp32 X as four 32-column boxes
constexpr uint32_t DYN = BT + 2 * XS + 1024;
constexpr int TA = 0;                   // tensor memory: terms of X in buffer b at TA + 192 b,
constexpr int TD = 384;                 //   the accumulators at TD .. TD + 6 SN
}  // namespace sct

// Tensor-memory column (from TD) of the accumulator of X_t [E_0 | .. | E_{2-t}] (3 - t) SN wide.
__host__ __device__ constexpr int dcol(int t) {
  return t == 0 ? 0 : (t == 1 ? 3 * sct::SN : 5 * sct::SN);
}

// (a, b) -> three bf16x2 words: the pair's hi, mid and lo terms (see above)
__device__ __forceinline__ void split3(float a, float b, uint32_t (&w)[3]) {
  const __nv_bfloat162 t0 = __floats2bfloat162_rn(a, b);
  const float2 f0 = __bfloat1622float2(t0);
  const float ra = a - f0.x, rb = b - f0.y;
  const __nv_bfloat162 t1 = __floats2bfloat162_rn(ra, rb);
  const float2 f1 = __bfloat1622float2(t1);
  const __nv_bfloat162 t2 = __floats2bfloat162_rn(ra - f1.x, rb - f1.y);
  w[0] = *reinterpret_cast<const uint32_t *>(&t0);
  w[1] = *reinterpret_cast<const uint32_t *>(&t1);
  w[2] = *reinterpret_cast<const uint32_t *>(&t2);
}

__global__ void __launch_bounds__(sct::NT, 1) kda_scan_tc(const __grid_constant__ CUtensorMap tm_x,
                                                          const float *__restrict__ X,
                                                          const float *__restrict__ Z, int n_seg,
                                                          int H, const float *__restrict__ S_init,
                                                          float *__restrict__ E_out,
                                                          float *__restrict__ S_final) {
  using sct::BT;
  using sct::CPT;
  using sct::PF;
  using sct::SN;
  using sct::TA;
  using sct::TD;
  using sct::XS;
  constexpr int D = 128;
  constexpr size_t HD = (size_t)D * D;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_xstage[2], bar_xfull[2], bar_xempty[2], bar_d;
  __shared__ uint32_t tmem_base;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const int h = blockIdx.x, q = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool egroup = warp < 8;
  const int c = (warp & 3) * 32 + lane;  // row of X and E = tensor-memory lane
  // E group: value columns CPT half .. + CPT of this CTA's SN; X group: K columns 64 half ..
  const int half = (warp >> 2) & 1;
  const int s_first = S_init ? 0 : 1;    // first step with products: E_0 = S_init, or E_1 = Z_0
  const size_t col = (size_t)c * D + q * SN + CPT * half;
  auto slab = [&](const float *base, int s) { return base + ((size_t)s * H + h) * HD; };
  auto oslab = [&](float *base, int s) { return base + ((size_t)s * H + h) * HD; };
  auto ld8 = [&](const float *p, float (&v)[CPT]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
  };
  auto st8 = [&](float *p, const float (&v)[CPT]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  };
  auto prefetch = [&](int s) {  // an eighth of X_s and Z_s per CTA (the eight cover the head)
    if (s >= s_first) prefetch_l2(slab(X, s) + q * (HD / 8), HD / 2);
    prefetch_l2(slab(Z, s) + q * (HD / 8), HD / 2);
  };
  // X group, one thread: X_s into staging slot `slot` by four tensor-map loads (32 columns x 128
  // rows each, 128-byte swizzle: the 16-byte chunk k of row r sits at chunk k ^ (r % 8))
  auto stage = [&](int s, int slot) {
    mbar_arrive_expect_tx(&bar_xstage[slot], XS);
#pragma unroll
    for (int bx = 0; bx < 4; ++bx)
      tma_load_2d(sm + BT + slot * XS + bx * 16384, &tm_x, 32 * bx, (s * H + h) * D,
                  &bar_xstage[slot]);
  };
  // E group: the terms of this thread's CPT values of row c into the B tile (one 16-byte
  // chunk per term)
  auto put_e = [&](const float (&e)[CPT]) {
    uint32_t w[3][4];
#pragma unroll
    for (int p2 = 0; p2 < 4; ++p2) {
      uint32_t t3[3];
      split3(e[2 * p2], e[2 * p2 + 1], t3);
      w[0][p2] = t3[0], w[1][p2] = t3[1], w[2][p2] = t3[2];
    }
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      const int n0 = SN * t + CPT * half;  // first value column of the chunk
      const uint32_t off = (n0 >> 6) * 16384 + c * 128 + ((((n0 & 63) >> 3) ^ (c & 7)) << 4);
      *reinterpret_cast<uint4 *>(sm + off) = make_uint4(w[t][0], w[t][1], w[t][2], w[t][3]);
    }
  };

  if (tid == 0)
    for (int s = 0; s < n_seg && s < PF; ++s) prefetch(s);
  float e[CPT], zc[CPT];
  if (s_first >= n_seg) {  // no products: the final state is the first entry state
    if (!egroup) return;
    if (S_init) {
      ld8(S_init + (size_t)h * HD + col, e);
    } else {
#pragma unroll
      for (int u = 0; u < CPT; ++u) e[u] = 0.f;
      if (n_seg > 0) ld8(slab(Z, 0) + col, e);
    }
    if (E_out && n_seg > 0) {  // n_seg = 1 without S_init: E_0 = 0
      const float zero[CPT] = {};
      st8(oslab(E_out, 0) + col, zero);
    }
    if (S_final) st8(S_final + (size_t)h * HD + col, e);
    return;
  }
  // both loads of the E group and both stagings of the X group in flight at once
  if (egroup) {
    ld8(S_init ? S_init + (size_t)h * HD + col : slab(Z, 0) + col, e);
    ld8(slab(Z, s_first) + col, zc);
  } else if (tid == 256) {
    for (int b = 0; b < 2; ++b) mbar_init(&bar_xstage[b], 1);
    fence_mbar_init();
    stage(s_first, 0);
    if (s_first + 1 < n_seg) stage(s_first + 1, 1);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_xfull[b], 8);  // one arrival per X-group warp
      mbar_init(&bar_xempty[b], 1);
    }
    mbar_init(&bar_d, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  bool ok = true;
  if (egroup) {
    if (E_out) {
      if (S_init) {
        st8(oslab(E_out, 0) + col, e);
      } else {
        const float zero[CPT] = {};
        st8(oslab(E_out, 0) + col, zero);
        st8(oslab(E_out, 1) + col, e);  // n_seg > 1 here
      }
    }
    put_e(e);
    fence_async_smem();
    named_bar(1, 256);  // the B tile of the first step is complete
    for (int s = s_first; s < n_seg; ++s) {
      const int i = s - s_first, b = i & 1;
      if (tid == 0) {
        // on a timeout nothing is issued, and the wait on bar_d below runs out as well
        if (mbar_wait(&bar_xfull[b], (i >> 1) & 1)) {
          tc_fence_after();
          // three independent accumulators, issued interleaved
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int t = 0; t < 3; ++t)
              mma_bf16_ts(tb + TD + dcol(t), tb + TA + 192 * b + 64 * t + 8 * kk,
                          desc_mnmajor(sb, 128, kk), idesc_bf16(128, 3 * SN - SN * t, 0, 1),
                          kk > 0 ? 1u : 0u);
          mma_commit(&bar_d);
          mma_commit(&bar_xempty[b]);
        }
        if (s + PF < n_seg) prefetch(s + PF);
      }
      const bool more = s + 1 < n_seg;
      float zn[CPT];
      if (more) ld8(slab(Z, s + 1) + col, zn);
      const bool good = mbar_wait(&bar_d, i & 1);
      tc_fence_after();
      if (good) {
        // X_a E_b at accumulator a, columns SN b
        float d00[CPT], d01[CPT], d02[CPT], d10[CPT], d11[CPT], d20[CPT];
        const uint32_t ta = tmem_addr(tb, (warp & 3) * 32, TD + CPT * half);
        tmem_ld8(ta + dcol(0), d00);
        tmem_ld8(ta + dcol(0) + SN, d01);
        tmem_ld8(ta + dcol(0) + 2 * SN, d02);
        tmem_ld8(ta + dcol(1), d10);
        tmem_ld8(ta + dcol(1) + SN, d11);
        tmem_ld8(ta + dcol(2), d20);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < CPT; ++u)
          e[u] = (d00[u] + ((d01[u] + d10[u]) + ((d02[u] + d11[u]) + d20[u]))) + zc[u];
        if (more) {
          if (E_out) st8(oslab(E_out, s + 1) + col, e);
          put_e(e);
        } else if (S_final) {
          st8(S_final + (size_t)h * HD + col, e);
        }
      }
      fence_async_smem();
      tc_fence_before();
      ok = named_bar_and(1, 256, good);
      tc_fence_after();
      if (!ok) break;
      if (more)
#pragma unroll
        for (int u = 0; u < CPT; ++u) zc[u] = zn[u];
    }
  } else {
    int issued = n_seg - s_first < 2 ? n_seg - s_first : 2, landed = 0;  // thread 256's counts
    for (int s = s_first; s < n_seg; ++s) {
      const int i = s - s_first, b = i & 1;
      bool good = mbar_wait(&bar_xstage[i & 1], (i >> 1) & 1);  // X_s has landed
      if (good) ++landed;
      if (good && i >= 2) good = mbar_wait(&bar_xempty[b], ((i >> 1) - 1) & 1);  // step s - 2 done
      tc_fence_after();
      if (good) {
        // boxes 2 half and 2 half + 1: K columns 64 half .. + 64 of row c
        const uint8_t *src = sm + BT + (i & 1) * XS + 2 * half * 16384 + c * 128;
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          uint32_t w[3][16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 x4 =
                *reinterpret_cast<const float4 *>(src + sub * 16384 + ((k ^ (c & 7)) << 4));
            uint32_t t3[3];
            split3(x4.x, x4.y, t3);
            w[0][2 * k] = t3[0], w[1][2 * k] = t3[1], w[2][2 * k] = t3[2];
            split3(x4.z, x4.w, t3);
            w[0][2 * k + 1] = t3[0], w[1][2 * k + 1] = t3[1], w[2][2 * k + 1] = t3[2];
          }
#pragma unroll
          for (int t = 0; t < 3; ++t)
            tmem_st16(
                tmem_addr(tb, (warp & 3) * 32, TA + 192 * b + 64 * t + 32 * half + 16 * sub),
                w[t]);
        }
      }
      // every X-group warp has read the slot before the loads that refill it are issued
      if (!named_bar_and(2, 256, good)) {
        ok = false;
        break;
      }
      if (tid == 256 && s + 2 < n_seg) {
        stage(s + 2, i & 1);
        ++issued;
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_xfull[b]);
    }
    if (!ok && tid == 256)  // loads still in flight land (bounded) before shared memory is freed
      for (; landed < issued; ++landed)
        if (!mbar_wait(&bar_xstage[landed & 1], (landed >> 1) & 1, 100000000ull)) break;
  }
  if (!ok && lane == 0) atomicOr(&g_scan_err, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

cudaError_t launch_scan_combine(const float *X, const float *Z, int n_seg, int H, int dk, int dv,
                                const float *S_init, float *E_out, float *S_final,
                                cudaStream_t st) {
  if (dk == 128 && dv == 128) {
    cudaError_t e = cudaFuncSetAttribute(kda_scan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sct::DYN);
    if (e != cudaSuccess) return e;
    CUtensorMap tm_x;  // X as (n_seg H 128) rows of 128 fp32 values
    memset(&tm_x, 0, sizeof(tm_x));
    if (n_seg > 0 && !make_rows_map_f32(&tm_x, X, (uint64_t)n_seg * H * 128))
      return cudaErrorInvalidValue;
    kda_scan_tc<<<dim3(H, 128 / sct::SN), sct::NT, sct::DYN, st>>>(tm_x, X, Z, n_seg, H, S_init,
                                                                   E_out, S_final);
    return cudaGetLastError();
  }
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
