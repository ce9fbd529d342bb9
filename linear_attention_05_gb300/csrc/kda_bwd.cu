// Chunked backward pass of KDA (fp32; the batched contractions and, at dk = dv = 128, the
// forward replay's and the reverse state pass on the tensor cores at fp32-level accuracy; the
// preparation, the substitutions and the element-wise work on CUDA cores).
//
// Gradients of L = <dO, o> + <dS_final, S_final> with respect to q, k, v,
// log_alpha, beta, gate and the initial state. The forward is the chunked form
// of K3 training overview (zuoshipin.com/article/18261) section 4 "FlashKDA"
// (per-chunk preparation, then the ordered state hand-off); section 4 presents it
// as a training kernel, so it needs these gradients. Per chunk, with S the state
// entering the chunk and S' the state leaving it (operands as in the forward):
//   U = U~ - W S,  O = Q~ S + P U,  S' = Diag(e^{G_C}) S + K_d^T U,  o = scale g O,
//   W = T diag(b) K~,  U~ = T diag(b) V,  T = (I + A)^-1,  A = strict_lower(diag(b) K~ K^^T).
// Reverse mode, given dS' and dO = scale g do:
//   dU  = P^T dO + K_d dS'                       dS  = Diag(e^{G_C}) dS' + Q~^T dO - W^T dU
//   dP  = lower(dO U^T)                          dQ~ = dO S^T + dP K^
//   dK_d = U dS'^T                               dW  = -dU S^T
//   [dB_k | dB_v] = T^T [dW | dU]                dA  = strict_lower(-dB_k W^T - dB_v U~^T)
//   dK~ = diag(b) (dA K^ + dB_k)                 dK^ = dP^T Q~ + dA^T diag(b) K~
//   db  = rowdot(K~, dA K^ + dB_k) + rowdot(V, dB_v),   dv = diag(b) dB_v
// then through K~ = k e^G, K^ = k e^-G, Q~ = q e^G, K_d = k e^{G_C - G}, e^{G_C}
// to k, q and the running log-decay G, whose reverse cumulative sum gives
// dlog_alpha, and through the optional L2 normalisation of q and k.
//
// Launch sequence (all on the caller's stream): chunk table; prep (forward
// operands + K^, diag(b)K~, A); forward state pass saving S and U per chunk;
// O = Q~ S + P U, V1 = P^T dO and R = Q~^T dO (batched tensor-core GEMMs); reverse state
// pass (dS' per chunk, dU, dS_0); seven more batched 64-row GEMMs; one triangular
// solve; the finishing kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_common.cuh"

namespace kda {

__device__ unsigned g_bwd_err;

namespace {

constexpr int C = kChunk;  // 64

__device__ __forceinline__ float bf(float x) { return x; }
__device__ __forceinline__ float bf(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T to_out(float x);
template <>
__device__ __forceinline__ float to_out<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float wsum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// token range of chunk ci (global index) -> (sequence, first token, valid rows)
__device__ __forceinline__ void chunk_rows(const int32_t *cu, int64_t fixed_len, int n_seq,
                                           const int *off, int ci, int *s_out, int64_t *t0,
                                           int *len) {
  int lo = 0, hi = n_seq - 1;  // last s with off[s] <= ci (skipping empty sequences)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= ci) lo = mid;
    else hi = mid - 1;
  }
  const int s = lo;
  int64_t ts, ls;
  if (cu) {
    ts = cu[s];
    ls = (int64_t)cu[s + 1] - cu[s];
  } else {
    ts = (int64_t)s * fixed_len;
    ls = fixed_len;
  }
  const int j = ci - off[s];
  *s_out = s;
  *t0 = ts + (int64_t)j * C;
  *len = (int)min((int64_t)C, ls - (int64_t)j * C);
}

// ---------------------------------------------------------------------------
// dO = scale * g * do in chunk layout [slab][64][dv] (zero on padded rows)
template <int DV, typename Tin>
__global__ void __launch_bounds__(256) kda_bwd_dO(const Tin *__restrict__ d_out,
                                                  const Tin *__restrict__ gate,
                                                  const int32_t *__restrict__ cu, int n_seq,
                                                  int64_t fixed_len, int H, float scale,
                                                  unsigned flags,
                                                  const ChunkMeta *__restrict__ meta,
                                                  const int *__restrict__ off,
                                                  float *__restrict__ dO) {
  const int ci = blockIdx.x, h = blockIdx.y;
  if (meta->invalid || ci >= meta->total_chunks) return;
  int s, len;
  int64_t t0;
  chunk_rows(cu, fixed_len, n_seq, off, ci, &s, &t0, &len);
  float *dst = dO + ((size_t)ci * H + h) * C * DV;
  for (int e = threadIdx.x; e < C * DV; e += 256) {
    const int r = e / DV, j = e % DV;
    float x = 0.f;
    if (r < len) {
      const size_t g = ((size_t)(t0 + r) * H + h) * DV + j;
      x = scale * bf(d_out[g]) * (gate ? prep_gate(bf(gate[g]), flags) : 1.f);
    }
    dst[e] = x;
  }
}

// ---------------------------------------------------------------------------
// Reverse state pass: one block per (sequence, head, 32 value columns), chunks
// last to first. With V1 = P^T dO and R = Q~^T dO precomputed per chunk (they do
// not depend on the state), the serial step is
//   dU = V1 + K_d dS',   dS = Diag(e^{G_C}) dS' + R - W^T dU.
// Writes dS' (the cotangent of the state leaving each chunk) and dU per chunk, and
// dS_0. Register-tiled: thread (rg, cg) = (tid >> 3, tid & 7) owns value columns
// 4cg..4cg+3 and key rows 4rg..4rg+3 of dS (rows 2rg, 2rg+1 of dU); W and K_d^T
// come from shared memory as 16- and 8-byte vectors, V1 and R straight from global
// memory. About 106 KB of shared memory at dk = 128: two blocks per SM.
constexpr int RBV = 32;

template <int DK, int DV>
__global__ void __launch_bounds__(256) kda_bwd_state(
    const float *__restrict__ dS_final, float *__restrict__ dS_init,
    const int32_t *__restrict__ cu, int n_seq, int64_t fixed_len, int H,
    const ChunkMeta *__restrict__ meta, const int *__restrict__ off,
    const float *__restrict__ Wg, const float *__restrict__ Kdg, const float *__restrict__ Dg,
    const float *__restrict__ V1g, const float *__restrict__ Rg, float *__restrict__ dSb,
    float *__restrict__ dUg) {
  static_assert(DK / 4 <= 32 && C / 2 <= 32, "row groups");
  constexpr int LK = DK + 4, LS = RBV + 4, LC = C + 4;  // float4-aligned pitches
  extern __shared__ __align__(16) float smem[];
  float *sS = smem;            // [DK][LS]   running dS (value-column slice)
  float *sU = sS + DK * LS;    // [C][LS]    dU slice
  float *sW = sU + C * LS;     // [C][LK]    W
  float *sKt = sW + C * LK;    // [DK][LC]   K_d^T
  float *sD = sKt + DK * LC;   // [DK]
  if (meta->invalid) return;
  const int chain = blockIdx.x, s = chain / H, h = chain % H, tid = threadIdx.x;
  const int j0 = blockIdx.y * RBV;
  const int cg = tid & 7, rg = tid >> 3;
  const int jl = 4 * cg;                 // local value column of this thread
  const bool s_rows = rg < DK / 4;       // dS rows 4rg..4rg+3
  const bool u_rows = rg < C / 2;        // dU rows 2rg, 2rg+1
  for (int e = tid; e < DK * RBV; e += 256) {
    const int c = e / RBV, jj = e % RBV;
    sS[c * LS + jj] =
        dS_final ? dS_final[(((size_t)s * H + h) * DK + c) * DV + j0 + jj] : 0.f;
  }
  int64_t ls;
  if (cu) ls = (int64_t)cu[s + 1] - cu[s];
  else ls = fixed_len;
  const int nchunks = (int)((ls + C - 1) / C);
  __syncthreads();
  for (int jc = nchunks - 1; jc >= 0; --jc) {
    const size_t slab = (size_t)(off[s] + jc) * H + h;
    if (tid == 0 && blockIdx.y == 0 && jc > 0) {  // the next chunk's operands into L2
      const size_t sp = slab - H;                  // chunk jc - 1 of this sequence and head
      prefetch_l2_bulk(Wg + sp * C * DK, C * DK * 4);
      prefetch_l2_bulk(Kdg + sp * C * DK, C * DK * 4);
      prefetch_l2_bulk(V1g + sp * C * DV, C * DV * 4);
      prefetch_l2_bulk(Rg + sp * DK * DV, DK * DV * 4);
    }
    for (int e = tid; e < DK * RBV; e += 256) {
      const int c = e / RBV, jj = e % RBV;
      dSb[(slab * DK + c) * DV + j0 + jj] = sS[c * LS + jj];
    }
    // this thread's V1 and R elements (issued early: they are read after the stores below)
    float4 v1a = make_float4(0.f, 0.f, 0.f, 0.f), v1b = v1a, rr[4];
    if (u_rows) {
      v1a = *reinterpret_cast<const float4 *>(V1g + (slab * C + 2 * rg) * DV + j0 + jl);
      v1b = *reinterpret_cast<const float4 *>(V1g + (slab * C + 2 * rg + 1) * DV + j0 + jl);
    }
    if (s_rows)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        rr[u] = *reinterpret_cast<const float4 *>(Rg + (slab * DK + 4 * rg + u) * DV + j0 + jl);
    {  // W and K_d of chunk jc: 16-byte loads, all issued before their stores
      constexpr int NK = C * DK / 4 / 256;
      const float *W = Wg + slab * C * DK, *Kd = Kdg + slab * C * DK;
      float4 rw[NK], rk[NK];
#pragma unroll
      for (int m = 0; m < NK; ++m) {
        rw[m] = *reinterpret_cast<const float4 *>(W + 4 * (tid + 256 * m));
        rk[m] = *reinterpret_cast<const float4 *>(Kd + 4 * (tid + 256 * m));
      }
#pragma unroll
      for (int m = 0; m < NK; ++m) {
        const int e = 4 * (tid + 256 * m), r = e / DK, c = e % DK;
        *reinterpret_cast<float4 *>(sW + r * LK + c) = rw[m];
        sKt[(c + 0) * LC + r] = rk[m].x; sKt[(c + 1) * LC + r] = rk[m].y;
        sKt[(c + 2) * LC + r] = rk[m].z; sKt[(c + 3) * LC + r] = rk[m].w;
      }
      if (tid < DK) sD[tid] = Dg[slab * DK + tid];
    }
    __syncthreads();
    // dU = V1 + K_d dS'
    if (u_rows) {
      const int r0 = 2 * rg;
      float a0[4] = {v1a.x, v1a.y, v1a.z, v1a.w}, a1[4] = {v1b.x, v1b.y, v1b.z, v1b.w};
#pragma unroll 4
      for (int c = 0; c < DK; ++c) {
        const float2 kd = *reinterpret_cast<const float2 *>(sKt + c * LC + r0);
        const float4 d = *reinterpret_cast<const float4 *>(sS + c * LS + jl);
        a0[0] = fmaf(kd.x, d.x, a0[0]); a0[1] = fmaf(kd.x, d.y, a0[1]);
        a0[2] = fmaf(kd.x, d.z, a0[2]); a0[3] = fmaf(kd.x, d.w, a0[3]);
        a1[0] = fmaf(kd.y, d.x, a1[0]); a1[1] = fmaf(kd.y, d.y, a1[1]);
        a1[2] = fmaf(kd.y, d.z, a1[2]); a1[3] = fmaf(kd.y, d.w, a1[3]);
      }
      *reinterpret_cast<float4 *>(sU + r0 * LS + jl) = make_float4(a0[0], a0[1], a0[2], a0[3]);
      *reinterpret_cast<float4 *>(sU + (r0 + 1) * LS + jl) = make_float4(a1[0], a1[1], a1[2], a1[3]);
      *reinterpret_cast<float4 *>(dUg + (slab * C + r0) * DV + j0 + jl) =
          make_float4(a0[0], a0[1], a0[2], a0[3]);
      *reinterpret_cast<float4 *>(dUg + (slab * C + r0 + 1) * DV + j0 + jl) =
          make_float4(a1[0], a1[1], a1[2], a1[3]);
    }
    __syncthreads();
    // dS = Diag(e^{G_C}) dS' + R - W^T dU
    float ns[4][4];
    if (s_rows) {
      const int c0 = 4 * rg;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 d = *reinterpret_cast<const float4 *>(sS + (c0 + u) * LS + jl);
        const float dc = sD[c0 + u];
        ns[u][0] = fmaf(dc, d.x, rr[u].x); ns[u][1] = fmaf(dc, d.y, rr[u].y);
        ns[u][2] = fmaf(dc, d.z, rr[u].z); ns[u][3] = fmaf(dc, d.w, rr[u].w);
      }
#pragma unroll 2
      for (int r = 0; r < C; ++r) {
        const float4 w = *reinterpret_cast<const float4 *>(sW + r * LK + c0);
        const float4 du = *reinterpret_cast<const float4 *>(sU + r * LS + jl);
        const float wa[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ns[u][0] = fmaf(-wa[u], du.x, ns[u][0]); ns[u][1] = fmaf(-wa[u], du.y, ns[u][1]);
          ns[u][2] = fmaf(-wa[u], du.z, ns[u][2]); ns[u][3] = fmaf(-wa[u], du.w, ns[u][3]);
        }
      }
    }
    __syncthreads();
    if (s_rows)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<float4 *>(sS + (4 * rg + u) * LS + jl) =
            make_float4(ns[u][0], ns[u][1], ns[u][2], ns[u][3]);
    __syncthreads();
  }
  if (dS_init)
    for (int e = tid; e < DK * RBV; e += 256) {
      const int c = e / RBV, jj = e % RBV;
      dS_init[(((size_t)s * H + h) * DK + c) * DV + j0 + jj] = sS[c * LS + jj];
    }
}

template <int DK>
constexpr size_t bwd_state_smem() {
  return sizeof(float) * (DK * (RBV + 4) + C * (RBV + 4) + C * (DK + 4) + DK * (C + 4) + DK);
}

// The state passes of the backward on the tensor cores (dk = dv = 128), one CTA (256 threads)
// per (sequence, head), the state kept transposed in tensor memory (lane = value column j,
// column = key c). Reverse (FWD = false), each chunk last to first:
//   dU^T  = dS'^T K_d^T + V1^T                    (M = 128 j, N = 64 tokens, K = 128 c)
//   dS^T  = Diag(e^{G_C}) dS'^T + R^T - dU^T W     (M = 128 j, N = 128 c,     K = 64 tokens)
// writing dS' and dU per chunk. The forward replay (FWD = true), first to last, is the same
// pair of products with the roles of W and K_d swapped:
//   U^T   = U~^T - S^T W^T,      S'^T = Diag(e^{G_C}) S^T + U^T K_d
// writing S and U per chunk. The accumulator of the second product is pre-loaded with its
// first terms. Every fp32
// operand enters as three bf16 terms (v0 = bf16(v), v1 = bf16(v - v0), v2 = bf16(v - v0 - v1))
// and the six products of terms a + b <= 2 are accumulated in fp32, so the pass keeps fp32-level
// accuracy. Shared memory: the A operand (the terms of dS'^T, then of dU^T, K-major) and the B
// operands (the terms of K_d, K-major, and of W, MN-major: both are [token][c] in memory).
namespace bst {
constexpr int NT = 256;
constexpr uint32_t SA = 0;            // 3 x 32 KB: dS'^T terms (128 x 128), later dU^T (128 x 64)
constexpr uint32_t SB1 = 3 * 32768;   // 3 x 16 KB: K_d terms, 64 token rows x 128 c
constexpr uint32_t SB2 = SB1 + 3 * 16384;  // 3 x 16 KB: W terms, 64 token rows x 128 c
constexpr uint32_t DYN = SB2 + 3 * 16384 + 1024;
constexpr int TS = 0;                 // tensor memory: the state dS^T in columns [0, 128)
constexpr int TU = 128;               //   dU^T in columns [128, 192)
}  // namespace bst

// (a, b) -> the bf16x2 words of the pair's three terms
__device__ __forceinline__ void bst_split(float a, float b, uint32_t (&w)[3]) {
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

// S_first: the state entering the first step (dS_final, or S_0), or null for 0; S_last: where
// the state after the last step goes (dS_0), or null. B1g, B2g: the [token][c] operands of the
// first and second product (K_d and W reversed, W and K_d forward); Xg: V1 or U~ ([token][j]);
// Rg: R ([c][j], reverse only); Sb, Ub: the per-chunk state and dU or U.
template <bool FWD>
__global__ void __launch_bounds__(bst::NT, 1) kda_bwd_state_tc(
    const float *__restrict__ S_first, float *__restrict__ S_last,
    const int32_t *__restrict__ cu, int n_seq, int64_t fixed_len, int H,
    const ChunkMeta *__restrict__ meta, const int *__restrict__ off,
    const float *__restrict__ B1g, const float *__restrict__ B2g, const float *__restrict__ Dg,
    const float *__restrict__ Xg, const float *__restrict__ Rg, float *__restrict__ Sb,
    float *__restrict__ Ub) {
  using namespace tc;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base;
  if (meta->invalid) return;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const int chain = blockIdx.x, s = chain / H, h = chain % H, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, quad = warp & 3, hh = warp >> 2;
  // this thread: value column j (tensor-memory lane), key columns 64 hh .. + 64 of the state,
  // tokens 32 hh .. + 32 of dU
  const int j = quad * 32 + lane;
  int64_t ls;
  if (cu) ls = (int64_t)cu[s + 1] - cu[s];
  else ls = fixed_len;
  const int nchunks = (int)((ls + C - 1) / C);
  const size_t st0 = ((size_t)s * H + h) * D * D;  // this chain's [dk][dv] state slab
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  const uint32_t trow = tmem_addr(tb, quad * 32, 0);
  {  // the state entering the first step
    float v[32];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int c = 64 * hh + 32 * half + u;
        v[u] = S_first ? S_first[st0 + (size_t)c * D + j] : 0.f;
      }
      tmem_st32(trow + bst::TS + 64 * hh + 32 * half, v);
    }
    tmem_wait_st();
  }
  uint32_t phase = 0;
  bool ok = true;
  for (int step = 0; step < nchunks; ++step) {
    const int jc = FWD ? step : nchunks - 1 - step;
    const size_t slab = (size_t)(off[s] + jc) * H + h;
    if (tid == 0 && step + 1 < nchunks) {  // the next chunk's operands into L2
      const size_t sp = FWD ? slab + H : slab - H;
      prefetch_l2(B1g + sp * C * D, C * D * 4);
      prefetch_l2(B2g + sp * C * D, C * D * 4);
      prefetch_l2(Xg + sp * C * D, C * D * 4);
      if (!FWD) prefetch_l2(Rg + sp * D * D, D * D * 4);
    }
    // R^T and V1^T (or U~^T) of this thread's row (read in steps 2 and 4), issued first
    float rr[64], v1[32];
#pragma unroll
    for (int u = 0; u < 64; ++u) rr[u] = FWD ? 0.f : Rg[(slab * D + 64 * hh + u) * D + j];
#pragma unroll
    for (int u = 0; u < 32; ++u) v1[u] = Xg[(slab * C + 32 * hh + u) * D + j];
    // (1) the terms of the two [token][c] operands (16-byte loads) into their B tiles
    {
      const float *Kd = B1g + slab * C * D, *W = B2g + slab * C * D;
      float4 xk[8], xw[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        xk[m] = *reinterpret_cast<const float4 *>(Kd + 4 * (tid + bst::NT * m));
        xw[m] = *reinterpret_cast<const float4 *>(W + 4 * (tid + bst::NT * m));
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int e = tid + bst::NT * m;
        const uint32_t o = sw128_off(e >> 5, 4 * (e & 31), 64);
        uint32_t wa[3], wb[3];
        bst_split(xk[m].x, xk[m].y, wa);
        bst_split(xk[m].z, xk[m].w, wb);
#pragma unroll
        for (int t = 0; t < 3; ++t)
          *reinterpret_cast<uint2 *>(sm + bst::SB1 + t * 16384 + o) = make_uint2(wa[t], wb[t]);
        bst_split(xw[m].x, xw[m].y, wa);
        bst_split(xw[m].z, xw[m].w, wb);
#pragma unroll
        for (int t = 0; t < 3; ++t)
          *reinterpret_cast<uint2 *>(sm + bst::SB2 + t * 16384 + o) = make_uint2(wa[t], wb[t]);
      }
    }
    // (2) dS' (the state leaving chunk jc) out; its terms into the A tile; the accumulator
    //     pre-loaded with e^{G_C} dS' + R
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int cb = 64 * hh + 32 * half;  // first key column of this half
      float v[32], dd[32];
      tmem_ld32(trow + bst::TS + cb, v);
#pragma unroll
      for (int u = 0; u < 32; u += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(Dg + slab * D + cb + u);
        dd[u] = x.x, dd[u + 1] = x.y, dd[u + 2] = x.z, dd[u + 3] = x.w;
      }
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 32; ++u) Sb[(slab * D + cb + u) * D + j] = v[u];
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t w[3][4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          uint32_t t3[3];
          bst_split(v[8 * q8 + 2 * p], v[8 * q8 + 2 * p + 1], t3);
          w[0][p] = t3[0], w[1][p] = t3[1], w[2][p] = t3[2];
        }
        const uint32_t o = sw128_chunk(j, (cb >> 3) + q8, 128);
#pragma unroll
        for (int t = 0; t < 3; ++t)
          *reinterpret_cast<uint4 *>(sm + bst::SA + t * 32768 + o) =
              make_uint4(w[t][0], w[t][1], w[t][2], w[t][3]);
      }
#pragma unroll
      for (int u = 0; u < 32; ++u) v[u] = FWD ? dd[u] * v[u] : fmaf(dd[u], v[u], rr[32 * half + u]);
      tmem_st32(trow + bst::TS + cb, v);
    }
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
    ok = named_bar_and(1, bst::NT, ok);
    tc_fence_after();
    if (!ok) break;
    // (3) dU^T = dS'^T K_d^T (six products of terms per K step)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int a = 0; a < 3; ++a)
#pragma unroll
          for (int b = 0; a + b < 3; ++b)
            mma_bf16(tb + bst::TU, desc_kmajor(sb + bst::SA + a * 32768, 128, kk),
                     desc_kmajor(sb + bst::SB1 + b * 16384, 64, kk), id,
                     (kk > 0 || a > 0 || b > 0) ? 1u : 0u);
      mma_commit(&bar_mma);
    }
    ok = mbar_wait(&bar_mma, phase) && ok;
    phase ^= 1u;
    tc_fence_after();
    // (4) dU = dU^T + V1^T out; its terms into the A tile (K = the chunk's 64 tokens)
    if (ok) {
      float u32[32];
      tmem_ld32(trow + bst::TU + 32 * hh, u32);
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        u32[u] = FWD ? v1[u] - u32[u] : u32[u] + v1[u];
        Ub[(slab * C + 32 * hh + u) * D + j] = u32[u];
      }
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t w[3][4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          uint32_t t3[3];
          bst_split(u32[8 * q8 + 2 * p], u32[8 * q8 + 2 * p + 1], t3);
          w[0][p] = t3[0], w[1][p] = t3[1], w[2][p] = t3[2];
        }
        const uint32_t o = sw128_chunk(j, 4 * hh + q8, 128);
#pragma unroll
        for (int t = 0; t < 3; ++t)
          *reinterpret_cast<uint4 *>(sm + bst::SA + t * 16384 + o) =
              make_uint4(w[t][0], w[t][1], w[t][2], w[t][3]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    ok = named_bar_and(1, bst::NT, ok);
    tc_fence_after();
    if (!ok) break;
    // (5) dS^T = (e^{G_C} dS'^T + R^T) - dU^T W
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 128, 0, 1) | (FWD ? 0u : kNegateA);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int a = 0; a < 3; ++a)
#pragma unroll
          for (int b = 0; a + b < 3; ++b)
            mma_bf16(tb + bst::TS, desc_kmajor(sb + bst::SA + a * 16384, 128, kk),
                     desc_mnmajor(sb + bst::SB2 + b * 16384, 64, kk), id, 1u);
      mma_commit(&bar_mma);
    }
    ok = mbar_wait(&bar_mma, phase) && ok;
    phase ^= 1u;
    tc_fence_after();
    ok = named_bar_and(1, bst::NT, ok);
    if (!ok) break;
  }
  if (ok && S_last) {  // the state after the last step
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[32];
      tmem_ld32(trow + bst::TS + 64 * hh + 32 * half, v);
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 32; ++u) S_last[st0 + (size_t)(64 * hh + 32 * half + u) * D + j] = v[u];
    }
  }
  if (!ok && lane == 0) atomicOr(&g_bwd_err, kErrTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}


// ---------------------------------------------------------------------------
// Batched 64-row GEMM over (chunk, head) slabs:
//   C = mask( sum_i alpha_i op(A_i) op(B_i) ),  C: [64, N] row-major,
// op(A)(m, k) = a_t ? A[k * lda + m] : A[m * lda + k],
// op(B)(k, n) = b_t ? B[n * ldb + k] : B[k * ldb + n].
// mask 0: none; 1: keep n <= m; 2: keep n < m.
struct GemmTerm {
  const float *A, *B;
  size_t sA, sB;  // per-slab strides (floats)
  int lda, ldb, a_t, b_t, K;
  float alpha;
};
struct GemmArgs {
  GemmTerm t[3];
  int nterms;
  float *Cm;
  size_t sC;
  int mask;
  // multi-product kernel (NPROD = 2 or 3): t[p] -> Cm / Cm2 / Cm3 with strides sC / sC2 / sC3
  // (no mask), their K tiles in turn; with two products and dot, also
  // dot[n] = sum_k op(B_0)[k][n] op(B_1)[k][n] per slab (both B stored n-major)
  float *Cm2, *Cm3, *dot;
  size_t sC2, sC3;
};

// On the tensor cores, at fp32-level accuracy: as
// C^T[n][m] = sum_i alpha_i op(B_i)^T op(A_i)^T, an M = 128 (n), N = 64 (m) tcgen05 product per
// 64-deep K tile (for N = 64 the accumulator rows 64..127 are computed from rows of the op(B)^T
// tile that are never written, and never read back). Each fp32 operand value v enters as three
// bf16 terms, v0 = bf16(v), v1 = bf16(v - v0), v2 = bf16(v - v0 - v1) (the differences are
// exact in fp32), and the six products of terms a + b <= 2 are accumulated in fp32 in tensor
// memory (what is dropped is below 2^-24 of the product). Both operands are staged as they lie in memory: op(B)^T is
// K-major when B is stored n-major (b_t) and MN-major otherwise, op(A)^T K-major when A is
// stored m-major (!a_t) and MN-major otherwise. The mask is applied as C is written. One CTA
// (256 threads) per (chunk, head), three per SM; thread 0 issues the 24 MMAs of a tile, the
// tiles of a CTA in turn. The multi-product instantiations (NPROD = 2, 3) compute two or three
// products of equal depth into their own accumulators, their K tiles in turn, at two CTAs per
// SM: with the per-row sums of GemmArgs::dot they need more than the 80 registers a thread of
// three CTAs per SM.
namespace bgt {
constexpr int NT = 256;
constexpr uint32_t TA = 128 * 64 * 2;  // one bf16 term of op(B)^T: 128 x 64
constexpr uint32_t TB = 64 * 64 * 2;   // one bf16 term of op(A)^T: 64 x 64
constexpr uint32_t SB = 3 * TA;        // the B terms after the three A terms
constexpr uint32_t DYN = 3 * TA + 3 * TB + 1024;
}  // namespace bgt

// (a, b) -> the bf16x2 words of the pair's three terms
__device__ __forceinline__ void split3_pair(float a, float b, uint32_t (&w)[3]) {
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

template <int N, int NPROD = 1>
__global__ void __launch_bounds__(bgt::NT, NPROD > 1 ? 2 : 3)
    kda_bwd_gemm_tc(GemmArgs g, int H, const ChunkMeta *__restrict__ meta) {
  using namespace tc;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_dot[N];  // two products with dot: the row sums, tile by tile
  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (meta->invalid || ci >= meta->total_chunks) return;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const size_t slab = (size_t)ci * H + h;
  // one 64-column accumulator per product (an allocation is a power of two)
  const uint32_t ncols = NPROD == 1 ? 64 : (NPROD == 2 ? 128 : 256);
  if (warp == 0) {
    tmem_alloc(&tmem_base, ncols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  const int nt0 = g.t[0].K / 64;
  int ntiles = 0;
  for (int q = 0; q < g.nterms; ++q) ntiles += g.t[q].K / 64;
  // A CTA holds one K tile of operands in flight (registers, then shared memory), so with more
  // than one tile the operand slabs of every term are prefetched into L2 at the start: later
  // tiles then load from L2 (2.81 -> 2.72 ms for the backward call). Each range lies within
  // its term's per-slab stride.
  if (ntiles > 1 && tid < 2 * g.nterms) {
    const GemmTerm &pt = g.t[tid >> 1];
    const float *base = (tid & 1) ? pt.B + slab * pt.sB : pt.A + slab * pt.sA;
    const uint32_t bytes = (uint32_t)(((tid & 1) ? pt.sB : pt.sA) * 4);
    for (uint32_t o = 0; o < bytes; o += 32768)
      prefetch_l2(reinterpret_cast<const char *>(base) + o, min(32768u, bytes - o));
  }
  auto put3 = [&](uint32_t base, uint32_t term_bytes, uint32_t off, const float4 &v) {
    uint32_t wa[3], wb[3];
    split3_pair(v.x, v.y, wa);
    split3_pair(v.z, v.w, wb);
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<uint2 *>(sm + base + t * term_bytes + off) = make_uint2(wa[t], wb[t]);
  };
  bool ok = true;
  for (int i = 0; i < ntiles; ++i) {
    // several products: their tiles in turn (equal depths); else the first term's, then the
    // second's
    const int term = NPROD > 1 ? i % NPROD : (i < nt0 ? 0 : 1);
    const int kt = NPROD > 1 ? i / NPROD : (i < nt0 ? i : i - nt0);
    const GemmTerm &t = g.t[term];
    const int k0 = kt * 64;
    const float *A = t.A + slab * t.sA, *B = t.B + slab * t.sB;
    // this tile's operands into registers (16-byte loads along each operand's contiguous axis)
    constexpr int NB = N / 16, NQ = N / 4;  // float4s of op(B)^T per thread, per row of n
    float4 vb[NB], va[4];
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      const int e = tid + bgt::NT * r;
      vb[r] = t.b_t ? *reinterpret_cast<const float4 *>(B + (size_t)(e >> 4) * t.ldb + k0 +
                                                         4 * (e & 15))           // (n, k)
                    : *reinterpret_cast<const float4 *>(B + (size_t)(k0 + e / NQ) * t.ldb +
                                                         4 * (e % NQ));          // (k, n)
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int e = tid + bgt::NT * r;
      const float4 v = t.a_t ? *reinterpret_cast<const float4 *>(
                                   A + (size_t)(k0 + (e >> 4)) * t.lda + 4 * (e & 15))  // (k, m)
                             : *reinterpret_cast<const float4 *>(
                                   A + (size_t)(e >> 4) * t.lda + k0 + 4 * (e & 15));   // (m, k)
      va[r] = make_float4(t.alpha * v.x, t.alpha * v.y, t.alpha * v.z, t.alpha * v.w);
    }
    // the previous tile's products are done with the shared-memory operands
    if (i > 0 && !mbar_wait(&bar_mma, (i - 1) & 1)) ok = false;
    tc_fence_after();
    const bool dot = NPROD == 2 && g.dot && term == 1;
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      const int e = tid + bgt::NT * r;
      const uint32_t o =
          t.b_t ? sw128_off(e >> 4, 4 * (e & 15), 128) : sw128_off(e / NQ, 4 * (e % NQ), 64);
      if (dot) {
        // the first term's B values at these positions, as their three terms still in shared
        // memory (written by this thread; their sum is the fp32 value to within 2^-27 of it)
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int tt = 0; tt < 3; ++tt) {
          const uint2 w = *reinterpret_cast<const uint2 *>(sm + tt * bgt::TA + o);
          const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.x));
          const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w.y));
          x[0] += lo.x, x[1] += lo.y, x[2] += hi.x, x[3] += hi.y;
        }
        float d = x[0] * vb[r].x;
        d = fmaf(x[1], vb[r].y, d);
        d = fmaf(x[2], vb[r].z, d);
        d = fmaf(x[3], vb[r].w, d);
#pragma unroll
        for (int sh = 1; sh < 16; sh <<= 1) d += __shfl_xor_sync(0xffffffffu, d, sh);
        // row e >> 4 is held by 16 consecutive lanes; the first of them adds the row's sum
        if ((tid & 15) == 0) s_dot[e >> 4] = (kt == 0 ? 0.f : s_dot[e >> 4]) + d;
      }
      put3(0, bgt::TA, o, vb[r]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int e = tid + bgt::NT * r;
      put3(bgt::SB, bgt::TB, sw128_off(e >> 4, 4 * (e & 15), 64), va[r]);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
      const uint32_t id = idesc_bf16(128, 64, t.b_t ? 0 : 1, t.a_t ? 1 : 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int a = 0; a < 3; ++a)
#pragma unroll
          for (int b = 0; a + b < 3; ++b) {
            const uint32_t ta = sb + a * bgt::TA, tbb = sb + bgt::SB + b * bgt::TB;
            const uint64_t ad = t.b_t ? desc_kmajor(ta, 128, kk) : desc_mnmajor(ta, 64, kk);
            const uint64_t bd = t.a_t ? desc_mnmajor(tbb, 64, kk) : desc_kmajor(tbb, 64, kk);
            const bool first = NPROD > 1 ? kt == 0 : i == 0;
            mma_bf16(tb + (NPROD > 1 ? 64u * term : 0u), ad, bd, id,
                     (!first || kk > 0 || a > 0 || b > 0) ? 1u : 0u);
          }
      mma_commit(&bar_mma);
    }
  }
  if (!mbar_wait(&bar_mma, (ntiles - 1) & 1)) ok = false;
  tc_fence_after();
  // C[m][n]: lane quadrant warp % 4 holds n = 32 (warp % 4) + lane, warp / 4 the half of m
  if (ok && (warp & 3) * 32 < N) {
#pragma unroll
    for (int acc = 0; acc < NPROD; ++acc) {
      float v[32];
      tmem_ld32(tmem_addr(tb, (warp & 3) * 32, 64 * acc + 32 * (warp >> 2)), v);
      tmem_wait_ld();
      float *Cm = acc == 0 ? g.Cm + slab * g.sC
                           : (acc == 1 ? g.Cm2 + slab * g.sC2 : g.Cm3 + slab * g.sC3);
      const int n = (warp & 3) * 32 + lane;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int m = 32 * (warp >> 2) + j;
        const bool keep = g.mask == 0 || (g.mask == 1 ? n <= m : n < m);
        Cm[(size_t)m * N + n] = keep ? v[j] : 0.f;
      }
    }
  } else if (!ok && lane == 0) {
    atomicOr(&g_bwd_err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (NPROD == 2 && g.dot && tid < N) g.dot[slab * N + tid] = s_dot[tid];
  if (warp == 0) tmem_dealloc(tb, ncols);
}

// ---------------------------------------------------------------------------
// [X1 | X2] = T^T [Y1 | Y2] in place, T = (I + A)^-1: back substitution on the
// unit upper-triangular (I + A)^T, X_r = Y_r - sum_{s > r} A[s][r] X_s.
// One thread per column (N1 + N2 <= 256), columns staged in shared memory.
template <int N1, int N2>
__global__ void __launch_bounds__(256) kda_bwd_solve(const float *__restrict__ Ag,
                                                     float *__restrict__ Y1,
                                                     float *__restrict__ Y2, int H,
                                                     const ChunkMeta *__restrict__ meta) {
  // A is held transposed (row r of sAt = column r of A, padded to 68 floats so every row starts
  // on a 16-byte boundary): row r's dot product reads 16-byte vectors. Y is held unpadded.
  constexpr int NC = N1 + N2, LA = C + 4;
  extern __shared__ __align__(16) float smem[];
  float *sAt = smem;         // [C][LA]  sAt[c][r] = A[r][c]
  float *sY = sAt + C * LA;  // [C][NC]
  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (meta->invalid || ci >= meta->total_chunks) return;
  const size_t slab = (size_t)ci * H + h;
  float *y1 = Y1 + slab * C * N1, *y2 = Y2 + slab * C * N2;
  {  // 16-byte loads, all issued before their stores. A: lane = row, so that the transposed
     // stores of a warp fall in different banks
    constexpr int NA = C * C / 4 / 256, NY1 = C * N1 / 4 / 256, NY2 = C * N2 / 4 / 256;
    float4 ra[NA], r1[NY1], r2[NY2];
    const int ar = tid % C, ac = 4 * (tid / C);  // row and first column of this thread's A loads
#pragma unroll
    for (int m = 0; m < NA; ++m)
      ra[m] = *reinterpret_cast<const float4 *>(Ag + slab * C * C + ar * C + ac + 16 * m);
#pragma unroll
    for (int m = 0; m < NY1; ++m) r1[m] = *reinterpret_cast<const float4 *>(y1 + 4 * (tid + 256 * m));
#pragma unroll
    for (int m = 0; m < NY2; ++m) r2[m] = *reinterpret_cast<const float4 *>(y2 + 4 * (tid + 256 * m));
#pragma unroll
    for (int m = 0; m < NA; ++m) {
      const int c = ac + 16 * m;
      sAt[(c + 0) * LA + ar] = ra[m].x; sAt[(c + 1) * LA + ar] = ra[m].y;
      sAt[(c + 2) * LA + ar] = ra[m].z; sAt[(c + 3) * LA + ar] = ra[m].w;
    }
#pragma unroll
    for (int m = 0; m < NY1; ++m) {
      const int e = 4 * (tid + 256 * m), r = e / N1, c = e % N1;
      *reinterpret_cast<float4 *>(sY + r * NC + c) = r1[m];
    }
#pragma unroll
    for (int m = 0; m < NY2; ++m) {
      const int e = 4 * (tid + 256 * m), r = e / N2, c = e % N2;
      *reinterpret_cast<float4 *>(sY + r * NC + N1 + c) = r2[m];
    }
  }
  __syncthreads();
  // (I + A)^T X = Y, back substitution: one thread per column, the column in registers
  // (indices fixed at compile time), each row's dot product in four partial sums (row s into
  // sum s mod 4), column r of A read as 16-byte vectors of sAt's row r
  if (tid < NC) {
    float *col = sY + tid;
    float x[C];
#pragma unroll
    for (int r = 0; r < C; ++r) x[r] = col[r * NC];
#pragma unroll
    for (int r = C - 2; r >= 0; --r) {
      const float *At = sAt + r * LA;
      float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s4 = (r + 1) & ~3; s4 < C; s4 += 4) {
        const float4 a4 = *reinterpret_cast<const float4 *>(At + s4);
        if (s4 + 0 > r) p[0] = fmaf(a4.x, x[s4 + 0], p[0]);
        if (s4 + 1 > r) p[1] = fmaf(a4.y, x[s4 + 1], p[1]);
        if (s4 + 2 > r) p[2] = fmaf(a4.z, x[s4 + 2], p[2]);
        if (s4 + 3 > r) p[3] = fmaf(a4.w, x[s4 + 3], p[3]);
      }
      x[r] -= (p[0] + p[1]) + (p[2] + p[3]);
    }
#pragma unroll
    for (int r = 0; r < C - 1; ++r) col[r * NC] = x[r];
  }
  __syncthreads();
#pragma unroll 4
  for (int e = 4 * tid; e < C * N1; e += 1024) {
    const int r = e / N1, c = e % N1;
    *reinterpret_cast<float4 *>(y1 + e) = *reinterpret_cast<const float4 *>(sY + r * NC + c);
  }
#pragma unroll 4
  for (int e = 4 * tid; e < C * N2; e += 1024) {
    const int r = e / N2, c = e % N2;
    *reinterpret_cast<float4 *>(y2 + e) = *reinterpret_cast<const float4 *>(sY + r * NC + N1 + c);
  }
}

// ---------------------------------------------------------------------------
// Finishing kernel, one block per (chunk, head): from the chunk-level cotangents
// to the token gradients. Warp w handles token rows w, w + 8, ...; lane l the NI = dk / 32
// consecutive key channels NI l .. NI l + NI - 1 and the NJ = dv / 32 consecutive value
// channels NJ l .., so that every global access of a row is one 8- or 16-byte vector. The
// per-channel rows in shared memory hold channel c at position (c % NI) 32 + c / NI: the
// row-wise accesses (lane l, i) and the column-wise serial sums (thread = position) are then
// both free of bank conflicts.
// fp32 loads: the finishing kernel is the last reader of everything it loads, so they carry the
// last-use cache hint (2.84 -> 2.82 ms for a call that starts with a cold L2; no change when
// calls run back to back)
template <int N>
__device__ __forceinline__ void ldv(const float *p, float (&v)[N]) {
  if constexpr (N == 4) {
    const float4 a = __ldlu(reinterpret_cast<const float4 *>(p));
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
  } else {
    const float2 a = __ldlu(reinterpret_cast<const float2 *>(p));
    v[0] = a.x, v[1] = a.y;
  }
}
template <int N>
__device__ __forceinline__ void ldv(const __nv_bfloat16 *p, float (&v)[N]) {
  if constexpr (N == 4) {
    const uint2 a = *reinterpret_cast<const uint2 *>(p);
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a.x));
    const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a.y));
    v[0] = x.x, v[1] = x.y, v[2] = y.x, v[3] = y.y;
  } else {
    const uint32_t a = *reinterpret_cast<const uint32_t *>(p);
    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a));
    v[0] = x.x, v[1] = x.y;
  }
}
template <int N>
__device__ __forceinline__ void stv(float *p, const float (&v)[N]) {
  if constexpr (N == 4)
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
  else
    *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
}
template <int N>
__device__ __forceinline__ void stv(__nv_bfloat16 *p, const float (&v)[N]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  if constexpr (N == 4) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    *reinterpret_cast<uint2 *>(p) =
        make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
  } else {
    *reinterpret_cast<uint32_t *>(p) = *reinterpret_cast<const uint32_t *>(&a);
  }
}

template <int DK, int DV, typename Tio>
__global__ void __launch_bounds__(256, 3) kda_bwd_finish(
    const Tio *__restrict__ q, const Tio *__restrict__ k, const Tio *__restrict__ v,
    const Tio *__restrict__ la, const Tio *__restrict__ beta, const Tio *__restrict__ gate,
    const Tio *__restrict__ d_out, Tio *__restrict__ dq, Tio *__restrict__ dk, Tio *__restrict__ dv, Tio *__restrict__ dla,
    Tio *__restrict__ dbeta, Tio *__restrict__ dgate, const int32_t *__restrict__ cu, int n_seq,
    int64_t fixed_len, int H, float scale, unsigned flags, const ChunkMeta *__restrict__ meta,
    const int *__restrict__ off, const float *__restrict__ Yg, const float *__restrict__ dBkg,
    const float *__restrict__ dBvg, const float *__restrict__ dKhg,
    const float *__restrict__ dQtg, const float *__restrict__ dKdg,
    const float *__restrict__ dDg, const float *__restrict__ Og) {
  constexpr int LK = DK + 1, NI = DK / 32, NJ = DV / 32;
  extern __shared__ float smem[];
  float *sG = smem;             // [C][LK]  running log-decay G (by position)
  float *sdG = sG + C * LK;     // [C][LK]  dL/dG (by position)
  float *sB = sdG + C * LK;     // [C]      beta
  float *sDc = sB + C;          // [DK]     e^{G_C} (by position)
  float *sdD = sDc + DK;        // [DK]     dL/d e^{G_C} from the state hand-off (by position)
  float *sGCp = sdD + DK;       // [8][DK]  per-warp partial dL/dG_C (by position)
  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (meta->invalid || ci >= meta->total_chunks) return;
  int s, len;
  int64_t t0;
  chunk_rows(cu, fixed_len, n_seq, off, ci, &s, &t0, &len);
  const size_t slab = (size_t)ci * H + h;
  const bool l2 = (flags & KDA_QK_L2NORM) != 0;
  auto pos = [](int c) { return (c % NI) * 32 + c / NI; };   // channel -> position
  auto chan = [](int p) { return NI * (p & 31) + (p >> 5); };  // position -> channel

  const bool logits = (flags & KDA_GATE_LOGITS) != 0;
  if (tid < C) sB[tid] = tid < len ? prep_beta(bf(beta[(size_t)(t0 + tid) * H + h]), flags) : 0.f;
  // log_alpha of the chunk into sG by 8-element vector loads of all threads (0 on padded rows),
  // so that the serial running sum below reads shared memory only
  {
    constexpr int NV = C * DK / 8 / 256;
    float lv[NV][8];
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int e = 8 * (tid + 256 * m), r = e / DK, c = e % DK;
      if (r < len) {
        load8(la + ((size_t)(t0 + r) * H + h) * DK + c, lv[m]);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) lv[m][u] = 0.f;
      }
    }
#pragma unroll
    for (int m = 0; m < NV; ++m) {
      const int e = 8 * (tid + 256 * m), r = e / DK, c = e % DK;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        sG[r * LK + pos(c + u)] = r < len ? prep_log_alpha(lv[m][u], flags) : 0.f;
    }
  }
  // dL/d e^{G_C}[c] = sum_j dS'[c][j] S[c][j], from the paired dK_d / dW products
  if (tid < DK) sdD[pos(tid)] = dDg[slab * DK + tid];
  __syncthreads();
  if (tid < DK) {  // position tid
    float G = 0.f;
    for (int r = 0; r < C; ++r) {
      G += sG[r * LK + tid];
      sG[r * LK + tid] = G;
    }
    sDc[tid] = expf(G);
  }
  __syncthreads();

  float gcp[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) gcp[i] = 0.f;
  for (int r = warp; r < C; r += 8) {
    if (r >= len) {
#pragma unroll
      for (int i = 0; i < NI; ++i) sdG[r * LK + 32 * i + lane] = 0.f;
      continue;
    }
    const size_t tok = (size_t)(t0 + r) * H + h;
    const float b = sB[r];
    const size_t rowk = (slab * C + r) * DK + NI * lane;
    float kn[NI], qn[NI], y[NI], y2[NI], dKh[NI], dQt[NI], dKd[NI];
    ldv(k + tok * DK + NI * lane, kn);
    ldv(q + tok * DK + NI * lane, qn);
    ldv(Yg + rowk, y);
    ldv(dBkg + rowk, y2);
    ldv(dKhg + rowk, dKh);
    ldv(dQtg + rowk, dQt);
    ldv(dKdg + rowk, dKd);
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      sk = fmaf(kn[i], kn[i], sk);
      sq = fmaf(qn[i], qn[i], sq);
    }
    float rk = 1.f, rq = 1.f;
    if (l2) {
      rk = rsqrtf(wsum(sk) + kL2Eps);
      rq = rsqrtf(wsum(sq) + kL2Eps);
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        kn[i] *= rk;
        qn[i] *= rq;
      }
    }
    float dkn[NI], dqn[NI], dbk = 0.f;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int p = 32 * i + lane;
      const float G = sG[r * LK + p], eP = expf(G), eN = expf(-G), Dc = sDc[p];
      const float Kt = kn[i] * eP, Kh = kn[i] * eN, Qt = qn[i] * eP, Kd = Kh * Dc;
      const float yy = y[i] + y2[i];
      const float dKt = b * yy;
      dkn[i] = dKt * eP + dKh[i] * eN + dKd[i] * eN * Dc;
      dqn[i] = dQt[i] * eP;
      sdG[r * LK + p] = dKt * Kt - dKh[i] * Kh + dQt[i] * Qt - dKd[i] * Kd;
      gcp[i] = fmaf(dKd[i], Kd, gcp[i]);
      dbk = fmaf(Kt, yy, dbk);
    }
    if (l2) {  // d(x / |x|) : dx = r (dn - n (n . dn))
      float pk = 0.f, pq = 0.f;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        pk = fmaf(kn[i], dkn[i], pk);
        pq = fmaf(qn[i], dqn[i], pq);
      }
      pk = wsum(pk);
      pq = wsum(pq);
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        dkn[i] = rk * (dkn[i] - kn[i] * pk);
        dqn[i] = rq * (dqn[i] - qn[i] * pq);
      }
    }
    stv(dk + tok * DK + NI * lane, dkn);
    stv(dq + tok * DK + NI * lane, dqn);
    const size_t rowv = (slab * C + r) * DV + NJ * lane;
    float vv[NJ], g[NJ], dvv[NJ];
    ldv(v + tok * DV + NJ * lane, vv);
    ldv(dBvg + rowv, g);
    float dbv = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      dbv = fmaf(vv[j], g[j], dbv);
      dvv[j] = b * g[j];
    }
    stv(dv + tok * DV + NJ * lane, dvv);
    if (dgate) {
      float dov[NJ], ov[NJ], dg[NJ];
      ldv(d_out + tok * DV + NJ * lane, dov);
      ldv(Og + rowv, ov);
#pragma unroll
      for (int j = 0; j < NJ; ++j) dg[j] = scale * dov[j] * ov[j];
      if (logits) {  // d sigmoid(x) / dx = s (1 - s)
        float gv[NJ];
        ldv(gate + tok * DV + NJ * lane, gv);
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const float gs = sigmoid_f(gv[j]);
          dg[j] *= gs * (1.f - gs);
        }
      }
      stv(dgate + tok * DV + NJ * lane, dg);
    }
    float db = wsum(dbk) + wsum(dbv);
    if (logits) db *= b * (1.f - b);
    if (lane == 0) dbeta[tok] = to_out<Tio>(db);
  }
#pragma unroll
  for (int i = 0; i < NI; ++i) sGCp[warp * DK + 32 * i + lane] = gcp[i];
  __syncthreads();
  if (tid < DK) {  // position tid, channel chan(tid)
    const int c = chan(tid);
    float dGC = sdD[tid] * sDc[tid];
#pragma unroll
    for (int w = 0; w < 8; ++w) dGC += sGCp[w * DK + tid];
    // G_r = sum_{s <= r} log_alpha_s and G_C = G_63: reverse cumulative sum
    float acc = 0.f;
    for (int r = C - 1; r >= 0; --r) {
      acc += sdG[r * LK + tid];
      if (r < len) {
        const size_t gi = ((size_t)(t0 + r) * H + h) * DK + c;
        float d = acc + dGC;
        if (logits) {  // log_alpha = max(-e^a, log 1/2): slope -e^a above the bound, 0 on it
          const float e = -expf(bf(la[gi]));
          d = e > kLogHalf ? d * e : 0.f;
        }
        dla[gi] = to_out<Tio>(d);
      }
    }
  }
}

template <int DK>
constexpr size_t bwd_finish_smem() {
  return sizeof(float) * (2 * C * (DK + 1) + C + 2 * DK + 8 * DK);
}

// ---------------------------------------------------------------------------
// workspace: the forward's SIMT chunk workspace, then the backward's buffers
struct BwdWs {
  ChunkWs fw;
  float *Kh, *Bk, *A, *Sb, *dSb, *R, *Ub, *O, *dO, *dU, *V1, *dP, *dQt, *dKd, *dW, *dM, *Y, *dKh;
  float *dD;  // [slab][dk] sum_j dS'[c][j] S[c][j]
};

// Per-slab buffer sizes of the backward's workspace (after the forward prep's part).
struct BwdSizes {
  size_t mk, mv, mc, ms, md;
  BwdSizes(int64_t T_total, int n_seq, int H, int dk, int dv) {
    const size_t per = ((size_t)(T_total / C) + (size_t)n_seq + 1) * H;
    mk = align_up(sizeof(float) * per * C * dk, 256);
    mv = align_up(sizeof(float) * per * C * dv, 256);
    mc = align_up(sizeof(float) * per * C * C, 256);
    ms = align_up(sizeof(float) * per * dk * dv, 256);
    md = align_up(sizeof(float) * per * dk, 256);
  }
  // R, V1 and dO are last read before the side stream joins back; dK_d, dW, dD, Y, dK^ and dA
  // are first written after it, so the two sets share one region
  size_t early() const { return ms + 2 * mv; }
  size_t late() const { return 4 * mk + mc + md; }
  size_t shared() const { return early() > late() ? early() : late(); }
  size_t bytes() const { return 3 * mk + 3 * mv + 2 * mc + 2 * ms + shared(); }
};

size_t bwd_extra_bytes(int64_t T_total, int n_seq, int H, int dk, int dv) {
  return BwdSizes(T_total, n_seq, H, dk, dv).bytes();
}

BwdWs bwd_ws_carve(void *ws, int64_t T_total, int n_seq, int H, int dk, int dv) {
  BwdWs w;
  w.fw = chunk_ws_carve(ws, T_total, n_seq, H, dk, dv);
  char *p = (char *)ws + chunk_ws_bytes(T_total, n_seq, H, dk, dv);
  const BwdSizes z(T_total, n_seq, H, dk, dv);
  auto take = [&](size_t n) {
    float *r = (float *)p;
    p += n;
    return r;
  };
  // live from their first write to the finishing kernel
  w.Kh = take(z.mk); w.Bk = take(z.mk); w.dQt = take(z.mk);
  w.Ub = take(z.mv); w.O = take(z.mv); w.dU = take(z.mv);
  w.A = take(z.mc); w.dP = take(z.mc);
  w.Sb = take(z.ms); w.dSb = take(z.ms);
  // the shared region: first R, V1, dO, then dK_d, dW, Y, dK^, dA, dD
  char *const sh = p;
  w.R = take(z.ms); w.V1 = take(z.mv); w.dO = take(z.mv);
  p = sh;
  w.dKd = take(z.mk); w.dW = take(z.mk); w.Y = take(z.mk); w.dKh = take(z.mk); w.dM = take(z.mc);
  w.dD = take(z.md);
  return w;
}

GemmTerm term(const float *A, size_t sA, int lda, int a_t, const float *B, size_t sB, int ldb,
              int b_t, int K, float alpha) {
  GemmTerm t;
  t.A = A; t.sA = sA; t.lda = lda; t.a_t = a_t;
  t.B = B; t.sB = sB; t.ldb = ldb; t.b_t = b_t;
  t.K = K; t.alpha = alpha;
  return t;
}

template <int N>
cudaError_t gemm(const GemmTerm &t0, const GemmTerm *t1, float *Cm, int mask, int mc, int H,
                 const ChunkMeta *meta, cudaStream_t st, size_t sC = 0) {
  GemmArgs g;
  g.t[0] = t0;
  g.t[1] = t1 ? *t1 : t0;
  g.t[2] = t0;
  g.nterms = t1 ? 2 : 1;
  g.Cm = Cm;
  g.sC = sC ? sC : (size_t)C * N;
  g.mask = mask;
  g.Cm2 = g.Cm3 = nullptr;
  g.sC2 = g.sC3 = 0;
  g.dot = nullptr;
  // every contraction depth is C, dk or dv: a multiple of the 64-deep tile
  if (t0.K % 64 != 0 || (t1 && t1->K % 64 != 0)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_gemm_tc<N>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bgt::DYN);
  if (e != cudaSuccess) return e;
  kda_bwd_gemm_tc<N><<<dim3(mc, H), bgt::NT, bgt::DYN, st>>>(g, H, meta);
  return cudaGetLastError();
}

// NP (2 or 3) products of one launch, C_p = op(A_p) op(B_p) with per-slab stride sC_p (equal
// depths, no mask); with two products and dot, also dot[n] = sum_k op(B_0)[k][n] op(B_1)[k][n]
// (both B stored n-major).
template <int N, int NP>
cudaError_t gemm_products(const GemmTerm (&t)[NP], float *const (&Cs)[NP],
                          const size_t (&sCs)[NP], float *dot, int mc, int H,
                          const ChunkMeta *meta, cudaStream_t st) {
  static_assert(NP == 2 || NP == 3, "two or three products");
  GemmArgs g;
  for (int p = 0; p < 3; ++p) g.t[p] = t[p < NP ? p : 0];
  g.nterms = NP;
  g.Cm = Cs[0];
  g.sC = sCs[0];
  g.Cm2 = Cs[1];
  g.sC2 = sCs[1];
  g.Cm3 = NP == 3 ? Cs[NP - 1] : nullptr;
  g.sC3 = NP == 3 ? sCs[NP - 1] : 0;
  g.mask = 0;
  g.dot = dot;
  if (t[0].K % 64 != 0) return cudaErrorInvalidValue;
  for (int p = 1; p < NP; ++p)
    if (t[p].K != t[0].K) return cudaErrorInvalidValue;
  if (dot && !(NP == 2 && t[0].b_t && t[1].b_t && t[0].ldb == t[1].ldb))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_gemm_tc<N, NP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, bgt::DYN);
  if (e != cudaSuccess) return e;
  kda_bwd_gemm_tc<N, NP><<<dim3(mc, H), bgt::NT, bgt::DYN, st>>>(g, H, meta);
  return cudaGetLastError();
}

#define KDA_TRY(x)              \
  do {                          \
    e = (x);                    \
    if (e != cudaSuccess) return e; \
  } while (0)

// The prep, both state passes and the products between them, on two streams (the schedule is
// drawn in bwd_t). `forked` is set once the side stream depends on st; the caller joins it back.
template <int DK, int DV, typename Tio>
cudaError_t mid_passes(const void *q, const void *k, const void *v, const void *la,
                       const void *beta, const void *gate, const float *S0, const void *d_out,
                       const float *dSf, float *dS0, const int32_t *cu, int n_seq, int64_t T_total,
                       int H, float scale, unsigned flags, kda_dtype dt, const BwdWs &w,
                       cudaStream_t st, cudaStream_t side, cudaEvent_t (&ev)[4], bool &forked) {
  const ChunkWs &fw = w.fw;
  const int mc = fw.max_chunks;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  cudaError_t e;
  KDA_TRY(cudaEventRecord(ev[0], st));  // the chunk table is in place
  KDA_TRY(cudaStreamWaitEvent(side, ev[0], 0));
  forked = true;
  // side: the gated output gradient (needs only the chunk table)
  kda_bwd_dO<DV, Tio><<<dim3(mc, H), 256, 0, side>>>((const Tio *)d_out, (const Tio *)gate, cu,
                                                     n_seq, fixed_len, H, scale, flags, fw.meta,
                                                     fw.seq_chunk_off, w.dO);
  KDA_TRY(cudaGetLastError());
  PrepSave ps;
  ps.Kh = w.Kh; ps.Bk = w.Bk; ps.A = w.A;
  KDA_TRY(launch_prep(q, k, v, la, beta, cu, n_seq, T_total, H, DK, DV, flags, dt, fw, true, st,
                      ps));
  KDA_TRY(cudaEventRecord(ev[1], st));  // the prep's outputs are in place
  // st: the forward replay saves S and U per chunk only; O comes from a batched GEMM below
  if (DK == 128 && DV == 128) {  // on the tensor cores
    KDA_TRY(cudaFuncSetAttribute(kda_bwd_state_tc<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bst::DYN));
    kda_bwd_state_tc<true><<<n_seq * H, bst::NT, bst::DYN, st>>>(
        S0, nullptr, cu, n_seq, fixed_len, H, fw.meta, fw.seq_chunk_off, fw.W, fw.Kd, fw.D, fw.U,
        nullptr, w.Sb, w.Ub);
    KDA_TRY(cudaGetLastError());
  } else {
    StateSave ss;
    ss.Sb = w.Sb; ss.Ub = w.Ub;
    KDA_TRY(launch_state_pass(0, flags, nullptr, nullptr, S0, nullptr, nullptr, nullptr, cu,
                              n_seq, T_total, H, DK, DV, scale, dt, fw, st, CkptOut(), ss));
  }
  const size_t sk = (size_t)C * DK, sv = (size_t)C * DV, scc = (size_t)C * C,
               ss2 = (size_t)DK * DV;
  // side: the state-independent parts of the reverse step: V1 = P^T dO, R = Q~^T dO (dk rows,
  // computed in 64-row halves), as the products of one launch that share dO
  KDA_TRY(cudaStreamWaitEvent(side, ev[1], 0));
  {
    const GemmTerm tv = term(fw.P, scc, C, 1, w.dO, sv, DV, 0, C, 1.f);
    const GemmTerm tr0 = term(fw.Q, sk, DK, 1, w.dO, sv, DV, 0, C, 1.f);
    if (DK == 2 * C) {
      const GemmTerm tp[3] = {tv, tr0, term(fw.Q + C, sk, DK, 1, w.dO, sv, DV, 0, C, 1.f)};
      float *const cp[3] = {w.V1, w.R, w.R + (size_t)C * DV};
      const size_t sp[3] = {sv, ss2, ss2};
      KDA_TRY((gemm_products<DV, 3>(tp, cp, sp, nullptr, mc, H, fw.meta, side)));
    } else {
      const GemmTerm tp[2] = {tv, tr0};
      float *const cp[2] = {w.V1, w.R};
      const size_t sp[2] = {sv, ss2};
      KDA_TRY((gemm_products<DV, 2>(tp, cp, sp, nullptr, mc, H, fw.meta, side)));
    }
  }
  KDA_TRY(cudaEventRecord(ev[2], side));  // dO, V1 and R are in place
  // side: the reverse state pass
  if (DK == 128 && DV == 128) {  // on the tensor cores
    KDA_TRY(cudaFuncSetAttribute(kda_bwd_state_tc<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bst::DYN));
    kda_bwd_state_tc<false><<<n_seq * H, bst::NT, bst::DYN, side>>>(
        dSf, dS0, cu, n_seq, fixed_len, H, fw.meta, fw.seq_chunk_off, fw.Kd, fw.W, fw.D, w.V1,
        w.R, w.dSb, w.dU);
    KDA_TRY(cudaGetLastError());
  } else {
    auto kern = kda_bwd_state<DK, DV>;
    constexpr size_t sm = bwd_state_smem<DK>();
    KDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
    kern<<<dim3(n_seq * H, DV / RBV), 256, sm, side>>>(dSf, dS0, cu, n_seq, fixed_len, H,
                                                       fw.meta, fw.seq_chunk_off, fw.W, fw.Kd,
                                                       fw.D, w.V1, w.R, w.dSb, w.dU);
    KDA_TRY(cudaGetLastError());
  }
  // st, after the replay and R: O = Q~ S + P U (pre-gate chunk output, for dg)
  KDA_TRY(cudaStreamWaitEvent(st, ev[2], 0));
  {
    GemmTerm t2 = term(fw.P, scc, C, 0, w.Ub, sv, DV, 0, C, 1.f);
    KDA_TRY(gemm<DV>(term(fw.Q, sk, DK, 0, w.Sb, ss2, DV, 0, DK, 1.f), &t2, w.O, 0, mc, H,
                     fw.meta, st));
  }
  // dP = lower(dO U^T)
  KDA_TRY(gemm<C>(term(w.dO, sv, DV, 0, w.Ub, sv, DV, 1, DV, 1.f), nullptr, w.dP, 1, mc, H,
                  fw.meta, st));
  // dQ~ = dO S^T + dP K^
  {
    GemmTerm t2 = term(w.dP, scc, C, 0, w.Kh, sk, DK, 0, C, 1.f);
    KDA_TRY(gemm<DK>(term(w.dO, sv, DV, 0, w.Sb, ss2, DV, 1, DV, 1.f), &t2, w.dQt, 0, mc, H,
                     fw.meta, st));
  }
  return cudaSuccess;
}

template <int DK, int DV, typename Tio>
cudaError_t bwd_t(const void *q, const void *k, const void *v, const void *la, const void *beta,
                  const void *gate, const float *S0, const void *d_out, const float *dSf,
                  void *dq, void *dk, void *dv, void *dla, void *dbeta, void *dgate, float *dS0,
                  const int32_t *cu, int n_seq, int64_t T_total, int H, float scale,
                  unsigned flags, kda_dtype dt, void *ws_raw, cudaStream_t st) {
  BwdWs w = bwd_ws_carve(ws_raw, T_total, n_seq, H, DK, DV);
  const ChunkWs &fw = w.fw;
  const int mc = fw.max_chunks;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  cudaError_t e;
  KDA_TRY(launch_chunk_table(cu, n_seq, T_total, fw, st));
  // The two state passes each run one CTA per (sequence, head) and do not depend on each other,
  // so they run side by side, together with the batched products around them:
  //   stream st:    prep -> forward replay ---------------------> O -> dP -> dQ~ -> (join) ...
  //   side stream:  dO ---------> V1, R (after the prep) -> reverse pass ------------^
  // The replay directly follows the prep in st, so its CTAs reach the SMs before those of the
  // products on the side stream; O waits for R, so the reverse pass (next in the side stream)
  // is placed before O's CTAs fill the GPU. Events fork the side stream off st and join it
  // back, also after a failed launch, so the call stays ordered on st (and can be captured).
  cudaStream_t side = nullptr;
  KDA_TRY(side_stream(&side));
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  for (cudaEvent_t &x : ev) {
    e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
    if (e != cudaSuccess) break;
  }
  bool forked = false;
  if (e == cudaSuccess) e = mid_passes<DK, DV, Tio>(q, k, v, la, beta, gate, S0, d_out, dSf, dS0,
                                                    cu, n_seq, T_total, H, scale, flags, dt, w,
                                                    st, side, ev, forked);
  if (forked) {  // join the side stream back into st
    cudaError_t j = cudaEventRecord(ev[3], side);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(st, ev[3], 0);
    if (e == cudaSuccess) e = j;
  }
  for (cudaEvent_t x : ev)
    if (x) cudaEventDestroy(x);
  if (e != cudaSuccess) return e;
  const size_t sk = (size_t)C * DK, sv = (size_t)C * DV, scc = (size_t)C * C,
               ss2 = (size_t)DK * DV;
  // dK_d = U dS'^T and dW = -dU S^T in one launch, with dD[c] = sum_j dS'[c][j] S[c][j] (the
  // gradient reaching e^{G_C} through the state hand-off)
  {
    const GemmTerm tp[2] = {term(w.Ub, sv, DV, 0, w.dSb, ss2, DV, 1, DV, 1.f),
                            term(w.dU, sv, DV, 0, w.Sb, ss2, DV, 1, DV, -1.f)};
    float *const cp[2] = {w.dKd, w.dW};
    const size_t sp[2] = {sk, sk};
    KDA_TRY((gemm_products<DK, 2>(tp, cp, sp, w.dD, mc, H, fw.meta, st)));
  }
  // [dB_k | dB_v] = T^T [dW | dU]   (in place)
  {
    auto kern = kda_bwd_solve<DK, DV>;
    constexpr size_t sm = sizeof(float) * (C * (C + 4) + C * (DK + DV));
    KDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
    kern<<<dim3(mc, H), 256, sm, st>>>(w.A, w.dW, w.dU, H, fw.meta);
    KDA_TRY(cudaGetLastError());
  }
  // dA = strict_lower(-dB_k W^T - dB_v U~^T)
  {
    GemmTerm t2 = term(w.dU, sv, DV, 0, fw.U, sv, DV, 1, DV, -1.f);
    KDA_TRY(gemm<C>(term(w.dW, sk, DK, 0, fw.W, sk, DK, 1, DK, -1.f), &t2, w.dM, 2, mc, H,
                    fw.meta, st));
  }
  // Y = dA K^
  KDA_TRY(gemm<DK>(term(w.dM, scc, C, 0, w.Kh, sk, DK, 0, C, 1.f), nullptr, w.Y, 0, mc, H,
                   fw.meta, st));
  // dK^ = dP^T Q~ + dA^T diag(b) K~
  {
    GemmTerm t2 = term(w.dM, scc, C, 1, w.Bk, sk, DK, 0, C, 1.f);
    KDA_TRY(gemm<DK>(term(w.dP, scc, C, 1, fw.Q, sk, DK, 0, C, 1.f), &t2, w.dKh, 0, mc, H,
                     fw.meta, st));
  }
  {
    auto kern = kda_bwd_finish<DK, DV, Tio>;
    constexpr size_t sm = bwd_finish_smem<DK>();
    KDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm));
    kern<<<dim3(mc, H), 256, sm, st>>>(
        (const Tio *)q, (const Tio *)k, (const Tio *)v, (const Tio *)la, (const Tio *)beta,
        (const Tio *)gate, (const Tio *)d_out, (Tio *)dq, (Tio *)dk, (Tio *)dv, (Tio *)dla, (Tio *)dbeta,
        gate ? (Tio *)dgate : nullptr, cu, n_seq, fixed_len, H, scale, flags, fw.meta,
        fw.seq_chunk_off, w.Y, w.dW, w.dU, w.dKh, w.dQt, w.dKd, w.dD, w.O);
    KDA_TRY(cudaGetLastError());
  }
#undef KDA_TRY
  return cudaSuccess;
}

}  // namespace

cudaError_t bwd_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_bwd_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

size_t chunk_bwd_ws_bytes(int64_t T_total, int n_seq, int H, int dk, int dv) {
  return chunk_ws_bytes(T_total, n_seq, H, dk, dv) + bwd_extra_bytes(T_total, n_seq, H, dk, dv);
}

cudaError_t launch_chunk_bwd(const void *q, const void *k, const void *v, const void *la,
                             const void *beta, const void *gate, const float *S0,
                             const void *d_out, const float *dSf, void *dq, void *dk, void *dv,
                             void *dla, void *dbeta, void *dgate, float *dS0, const int32_t *cu,
                             int n_seq, int64_t T_total, int H, int dk_, int dv_, float scale,
                             unsigned flags, kda_dtype dt, void *ws, cudaStream_t st) {
#define KDA_BWD_ARGS                                                                          \
  q, k, v, la, beta, gate, S0, d_out, dSf, dq, dk, dv, dla, dbeta, dgate, dS0, cu, n_seq, \
      T_total, H, scale, flags, dt, ws, st
  if (dt == KDA_DTYPE_BF16) {
    if (dk_ == 128 && dv_ == 128) return bwd_t<128, 128, __nv_bfloat16>(KDA_BWD_ARGS);
    if (dk_ == 64 && dv_ == 64) return bwd_t<64, 64, __nv_bfloat16>(KDA_BWD_ARGS);
    if (dk_ == 128 && dv_ == 64) return bwd_t<128, 64, __nv_bfloat16>(KDA_BWD_ARGS);
    if (dk_ == 64 && dv_ == 128) return bwd_t<64, 128, __nv_bfloat16>(KDA_BWD_ARGS);
  } else {
    if (dk_ == 128 && dv_ == 128) return bwd_t<128, 128, float>(KDA_BWD_ARGS);
    if (dk_ == 64 && dv_ == 64) return bwd_t<64, 64, float>(KDA_BWD_ARGS);
    if (dk_ == 128 && dv_ == 64) return bwd_t<128, 64, float>(KDA_BWD_ARGS);
    if (dk_ == 64 && dv_ == 128) return bwd_t<64, 128, float>(KDA_BWD_ARGS);
  }
#undef KDA_BWD_ARGS
  return cudaErrorInvalidValue;
}

}  // namespace kda
