// Chunked KDA forward on the sm_103a tensor cores (bf16 inputs, dk = dv = 128).
//
// Structure (K3 training overview, zuoshipin.com/article/18261, section 4
// "FlashKDA": per-chunk update cards prepared in parallel; only the state
// hand-off and read-out run in order):
//
// Stage A, kda_card_tc: one CTA per (chunk, head), two per SM, builds the
// chunk's update card from TMA-loaded, 128-byte-swizzled input tiles. With G the inclusive running sum of log_alpha inside the chunk,
// Kt = k e^{G}, Kh = k e^{-G}, Qt = q e^{G}, Kd = k e^{G_C - G} (k, q L2-normalised):
//   M  = strict_lower(diag(b) Kt Kh^T),   P = lower(Qt Kh^T)              (GEMM 1)
//   T  = (I + M)^{-1}  (blocked forward substitution), T' = T diag(b)
//   W^T = Kt^T T'^T,   Ut^T = V^T T'^T                                    (GEMM 2)
//   Q'  = Qt - P W,    O_intra = P Ut                                     (GEMM 3)
//   Phi' = -Kd^T W,    B_c = Kd^T Ut                                      (GEMM 4)
// so that, for the state S entering the chunk,
//   S_next = Diag(e^{G_C}) S + Phi' S + B_c,   O = Q' S + O_intra,  o = scale g O.
// (Derivation: U = Ut - W S, O = Qt S + P U, S_next = Diag(e^{G_C}) S + Kd^T U.)
//
// Stage B, kda_state_tc: one CTA per (sequence, head). The fp32 state lives in
// tensor memory as S^T (lane = value channel). Per chunk the CTA pre-loads
// Diag(e^{G_C}) S + B_c into tensor memory and issues one group of MMAs,
// bf16(S^T) x [Phi'^T | Q'^T], accumulating onto it, so the serial path has a
// single tensor-core round trip per chunk; two warpgroups stage the state and a
// third turns the output accumulators into o while the next chunk's MMAs run.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kda_common.cuh"
#include "tc_common.cuh"

namespace kda {

__device__ unsigned g_tc_err;

namespace {

using namespace tc;

constexpr int C = kChunk;  // 64
constexpr int DD = 128;    // dk = dv

// ---- update card (per chunk and head), bytes
constexpr int CARD_PHIQ = 0;       // [Phi'^T | Q'^T]: MN-major tile, 128 rows x 192 cols, 3 atom cols
constexpr int CARD_BCT = 49152;    // B_c^T: [16][128][8] bf16 (8-column chunks, lane-interleaved)
constexpr int CARD_D = 81920;      // e^{G_C}: 128 fp32
constexpr int CARD_OIT = 82432;    // O_intra^T: [8][128][8] bf16
constexpr int CARD_BYTES = 98816;

// ---- stage B shared memory
constexpr int B_NSTAGE = 3;            // card ring depth
constexpr int kPrefetch = 3;           // cards prefetched into L2 beyond the ring
constexpr int B_STAGE_TX = CARD_BCT + 512;  // [Phi'^T | Q'^T] then e^{G_C} (49664 bytes)
constexpr int B_STAGE_BYTES = 50176;  // B_STAGE_TX rounded up to 1024
constexpr int B_SA = B_NSTAGE * B_STAGE_BYTES;  // S^T bf16 operand, 128 x 128 K-major (32768)
constexpr int B_OT = B_SA + 32768;         // output tile: 64 tokens x (128 + 4) fp32
constexpr int B_DYN = B_OT + 64 * (DD + 4) * 4 + 1024;

__device__ __forceinline__ void set_err(unsigned bits) { atomicOr(&g_tc_err, bits); }

__device__ __forceinline__ int find_seq(const int *off, int n_seq, int ci) {
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= ci) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void seq_range(const int32_t *cu, int64_t fixed_len, int s, int64_t *t0,
                                          int64_t *len) {
  if (cu) {
    *t0 = cu[s];
    *len = (int64_t)cu[s + 1] - cu[s];
  } else {
    *t0 = (int64_t)s * fixed_len;
    *len = fixed_len;
  }
}

__device__ __forceinline__ float bf(const uint8_t *base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}
__device__ __forceinline__ uint4 pack8(const float *v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  return u;
}
__device__ __forceinline__ void unpack8(uint4 u, float *v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// fp32 64x64 matrix in shared memory with a padded row pitch.
__device__ __forceinline__ int mix(int r, int c) { return r * 65 + c; }

// ===========================================================================
// Stage A: update cards. One CTA (256 threads, two per SM) per (chunk, head).
// The four input tiles arrive by TMA with 128-byte swizzling, i.e. already in
// the tensor-core operand layout, and the element-wise pass rewrites them in
// place: k -> Kt, q -> Qt (one 128-row tile [Kt ; Qt]), log_alpha -> Kh -> Kd.
// Shared memory (offsets from a 1024-aligned base):
constexpr int A_X1 = 0;          // 32768: [k|Kt ; q|Qt] 128-row tile; later P (64-row) at 0
constexpr int A_LA = 32768;      // 16384: log_alpha -> Kh -> Kd (64-row tile)
constexpr int A_V = 49152;       // 16384: V (64-row tile)
constexpr int A_M = 65536;       // 16640: M (fp32, 64 x 65 padded); later W^T (128-row x 64)
constexpr int A_T = 82176;       // 16640: T (fp32, 64 x 65 padded)
constexpr int A_TB = 99328;      // 8192:  T' = T diag(b) (bf16 64-row tile); later identity
constexpr int A_XT = 107520;     // 3072:  block temporaries of the solve
constexpr int A_DYN = 110592 + 1024;  // with alignment slack
constexpr int LDM = 65;          // row pitch of M and T (conflict-free rows and columns)
constexpr uint32_t A_TMA_BYTES = 8 * 8192;

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(256, 2) kda_card_tc(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16 *__restrict__ beta, const int32_t *__restrict__ cu, int n_seq,
    int64_t fixed_len, int H, unsigned flags, const ChunkMeta *__restrict__ meta,
    const int *__restrict__ off, uint8_t *__restrict__ cards) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_rk[C], s_rq[C], s_b[C], s_d[DD];

  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, quad = warp & 3, grp = warp >> 2;
  if (meta->invalid || ci >= meta->total_chunks) return;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);

  const int s = find_seq(off, n_seq, ci);
  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int64_t t0 = ts + (int64_t)(ci - off[s]) * C;
  const int len = (int)min((int64_t)C, ls - (int64_t)(ci - off[s]) * C);
  const bool l2 = (flags & KDA_QK_L2NORM) != 0;
  const bool dbg = (flags & KDA_DEBUG_CHECK) != 0;

  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar_tma, A_TMA_BYTES);
    for (int a = 0; a < 2; ++a) {
      tma_load_3d(sm + A_X1 + a * 16384, &tm_k, 64 * a, h, (int)t0, &bar_tma);
      tma_load_3d(sm + A_X1 + a * 16384 + 8192, &tm_q, 64 * a, h, (int)t0, &bar_tma);
      tma_load_3d(sm + A_LA + a * 8192, &tm_la, 64 * a, h, (int)t0, &bar_tma);
      tma_load_3d(sm + A_V + a * 8192, &tm_v, 64 * a, h, (int)t0, &bar_tma);
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  if (tid < C) {
    float b = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    if (tid < len && (flags & KDA_GATE_LOGITS)) b = __frcp_rn(1.f + __expf(-b));  // sigmoid
    if (dbg && tid < len && !(b >= 0.f && b <= 1.f)) set_err(kErrPrecondition);
    s_b[tid] = b;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  bool ok = mbar_wait(&bar_tma, 0);

  // ---------------- element-wise phase: thread = (8-channel chunk cc, rows 4*rg .. 4*rg+3)
  const int cc = tid & 15, rg = tid >> 4;
  float* part = reinterpret_cast<float *>(sm + A_M);  // [16 row groups][128 channels], before M
  float la8[4][8];
  {
    float ssk[4], ssq[4], tot[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) tot[u] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rg * 4 + i;
      float kk[8], qq[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + A_X1 + sw128_chunk(r, cc, 128)), kk);
      unpack8(*reinterpret_cast<const uint4 *>(sm + A_X1 + sw128_chunk(64 + r, cc, 128)), qq);
      unpack8(*reinterpret_cast<const uint4 *>(sm + A_LA + sw128_chunk(r, cc, 64)), la8[i]);
      ssk[i] = 0.f;
      ssq[i] = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        ssk[i] = fmaf(kk[u], kk[u], ssk[i]);
        ssq[i] = fmaf(qq[u], qq[u], ssq[i]);
        // with gate logits: log(alpha) = max(-e^a, log 1/2)
        la8[i][u] = r >= len ? 0.f
                    : (flags & KDA_GATE_LOGITS) ? fmaxf(-__expf(la8[i][u]), kLogHalf)
                                                : la8[i][u];
        if (dbg && r < len && !(la8[i][u] >= kLogAlphaMin && la8[i][u] <= 0.f))
          set_err(kErrPrecondition);
        tot[u] += la8[i][u];
      }
    }
    // row sums over the 16 threads of a half-warp (same rows, all 128 channels)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        ssk[i] += __shfl_xor_sync(0xffffffffu, ssk[i], o);
        ssq[i] += __shfl_xor_sync(0xffffffffu, ssq[i], o);
      }
    if (cc == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = rg * 4 + i;
        // padded rows (r >= len) are scaled to zero: no contribution anywhere
        s_rk[r] = r >= len ? 0.f : (l2 ? rsqrtf(ssk[i] + kL2Eps) : 1.f);
        s_rq[r] = r >= len ? 0.f : (l2 ? rsqrtf(ssq[i] + kL2Eps) : 1.f);
      }
    *reinterpret_cast<float4 *>(part + rg * 128 + cc * 8) = make_float4(tot[0], tot[1], tot[2], tot[3]);
    *reinterpret_cast<float4 *>(part + rg * 128 + cc * 8 + 4) = make_float4(tot[4], tot[5], tot[6], tot[7]);
  }
  __syncthreads();
  {
    // running log-decay G entering this thread's first row: sum over earlier row groups
    float G[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) G[u] = 0.f;
    for (int g = 0; g < rg; ++g) {
      const float4 x0 = *reinterpret_cast<const float4 *>(part + g * 128 + cc * 8);
      const float4 x1 = *reinterpret_cast<const float4 *>(part + g * 128 + cc * 8 + 4);
      G[0] += x0.x; G[1] += x0.y; G[2] += x0.z; G[3] += x0.w;
      G[4] += x1.x; G[5] += x1.y; G[6] += x1.z; G[7] += x1.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = rg * 4 + i;
      float kk[8], qq[8], kt[8], qt[8], kh[8];
      unpack8(*reinterpret_cast<const uint4 *>(sm + A_X1 + sw128_chunk(r, cc, 128)), kk);
      unpack8(*reinterpret_cast<const uint4 *>(sm + A_X1 + sw128_chunk(64 + r, cc, 128)), qq);
      const float rk = s_rk[r], rq = s_rq[r];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        G[u] += la8[i][u];
        const float ep = __expf(G[u]), en = __expf(-G[u]);
        const float kn = kk[u] * rk;
        kt[u] = kn * ep;
        kh[u] = kn * en;
        qt[u] = qq[u] * rq * ep;
      }
      *reinterpret_cast<uint4 *>(sm + A_X1 + sw128_chunk(r, cc, 128)) = pack8(kt);
      *reinterpret_cast<uint4 *>(sm + A_X1 + sw128_chunk(64 + r, cc, 128)) = pack8(qt);
      *reinterpret_cast<uint4 *>(sm + A_LA + sw128_chunk(r, cc, 64)) = pack8(kh);
    }
    if (rg == 15)  // after the last row: G = G_C
#pragma unroll
      for (int u = 0; u < 8; ++u) s_d[cc * 8 + u] = __expf(G[u]);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t phase = 0;
  auto wait_mma = [&]() {
    if (ok && !mbar_wait(&bar_mma, phase)) ok = false;
    phase ^= 1u;
    tc_fence_after();
  };

  // ---------------- GEMM 1: D1[0,64) = [Kt ; Qt] Kh^T   (M=128, N=64, K=128)
  if (tid == 0 && ok) {
    const uint32_t id = idesc_bf16(128, 64, 0, 0);
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(tb + 0, desc_kmajor(sb + A_X1, 128, kk), desc_kmajor(sb + A_LA, 64, kk), id, kk > 0);
    mma_commit(&bar_mma);
  }
  wait_mma();
  {
    // lanes 0-63: M = strict_lower(diag(b) Kt Kh^T) -> fp32; group g takes columns [32g, 32g+32)
    if (quad < 2) {
      const int r = quad * 32 + lane;
      float a[32];
      tmem_ld32(tmem_addr(tb, quad * 32, 32 * grp), a);
      tmem_wait_ld();
      float *Ms = reinterpret_cast<float *>(sm + A_M);
      const float b = s_b[r];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int col = 32 * grp + i;
        Ms[mix(r, col)] = col < r ? b * a[i] : 0.f;
      }
    }
    // Kh is no longer read by the tensor cores: Kd = Kh * e^{G_C} in place
    float eC[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) eC[u] = s_d[cc * 8 + u];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 *p = reinterpret_cast<uint4 *>(sm + A_LA + sw128_chunk(rg * 4 + i, cc, 64));
      float x[8];
      unpack8(*p, x);
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] *= eC[u];
      *p = pack8(x);
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---------------- T = (I + M)^{-1}, blocked by 16 (fp32)
  {
    const float *Ms = reinterpret_cast<const float *>(sm + A_M);
    float *Ts = reinterpret_cast<float *>(sm + A_T);
    float *Xt = reinterpret_cast<float *>(sm + A_XT);
    if (tid < 64) {  // diagonal blocks: thread = (block a, column j); right-looking
      const int a = tid >> 4, j = tid & 15, o = 16 * a;
      float acc[16], t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
      for (int kx = 0; kx < 16; ++kx) {
        t[kx] = (kx == j) ? 1.f : (kx < j ? 0.f : -acc[kx]);
#pragma unroll
        for (int i = kx + 1; i < 16; ++i) acc[i] = fmaf(Ms[mix(o + i, o + kx)], t[kx], acc[i]);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Ts[mix(o + i, o + j)] = t[i];
    }
    __syncthreads();
    // Off-diagonal blocks by a two-level recursion (T lower triangular, T_aa known):
    // (1) inside each 32-row half: T_{a+1,a} = -T_{a+1,a+1} (M_{a+1,a} T_{a,a}), a = 0, 2;
    // (2) T_21 = -T_22 (M_21 T_11) for the 32 x 32 halves. Y = M_21 T_11 is parked in the
    // unused upper triangle of T (rows 0-31, columns 32-63).
    {
      const int a = 2 * (tid >> 7), j = tid & 15, i0 = ((tid >> 4) & 7) * 2;  // 2 rows each
      const int ro = 16 * (a + 1), co = 16 * a;
      float x0 = 0.f, x1 = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {  // X = M_{a+1,a} T_aa; T_aa[k][j] = 0 for k < j
        const float t = k >= j ? Ts[mix(co + k, co + j)] : 0.f;
        x0 = fmaf(Ms[mix(ro + i0, co + k)], t, x0);
        x1 = fmaf(Ms[mix(ro + i0 + 1, co + k)], t, x1);
      }
      Xt[(tid >> 7) * 256 + i0 * 16 + j] = x0;
      Xt[(tid >> 7) * 256 + (i0 + 1) * 16 + j] = x1;
      __syncthreads();
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int k = 0; k < 16; ++k) {  // T_{a+1,a} = -T_{a+1,a+1} X; T_bb[i][k] = 0 for k > i
        const float xk = Xt[(tid >> 7) * 256 + k * 16 + j];
        if (k <= i0) y0 = fmaf(Ts[mix(ro + i0, ro + k)], xk, y0);
        if (k <= i0 + 1) y1 = fmaf(Ts[mix(ro + i0 + 1, ro + k)], xk, y1);
      }
      Ts[mix(ro + i0, co + j)] = -y0;
      Ts[mix(ro + i0 + 1, co + j)] = -y1;
      __syncthreads();
    }
    {
      const int j = tid & 31, i0 = (tid >> 5) * 4;  // column j, rows i0..i0+3 of the 32 x 32 block
      float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int k = j; k < 32; ++k) {  // Y = M_21 T_11 (T_11[k][j] = 0 for k < j)
        const float t = Ts[mix(k, j)];
#pragma unroll
        for (int u = 0; u < 4; ++u) y[u] = fmaf(Ms[mix(32 + i0 + u, k)], t, y[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) Ts[mix(i0 + u, 32 + j)] = y[u];
      __syncthreads();
      float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int k = 0; k < i0 + 4; ++k) {  // T_21 = -T_22 Y (T_22[i][k] = 0 for k > i)
        const float yk = Ts[mix(k, 32 + j)];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (k <= i0 + u) z[u] = fmaf(Ts[mix(32 + i0 + u, 32 + k)], yk, z[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) Ts[mix(32 + i0 + u, j)] = -z[u];
      __syncthreads();
    }
    // T' = T diag(b) -> bf16 64-row K-major tile (rows r, columns j): 16 columns per thread
    {
      const int r = tid >> 2, qc = tid & 3;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = qc * 16 + ch * 8 + u;
          e[u] = (j <= r) ? Ts[mix(r, j)] * s_b[j] : 0.f;
        }
        *reinterpret_cast<uint4 *>(sm + A_TB + sw128_chunk(r, qc * 2 + ch, 64)) = pack8(e);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---------------- GEMM 2: W^T -> [64,128), Ut^T -> [128,192)   (M=128, N=64, K=64)
  if (tid == 0 && ok) {
    const uint32_t id = idesc_bf16(128, 64, 1, 0);
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t bd = desc_kmajor(sb + A_TB, 64, kk);
      mma_bf16(tb + 64, sdesc_sw128(sb + A_X1 + kk * 2048, 128 * 128, 1024), bd, id, kk > 0);
      mma_bf16(tb + 128, sdesc_sw128(sb + A_V + kk * 2048, 64 * 128, 1024), bd, id, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  wait_mma();
  {
    const int L = quad * 32 + lane;
    // group 0: W^T rows -> tile at A_M; group 1: Ut^T rows -> tile at A_V (128-row K-major;
    // V is no longer read)
    uint8_t *dst = sm + (grp == 0 ? A_M : A_V);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float t32[32];
      tmem_ld32(tmem_addr(tb, quad * 32, 64 + 64 * grp + 32 * half), t32);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(dst + sw128_chunk(L, half * 4 + ch, 128)) = pack8(t32 + ch * 8);
    }
    // identity (64 x 64, bf16) in the T' tile, which GEMM 2 has finished reading
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int e = tid * 2 + i, row = e >> 3, ch = e & 7;
      float v8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v8[u] = (ch * 8 + u == row) ? 1.f : 0.f;
      *reinterpret_cast<uint4 *>(sm + A_TB + sw128_chunk(row, ch, 64)) = pack8(v8);
    }
    // lanes 64-127 of D1 hold Qt Kh^T: P = lower(.) -> bf16 64-row tile at A_X1 (Kt is dead)
    if (quad >= 2) {
      const int r = L - 64;
      float a[32];
      tmem_ld32(tmem_addr(tb, quad * 32, 32 * grp), a);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e[u] = (32 * grp + ch * 8 + u <= r) ? a[ch * 8 + u] : 0.f;
        *reinterpret_cast<uint4 *>(sm + A_X1 + sw128_chunk(r, grp * 4 + ch, 64)) = pack8(e);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint8_t *card = cards + ((size_t)ci * H + h) * CARD_BYTES;
  const int L = quad * 32 + lane;  // tensor-memory lane: key channel (a) / value channel (b)
  // ---------------- GEMMs 3a/4a: Q'^T = Qt^T I - W^T P^T -> [0,64), Phi'^T = -W^T Kd -> [64,192)
  // (A negated through the instruction descriptor)
  if (tid == 0 && ok) {
    const uint32_t idI = idesc_bf16(128, 64, 1, 0);
    const uint32_t id3 = idesc_bf16(128, 64, 0, 0) | kNegateA;
    const uint32_t id4 = idesc_bf16(128, 128, 0, 1) | kNegateA;
    for (int kk = 0; kk < 4; ++kk)
      mma_bf16(tb + 0, sdesc_sw128(sb + A_X1 + 8192 + kk * 2048, 128 * 128, 1024),
               desc_kmajor(sb + A_TB, 64, kk), idI, kk > 0);
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = desc_kmajor(sb + A_M, 128, kk);
      mma_bf16(tb + 0, ad, desc_kmajor(sb + A_X1, 64, kk), id3, 1u);
      mma_bf16(tb + 64, ad, desc_mnmajor(sb + A_LA, 64, kk), id4, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  wait_mma();
  // [Phi'^T | Q'^T] card tile: six 32-column pieces in tensor memory (0-1 Q'^T = tile atom 2,
  // 2-3 atom 0, 4-5 atom 1). Each warp stages whole 32-row x 128-byte blocks of the swizzled
  // tile in shared memory that GEMMs 3b/4b do not read (the dead Q~/K~ rows and W^T, T), and
  // writes each block with one 4 KB bulk copy: its rows are contiguous in the card, whereas
  // 16-byte stores from registers would touch 32 rows per instruction.
  {
    const int L0 = quad * 32;
    auto stage_half = [&](uint8_t *blk, int half, const float *t32) {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(blk + lane * 128 + ((((half * 4 + ch) ^ (lane & 7))) << 4)) =
            pack8(t32 + ch * 8);
    };
    uint8_t *blk = sm + 65536 + (grp * 4 + quad) * 4096;  // (quadrant, atom grp)
    uint8_t *blk2 = sm + 8192 + quad * 4096;               // (quadrant, atom 2), shared by grp 0/1
    float ta[32], tb2[32];
    tmem_ld32(tmem_addr(tb, quad * 32, 32 * (2 + 2 * grp)), ta);
    tmem_ld32(tmem_addr(tb, quad * 32, 32 * (3 + 2 * grp)), tb2);
    tmem_wait_ld();
    stage_half(blk, 0, ta);
    stage_half(blk, 1, tb2);
    tmem_ld32(tmem_addr(tb, quad * 32, 32 * grp), ta);
    tmem_wait_ld();
    stage_half(blk2, grp, ta);
    fence_async_smem();  // this thread's shared-memory writes -> visible to the bulk copies
    __syncwarp();
    if (lane == 0) {
      bulk_s2g(card + CARD_PHIQ + grp * 16384 + L0 * 128, blk, 4096);
      bulk_commit();
    }
    named_bar(2 + quad, 64);  // both halves of the atom-2 block are staged
    if (grp == 0 && lane == 0) {
      bulk_s2g(card + CARD_PHIQ + 2 * 16384 + L0 * 128, blk2, 4096);
      bulk_commit();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // ---------------- GEMMs 3b/4b on Ut^T: O_intra^T -> [0,64), B_c^T -> [64,192)
  if (tid == 0 && ok) {
    const uint32_t id3 = idesc_bf16(128, 64, 0, 0), id4 = idesc_bf16(128, 128, 0, 1);
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = desc_kmajor(sb + A_V, 128, kk);
      mma_bf16(tb + 0, ad, desc_kmajor(sb + A_X1, 64, kk), id3, kk > 0);
      mma_bf16(tb + 64, ad, desc_mnmajor(sb + A_LA, 64, kk), id4, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  wait_mma();
  {
    auto store_ob = [&](int p, const float *t32) {
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int off8 = p < 2 ? CARD_OIT + ((p * 4 + ch) * 128 + L) * 16
                               : CARD_BCT + (((p - 2) * 4 + ch) * 128 + L) * 16;
        *reinterpret_cast<uint4 *>(card + off8) = pack8(t32 + ch * 8);
      }
    };
    const int p0 = 3 * grp;
    float ta[32], tb2[32];
    tmem_ld32(tmem_addr(tb, quad * 32, 32 * p0), ta);
    tmem_ld32(tmem_addr(tb, quad * 32, 32 * (p0 + 1)), tb2);
    tmem_wait_ld();
    store_ob(p0, ta);
    store_ob(p0 + 1, tb2);
    tmem_ld32(tmem_addr(tb, quad * 32, 32 * (p0 + 2)), ta);
    tmem_wait_ld();
    store_ob(p0 + 2, ta);
  }
  if (tid < DD) reinterpret_cast<float *>(card + CARD_D)[tid] = s_d[tid];
  if (!ok && lane == 0) set_err(kErrTimeout);
  if (lane == 0) bulk_wait_all();  // the card-tile bulk stores have completed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tb, 256);
}

// ===========================================================================
// Stage B: the sequential state pass, one CTA per (sequence, head), 384 threads.
// Warps 0-7 (state group) carry the serial path: warp w serves tensor-memory
// lanes 32*(w%4).. (lane j = value channel j, i.e. row j of S^T) and the key
// columns [64*(w/4), 64*(w/4) + 64) of that row. Warps 8-11 (output group) read
// the chunk outputs from the same lanes, add O_intra, apply scale and gate and
// store o, off the serial path. mode 0: prefill; mode 1: segment summary on
// [X | Z] (blockIdx.y = 0: X with entry I; 1: Z with entry 0), no output.
//
// Tensor memory holds two accumulator sets, chunk n using set n % 2: columns
// [256b, 256b+128) the fp32 state S^T, [256b+128, 256b+192) the output block.
// Before the MMAs of chunk n the set is pre-loaded with Diag(e^{G_C}) S + B_c
// (state group) and zeros (output group), so one N = 192 MMA chain per chunk
// produces both the next state and the chunk output.
// mbarriers: bar_full[3] card stages landed; bar_mma chunk MMAs done (state
// group); bar_ofull[2] output block written (output group); bar_ofree[2]
// output block read and re-zeroed (MMA issuer).
__global__ void __launch_bounds__(384, 1) kda_state_tc(
    int mode, unsigned flags, const __nv_bfloat16 *__restrict__ gate,
    __nv_bfloat16 *__restrict__ out,
    const float *__restrict__ S0, float *__restrict__ S_final, float *__restrict__ X_out,
    float *__restrict__ Z_out, const int32_t *__restrict__ cu, int n_seq, int64_t fixed_len,
    int H, float scale, const ChunkMeta *__restrict__ meta, const int *__restrict__ off,
    const uint8_t *__restrict__ cards, CkptOut ck) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[B_NSTAGE], bar_mma, bar_ofull[2], bar_ofree[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  if (meta->invalid) return;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const int chain = blockIdx.x, s = chain / H, h = chain % H, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool state_grp = warp < 8;
  const int quad = warp & 3;           // lane quadrant of this warp
  const int j = quad * 32 + lane;      // tensor-memory lane / value channel
  const int half = (warp >> 2) & 1;    // state group: which 64 key columns
  const bool xpart = (mode == 1 && blockIdx.y == 0);
  const bool with_bc = !xpart;
  const bool with_o = (mode == 0 && out != nullptr);

  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int nchunks = (int)((ls + C - 1) / C);
  const int cbase = nchunks > 0 ? off[s] : 0;
  auto card_of = [&](int n) { return cards + ((size_t)(cbase + n) * H + h) * CARD_BYTES; };
  // element (c, j) of the entry state, and where element (c, j) of the result goes
  auto entry = [&](int c) -> float {
    if (mode == 0) return S0 ? S0[(((size_t)s * H + h) * DD + c) * DD + j] : 0.f;
    return (xpart && c == j) ? 1.f : 0.f;
  };
  auto result_ptr = [&](int c) -> float * {
    if (mode == 0) return S_final ? S_final + (((size_t)s * H + h) * DD + c) * DD + j : nullptr;
    if (xpart) return X_out + (((size_t)s * H + h) * DD + c) * DD + j;
    return Z_out + (((size_t)s * H + h) * DD + c) * DD + j;
  };
  // prefix-cache checkpoint after chunk n (mode 0): this thread's 64 rows of column j
  auto save_ckpt = [&](int n, const float *x0, const float *x1) {
    if (mode != 0) return;
    float *cp = ckpt_after_chunk(ck, s, n, ls, H, h, DD, DD);
    if (cp == nullptr) return;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      cp[(size_t)(64 * half + u) * DD + j] = x0[u];
      cp[(size_t)(64 * half + 32 + u) * DD + j] = x1[u];
    }
  };
  if (nchunks == 0) {
    if (state_grp)
      for (int c = 64 * half; c < 64 * half + 64; ++c) {
        float *p = result_ptr(c);
        if (p) *p = entry(c);
      }
    return;
  }

  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < B_NSTAGE; ++i) mbar_init(&bar_full[i], 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_ofull[0], 1);
    mbar_init(&bar_ofull[1], 1);
    mbar_init(&bar_ofree[0], 128);
    mbar_init(&bar_ofree[1], 128);
    fence_mbar_init();
    s_fail = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  auto set_col = [](int n) { return 256 * (n & 1); };
  if (state_grp) {
    int loads_issued = 0, loads_done = 0;
    uint32_t full_phase[B_NSTAGE] = {}, mma_phase = 0u;
    bool ok = true;
    const bool loader = (tid == 32);  // issues the card copies, off the MMA issuer's path
    auto stage_of = [](int n) { return n % B_NSTAGE; };
    // card n -> stage n % 3: [Phi'^T | Q'^T] and e^{G_C}
    auto load_card = [&](int n) {
      const int st = stage_of(n);
      uint8_t *dst = sm + st * B_STAGE_BYTES;
      const uint8_t *src = card_of(n);
      mbar_arrive_expect_tx(&bar_full[st], B_STAGE_TX);
      for (int o = 0; o < CARD_BCT; o += 16384) bulk_g2s(dst + o, src + o, 16384, &bar_full[st]);
      bulk_g2s(dst + CARD_BCT, src + CARD_D, 512, &bar_full[st]);
      ++loads_issued;
    };
    auto wait_full = [&](int n) -> bool {
      const int st = stage_of(n);
      const bool r = mbar_wait(&bar_full[st], full_phase[st]);
      full_phase[st] ^= 1u;
      if (r) ++loads_done;
      return r;
    };
    // this thread's 64 columns of B_c^T row j of chunk n, straight from the card in global
    // memory (lane-interleaved: a warp reads 512 contiguous bytes per 8-column chunk)
    uint4 bcr[8];
    auto fetch_bc = [&](int n) {
      if (!with_bc || n >= nchunks) return;
      const uint8_t *src = card_of(n) + CARD_BCT;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8)
        bcr[c8] = *reinterpret_cast<const uint4 *>(src + ((8 * half + c8) * 128 + j) * 16);
    };
    // Pre-load for chunk n: tensor memory <- Diag(e^{G_C}) S + B_c (fp32) and the bf16
    // operand S^T (row j) in shared memory, from the 32 key columns 64*half + 32*qq.
    auto stage_piece = [&](int n, int qq, const float *x) {
      const float *dv =
          reinterpret_cast<const float *>(sm + stage_of(n) * B_STAGE_BYTES + CARD_BCT);
      const int q4 = 2 * half + qq;
      float init[32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float bc[8];
        if (with_bc) unpack8(bcr[qq * 4 + ch], bc);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = q4 * 32 + ch * 8 + u;
          init[ch * 8 + u] = dv[c] * x[ch * 8 + u] + (with_bc ? bc[u] : 0.f);
        }
        *reinterpret_cast<uint4 *>(sm + B_SA + sw128_chunk(j, q4 * 4 + ch, 128)) =
            pack8(x + ch * 8);
      }
      tmem_st32(tmem_addr(tb, quad * 32, set_col(n) + 32 * q4), init);
    };
    auto finish_stage = [&]() {
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
    };
    auto issue_mma = [&](int n) -> bool {  // by thread 0
      // the output block of set n % 2 is read and zeroed (prologue, then chunk n - 2)
      if (with_o && !mbar_wait(&bar_ofree[n & 1], (n >> 1) & 1)) return false;
      tc_fence_after();
      const uint32_t stg = sb + stage_of(n) * B_STAGE_BYTES;
      const uint32_t id = idesc_bf16(128, with_o ? 192 : 128, 0, 1);
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tb + set_col(n), desc_kmajor(sb + B_SA, 128, kk),
                 sdesc_sw128(stg + CARD_PHIQ + kk * 2048, 128 * 128, 1024), id, 1u);
      mma_commit(&bar_mma);
      if (with_o) mma_commit(&bar_ofull[n & 1]);
      return true;
    };

    // whole cards into L2 ahead of their bulk copies (which otherwise wait on HBM latency)
    auto prefetch_card = [&](int n) {
      if (n >= nchunks) return;
      const uint8_t *src = card_of(n);
      for (int o = 0; o < CARD_BYTES; o += 32768)
        prefetch_l2(src + o, min(32768, CARD_BYTES - o));
    };
    if (loader) {
      for (int n = 0; n < B_NSTAGE && n < nchunks; ++n) load_card(n);
      for (int n = B_NSTAGE; n < B_NSTAGE + kPrefetch; ++n) prefetch_card(n);
    }
    fetch_bc(0);
    // chunk 0: entry state from global memory
    if (!wait_full(0)) ok = false;
    if (ok) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        float x[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = entry(64 * half + 32 * qq + u);
        stage_piece(0, qq, x);
      }
      finish_stage();
    }
    // all state threads agree on `ok`, so none is left waiting at a later barrier
    ok = named_bar_and(1, 256, ok);
    tc_fence_after();
    if (tid == 0 && ok && !issue_mma(0)) s_fail = 1;
    fetch_bc(1);

    for (int n = 0; n < nchunks && ok; ++n) {
      // a timed-out wait only clears `good`; the group votes on it at the barrier below
      bool good = mbar_wait(&bar_mma, mma_phase);
      mma_phase ^= 1u;
      tc_fence_after();
      // the card of chunk n is consumed: refill its stage with chunk n + 3
      if (good && loader && n + B_NSTAGE < nchunks) {
        load_card(n + B_NSTAGE);
        prefetch_card(n + B_NSTAGE + kPrefetch);
      }
      const bool last = (n + 1 == nchunks);
      if (good && !last) good = wait_full(n + 1);
      // state after chunk n: stage it for chunk n + 1, or write it out
      float x0[32], x1[32];
      if (good) {
        tmem_ld32(tmem_addr(tb, quad * 32, set_col(n) + 64 * half), x0);
        tmem_ld32(tmem_addr(tb, quad * 32, set_col(n) + 64 * half + 32), x1);
        tmem_wait_ld();
      }
      if (last) {
        if (good)
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            float *p0 = result_ptr(64 * half + u), *p1 = result_ptr(64 * half + 32 + u);
            if (p0) *p0 = x0[u];
            if (p1) *p1 = x1[u];
          }
        else
          ok = false;
        if (good) save_ckpt(n, x0, x1);
      } else {
        if (good) {
          stage_piece(n + 1, 0, x0);
          stage_piece(n + 1, 1, x1);
          finish_stage();
        }
        ok = named_bar_and(1, 256, good);
        tc_fence_after();
        if (!ok) break;
        if (tid == 0 && !issue_mma(n + 1)) s_fail = 1;
        save_ckpt(n, x0, x1);  // off the serial path: the next chunk's MMAs are in flight
        fetch_bc(n + 2);
      }
    }
    if (!ok || s_fail) {
      if (lane == 0) set_err(kErrTimeout);
      // let copies still in flight land (bounded) before shared memory is released
      if (loader)
        for (int n = loads_done; n < loads_issued; ++n) {
          const int st = stage_of(n);
          if (!mbar_wait(&bar_full[st], full_phase[st], 100000000ull)) break;
          full_phase[st] ^= 1u;
        }
    }
  } else if (with_o) {
    // output group: o = scale * g * (Q' S + O_intra) for chunk n. The output block of chunk n
    // starts as O_intra^T (seeded two chunks ahead from the card), so the MMA leaves
    // Q' S + O_intra in it. The four warps copy their lane quadrants (channels) into one
    // [64 tokens][128 channels] fp32 tile; then each thread takes 8 tokens x 8 channels, so
    // that a warp's gate loads and output stores cover two whole 256-byte rows per
    // instruction. The gate of the next chunk is loaded (same mapping) as this one is used.
    constexpr int LDT = DD + 4;  // tile row pitch (floats)
    float *tile = reinterpret_cast<float *>(sm + B_OT);
    const int ot = tid - 256;                   // output thread 0..127
    const int c8 = ot & 15, r0 = ot >> 4;       // store phase: channels 8*c8.., tokens r0 + 8m
    const bool logits = gate && (flags & KDA_GATE_LOGITS);
    // this lane's O_intra^T row (all 64 tokens, bf16) of chunk c, from the card
    auto load_oi = [&](int c, uint4 *oi) {
      const uint8_t *card = card_of(c);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        oi[ch] = c < nchunks ? *reinterpret_cast<const uint4 *>(card + CARD_OIT + (ch * 128 + j) * 16)
                             : make_uint4(0u, 0u, 0u, 0u);
    };
    auto seed = [&](int c, const uint4 *oi) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float x[32];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) unpack8(oi[hf * 4 + ch], x + ch * 8);
        tmem_st32(tmem_addr(tb, quad * 32, set_col(c) + 128 + 32 * hf), x);
      }
    };
    // gate of tokens r0 + 8m, channels 8*c8 .. 8*c8 + 7 of chunk c (1.0 when absent)
    auto load_gate = [&](int c, uint4 *gq) {
      const int64_t tc0 = ts + (int64_t)c * C;
      const int lc = (int)min((int64_t)C, ls - (int64_t)c * C);
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int r = r0 + 8 * m;
        gq[m] = (gate && c < nchunks && r < lc)
                    ? *reinterpret_cast<const uint4 *>(gate + ((size_t)(tc0 + r) * H + h) * DD + c8 * 8)
                    : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
      }
    };
    {
      uint4 oi[8];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        load_oi(b, oi);
        seed(b, oi);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bar_ofree[0]);
    mbar_arrive(&bar_ofree[1]);
    uint32_t ofull_phase[2] = {0u, 0u};
    uint4 gq[8];
    load_gate(0, gq);
    bool ok = true;
    for (int n = 0; n < nchunks; ++n) {
      const int64_t t0 = ts + (int64_t)n * C;
      const int len = (int)min((int64_t)C, ls - (int64_t)n * C);
      uint4 oi[8];
      load_oi(n + 2, oi);  // its latency overlaps the wait below
      // every output thread takes the same branch, so a timeout cannot strand the others
      ok = named_bar_and(2, 128, mbar_wait(&bar_ofull[n & 1], ofull_phase[n & 1]));
      if (!ok) break;
      ofull_phase[n & 1] ^= 1u;
      tc_fence_after();
      // both halves into the tile (token row, this lane's channel)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float t[32];
        tmem_ld32(tmem_addr(tb, quad * 32, set_col(n) + 128 + 32 * hf), t);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) tile[(hf * 32 + u) * LDT + j] = t[u];
      }
      // the block is read: seed it with O_intra^T of chunk n + 2, hand it back to the issuer
      seed(n + 2, oi);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_ofree[n & 1]);
      named_bar(2, 128);  // tile complete
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int r = r0 + 8 * m;
        const float4 a = *reinterpret_cast<const float4 *>(tile + r * LDT + c8 * 8);
        const float4 b = *reinterpret_cast<const float4 *>(tile + r * LDT + c8 * 8 + 4);
        float g8[8], e[8];
        unpack8(gq[m], g8);
        const float x8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < 8; ++u)
          e[u] = scale * (logits ? sigmoid_approx(g8[u]) : g8[u]) * x8[u];
        if (r < len)
          *reinterpret_cast<uint4 *>(out + ((size_t)(t0 + r) * H + h) * DD + c8 * 8) = pack8(e);
      }
      load_gate(n + 1, gq);  // the next chunk's gate, while its MMAs run
      named_bar(2, 128);     // tile consumed before the next chunk overwrites it
    }
    if (!ok && ot == 0) set_err(kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

bool tc_path(int dk, int dv, kda_dtype dt) {
  return dt == KDA_DTYPE_BF16 && dk == DD && dv == DD;
}

size_t tc_ws_bytes(int64_t T_total, int n_seq, int H) {
  const size_t mc = (size_t)(T_total / C) + (size_t)n_seq + 1;
  size_t b = align_up(sizeof(ChunkMeta), 256);
  b += align_up(sizeof(int) * (size_t)(n_seq + 1), 256);
  b += (size_t)mc * H * CARD_BYTES;
  return b;
}

ChunkWs tc_ws_carve(void *ws, int64_t T_total, int n_seq, int H) {
  ChunkWs w = {};
  char *p = (char *)ws;
  w.meta = (ChunkMeta *)p;
  p += align_up(sizeof(ChunkMeta), 256);
  w.seq_chunk_off = (int *)p;
  p += align_up(sizeof(int) * (size_t)(n_seq + 1), 256);
  w.cards = (uint8_t *)p;
  w.max_chunks = (int)((size_t)(T_total / C) + (size_t)n_seq + 1);
  return w;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map over a packed [T_total, H, 128] bf16 tensor; box = 64 channels x 1 head x 64 tokens,
// 128-byte swizzle (the tensor-core tile layout), zero fill past T_total.
static bool make_token_map(CUtensorMap *m, const void *base, int64_t T_total, int H) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)DD, (cuuint64_t)H, (cuuint64_t)T_total};
  cuuint64_t strides[2] = {(cuuint64_t)DD * 2, (cuuint64_t)H * DD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_card_tc(const void *q, const void *k, const void *v, const void *la,
                           const void *beta, const int32_t *cu, int n_seq, int64_t T_total, int H,
                           unsigned flags, const ChunkWs &ws, cudaStream_t st) {
  if (T_total == 0) return cudaSuccess;  // no chunk has tokens
  CUtensorMap mk, mq, mla, mv;
  if (!make_token_map(&mk, k, T_total, H) || !make_token_map(&mq, q, T_total, H) ||
      !make_token_map(&mla, la, T_total, H) || !make_token_map(&mv, v, T_total, H))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(kda_card_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, A_DYN);
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  kda_card_tc<<<dim3(ws.max_chunks, H), 256, A_DYN, st>>>(
      mk, mq, mla, mv, (const __nv_bfloat16 *)beta, cu, n_seq, fixed_len, H, flags, ws.meta,
      ws.seq_chunk_off, ws.cards);
  return cudaGetLastError();
}

cudaError_t launch_state_tc(int mode, unsigned flags, const void *gate, void *out, const float *S0,
                            float *S_final, float *X_out, float *Z_out, const int32_t *cu,
                            int n_seq, int64_t T_total, int H, float scale, const ChunkWs &ws,
                            cudaStream_t st, CkptOut ck) {
  cudaError_t e =
      cudaFuncSetAttribute(kda_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, B_DYN);
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  kda_state_tc<<<dim3(n_seq * H, mode == 0 ? 1 : 2), 384, B_DYN, st>>>(
      mode, flags, (const __nv_bfloat16 *)gate, (__nv_bfloat16 *)out, S0, S_final, X_out, Z_out, cu,
      n_seq, fixed_len, H, scale, ws.meta, ws.seq_chunk_off, ws.cards, ck);
  return cudaGetLastError();
}

cudaError_t tc_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_tc_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

}  // namespace kda
