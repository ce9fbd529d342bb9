// The update card of one (chunk, head) on the sm_103a tensor cores, as a device function run by
// a group of 256 threads: the one-card-per-CTA kernel (kda_card_tc.cu) and the persistent
// prefill kernel (kda_prefill_fused.cu) both build their cards with it.
//
// K3 training overview (zuoshipin.com/article/18261), section 4 "FlashKDA": the update cards
// (forget gate, Q/K normalisation, decay, intra-chunk correction matrix) are prepared in
// parallel across chunks. From TMA-loaded, 128-byte-swizzled input tiles (card layout and
// the resulting affine step in tc_card_layout.cuh):
//   M  = strict_lower(diag(b) Kt Kh^T),   P = lower(Qt Kh^T)              (GEMM 1)
//   T  = (I + M)^{-1}  (16 x 16 diagonal blocks, two-level recursion), T' = T diag(b)
//   W^T = Kt^T T'^T,   Ut^T = V^T T'^T                                    (GEMM 2)
//   Q'  = Qt - P W,    O_intra = P Ut                                     (GEMM 3)
//   Phi' = -Kd^T W,    B_c = Kd^T Ut                                      (GEMM 4)
// (Derivation: U = Ut - W S, O = Qt S + P U, S_next = Diag(e^{G_C}) S + Kd^T U.)
// Ut enters GEMMs 3b/4b as two bf16 terms, Ut = hi + lo (hi = bf16(Ut), lo = bf16(Ut - hi)):
// when one key is re-written by many tokens of a chunk, Ut holds differences of successive
// values that the product with Kd sums back up (a telescoping sum), and a single bf16
// rounding of each term would add up to a few 1e-2 of the state.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_card_layout.cuh"
#include "tc_common.cuh"

namespace kda {
namespace tcb {

using namespace tc;
using namespace tcl;

// ===========================================================================
// Shared memory of one card-building group (256 threads). The four input tiles arrive by TMA
// with 128-byte swizzling, i.e. already in the tensor-core operand layout, and the
// element-wise pass rewrites them in place: k -> Kt, q -> Qt (one 128-row tile [Kt ; Qt]),
// log_alpha -> Kh -> Kd. Offsets from a 1024-aligned base:
constexpr int A_X1 = 0;          // 32768: [k|Kt ; q|Qt] 128-row tile; later P (64-row) at 0
constexpr int A_LA = 32768;      // 16384: log_alpha -> Kh -> Kd (64-row tile)
constexpr int A_V = 49152;       // 16384: V (64-row tile)
constexpr int A_M = 65536;       // 17408: M (fp32, 64 x 68 padded); later W^T (128-row x 64)
constexpr int A_T = 82944;       // 17408: T (fp32, 64 x 68 padded)
constexpr int A_TB = 100352;     // 8192:  T' = T diag(b) (bf16 64-row tile); later identity
constexpr int A_XT = 108544;     // 3072:  block temporaries of the solve
constexpr int A_UL = 82944;      // 16384: after GEMM 2, the low bf16 part of Ut^T (128-row
                                 // K-major tile) in the dead T
constexpr int A_BODY = 111616;        // bytes of one group region
constexpr int A_DYN = A_BODY + 1024;  // one group, with alignment slack
constexpr uint32_t A_TMA_BYTES = 8 * 8192;

__device__ __forceinline__ int mix(int r, int c) { return r * 68 + c; }

// The inputs of the cards.
struct CardIn {
  const CUtensorMap *k, *q, *la, *v;  // [T_total, H, 128] bf16, box 64 channels x 1 head x 64 tokens
  const __nv_bfloat16 *beta;          // [T_total, H]
  int H;
  unsigned flags;
  uint8_t *cards;                     // one card per (chunk, head): cards + (ci * H + h) * CARD_BYTES
};

// One card-building group: 256 threads with their own shared memory, tensor memory, mbarriers
// and named barriers.
struct CardGroup {
  uint8_t *sm;                // A_BODY bytes, 1024-byte aligned
  const uint32_t *tmem_base;  // shared word holding the CTA's tensor-memory base
  uint32_t tmem_col;          // first of this group's 256 tensor-memory columns
  uint64_t *bar_tma, *bar_mma;
  float *s_rk, *s_rq, *s_b, *s_d;  // [64], [64], [64], [128]
  unsigned *err;              // device error word
  int tid;                    // 0..255 within the group
  int bar_main;               // named barrier of all 256 threads
  int bar_quad;               // bar_quad + q: the two warps of lane quadrant q (64 threads)
};

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// The four input tiles of the chunk starting at token t0 of head h, completing on bar_tma
// (one thread issues them; zero fill past the end of the tensors).
__device__ __forceinline__ void card_issue_loads(const CardIn &in, const CardGroup &G, int h,
                                                 int64_t t0) {
  mbar_arrive_expect_tx(G.bar_tma, A_TMA_BYTES);
  for (int a = 0; a < 2; ++a) {
    tma_load_3d(G.sm + A_X1 + a * 16384, in.k, 64 * a, h, (int)t0, G.bar_tma);
    tma_load_3d(G.sm + A_X1 + a * 16384 + 8192, in.q, 64 * a, h, (int)t0, G.bar_tma);
    tma_load_3d(G.sm + A_LA + a * 8192, in.la, 64 * a, h, (int)t0, G.bar_tma);
    tma_load_3d(G.sm + A_V + a * 8192, in.v, 64 * a, h, (int)t0, G.bar_tma);
  }
}

// Raises the ready flag of the group's previous card (persistent prefill): each warp's bulk
// stores of that card have completed and are fenced against the generic proxy, the barrier
// that follows makes every thread's stores visible to thread 0, and its gpu-scope fence
// (cumulative) and release store publish the whole card. Call it with every thread of the
// group; `flag` is null when there is nothing to publish.
__device__ __forceinline__ void card_publish(const CardGroup &G, unsigned *flag) {
  if (flag == nullptr) return;
  if ((G.tid & 31) == 0) {
    bulk_wait_all();
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  named_bar(G.bar_main, 256);
  if (G.tid == 0) {
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flag), "r"(1u) : "memory");
  }
}

// The card of global chunk ci (tokens [t0, t0 + len) of head h), its input tiles already
// issued by card_issue_loads; bar_tma completes in phase tma_parity, bar_mma runs four phases
// (its parity is the same before and after). Every thread of the group calls it and gets back
// whether all of its bounded waits succeeded (a timeout is also recorded in the error word).
// prev_flag: the ready flag of the group's previous card, raised (card_publish) while this
// card's inputs are in flight, or null.
__device__ __forceinline__ bool card_body(const CardIn &in, const CardGroup &G, int ci, int h,
                                          int64_t t0, int len, uint32_t tma_parity,
                                          unsigned *prev_flag = nullptr) {
  uint8_t *sm = G.sm;
  const uint32_t sb = smem_u32(sm);
  const int tid = G.tid;
  const int warp = tid >> 5, lane = tid & 31, quad = warp & 3, grp = warp >> 2;
  uint64_t &bar_tma = *G.bar_tma;
  uint64_t &bar_mma = *G.bar_mma;
  float *s_rk = G.s_rk, *s_rq = G.s_rq, *s_b = G.s_b, *s_d = G.s_d;
  const unsigned flags = in.flags;
  const int H = in.H;
  const __nv_bfloat16 *beta = in.beta;
  uint8_t *cards = in.cards;
  const bool l2 = (flags & KDA_QK_L2NORM) != 0;
  const bool dbg = (flags & KDA_DEBUG_CHECK) != 0;

  if (tid < C) {
    float b = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    if (tid < len && (flags & KDA_GATE_LOGITS)) b = __frcp_rn(1.f + __expf(-b));  // sigmoid
    if (dbg && tid < len && !(b >= 0.f && b <= 1.f)) atomicOr(G.err, kErrPrecondition);
    s_b[tid] = b;
  }
  card_publish(G, prev_flag);
  tc_fence_before();
  named_bar(G.bar_main, 256);
  tc_fence_after();
  const uint32_t tb = *G.tmem_base + G.tmem_col;
  bool ok = mbar_wait(&bar_tma, tma_parity);

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
      }
      // with gate logits: log(alpha) = max(-e^a, log 1/2) (uniform branches: the exponentials
      // and the checks are not evaluated when their flag is off)
      if (flags & KDA_GATE_LOGITS)
#pragma unroll
        for (int u = 0; u < 8; ++u) la8[i][u] = fmaxf(-__expf(la8[i][u]), kLogHalf);
      if (dbg && r < len)
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (!(la8[i][u] >= kLogAlphaMin && la8[i][u] <= 0.f)) atomicOr(G.err, kErrPrecondition);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (r >= len) la8[i][u] = 0.f;
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
  named_bar(G.bar_main, 256);
  // exclusive prefix of the row-group partial sums, in place: one thread per channel walks the
  // 16 groups once (a thread per (channel group, row group) re-reading every earlier group
  // made this the second-slowest step of the card)
  if (tid < DD) {
    float x[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) x[g] = part[g * 128 + tid];
    float run = 0.f;
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      part[g * 128 + tid] = run;
      run += x[g];
    }
  }
  named_bar(G.bar_main, 256);
  {
    // running log-decay G entering this thread's first row: sum over earlier row groups
    float G[8];
    {
      const float4 x0 = *reinterpret_cast<const float4 *>(part + rg * 128 + cc * 8);
      const float4 x1 = *reinterpret_cast<const float4 *>(part + rg * 128 + cc * 8 + 4);
      G[0] = x0.x; G[1] = x0.y; G[2] = x0.z; G[3] = x0.w;
      G[4] = x1.x; G[5] = x1.y; G[6] = x1.z; G[7] = x1.w;
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
  named_bar(G.bar_main, 256);
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
      for (int i = 0; i < 32; i += 4) {  // 16-byte stores (68-float rows)
        const int col = 32 * grp + i;
        *reinterpret_cast<float4 *>(Ms + mix(r, col)) =
            make_float4(col < r ? b * a[i] : 0.f, col + 1 < r ? b * a[i + 1] : 0.f,
                        col + 2 < r ? b * a[i + 2] : 0.f, col + 3 < r ? b * a[i + 3] : 0.f);
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
  named_bar(G.bar_main, 256);

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
    named_bar(G.bar_main, 256);
    // Off-diagonal blocks by a two-level recursion (T lower triangular, T_aa known):
    // (1) inside each 32-row half: T_{a+1,a} = -T_{a+1,a+1} (M_{a+1,a} T_{a,a}), a = 0, 2;
    // (2) T_21 = -T_22 (M_21 T_11) for the 32 x 32 halves. Y = M_21 T_11 is parked in the
    // unused upper triangle of T (rows 0-31, columns 32-63).
    {
      const int a = 2 * (tid >> 7), j = tid & 15, i0 = ((tid >> 4) & 7) * 2;  // 2 rows each
      const int ro = 16 * (a + 1), co = 16 * a;
      float x0 = 0.f, x1 = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 16; k4 += 4) {  // X = M_{a+1,a} T_aa; T_aa[k][j] = 0 for k < j
        const float4 m0 = *reinterpret_cast<const float4 *>(Ms + mix(ro + i0, co + k4));
        const float4 m1 = *reinterpret_cast<const float4 *>(Ms + mix(ro + i0 + 1, co + k4));
        const float a0[4] = {m0.x, m0.y, m0.z, m0.w}, a1[4] = {m1.x, m1.y, m1.z, m1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = k4 + u;
          const float t = k >= j ? Ts[mix(co + k, co + j)] : 0.f;
          x0 = fmaf(a0[u], t, x0);
          x1 = fmaf(a1[u], t, x1);
        }
      }
      Xt[(tid >> 7) * 256 + i0 * 16 + j] = x0;
      Xt[(tid >> 7) * 256 + (i0 + 1) * 16 + j] = x1;
      named_bar(G.bar_main, 256);
      float y0 = 0.f, y1 = 0.f;
#pragma unroll
      for (int k4 = 0; k4 < 16; k4 += 4) {  // T_{a+1,a} = -T_{a+1,a+1} X; T_bb[i][k] = 0, k > i
        const float4 t0 = *reinterpret_cast<const float4 *>(Ts + mix(ro + i0, ro + k4));
        const float4 t1 = *reinterpret_cast<const float4 *>(Ts + mix(ro + i0 + 1, ro + k4));
        const float b0[4] = {t0.x, t0.y, t0.z, t0.w}, b1[4] = {t1.x, t1.y, t1.z, t1.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k = k4 + u;
          const float xk = Xt[(tid >> 7) * 256 + k * 16 + j];
          if (k <= i0) y0 = fmaf(b0[u], xk, y0);
          if (k <= i0 + 1) y1 = fmaf(b1[u], xk, y1);
        }
      }
      Ts[mix(ro + i0, co + j)] = -y0;
      Ts[mix(ro + i0 + 1, co + j)] = -y1;
      named_bar(G.bar_main, 256);
    }
    {
      const int j = tid & 31, i0 = (tid >> 5) * 4;  // column j, rows i0..i0+3 of the 32 x 32 block
      float y[4] = {0.f, 0.f, 0.f, 0.f};
      // Y = M_21 T_11, T_11[k][j] = 0 for k < j (not stored there: masked). The loop runs
      // over all k in every lane: a lane-dependent start made the warps diverge.
#pragma unroll
      for (int k4 = 0; k4 < 32; k4 += 4) {
        float mr[4][4];  // rows 32 + i0 + u, columns k4 .. k4 + 3 (warp-uniform 16-byte loads)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 m = *reinterpret_cast<const float4 *>(Ms + mix(32 + i0 + u, k4));
          mr[u][0] = m.x, mr[u][1] = m.y, mr[u][2] = m.z, mr[u][3] = m.w;
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = k4 + kk;
          const float t = k >= j ? Ts[mix(k, j)] : 0.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) y[u] = fmaf(mr[u][kk], t, y[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) Ts[mix(i0 + u, 32 + j)] = y[u];
      named_bar(G.bar_main, 256);
      float z[4] = {0.f, 0.f, 0.f, 0.f};
      // T_21 = -T_22 Y, T_22[i][k] = 0 for k > i (masked): every warp runs all 32 steps, so
      // the warps with the lower rows no longer hold the barrier for those with the higher
#pragma unroll
      for (int k4 = 0; k4 < 32; k4 += 4) {
        float tr[4][4];  // rows 32 + i0 + u, columns 32 + k4 .. + 3 (masked below)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 v = *reinterpret_cast<const float4 *>(Ts + mix(32 + i0 + u, 32 + k4));
          tr[u][0] = v.x, tr[u][1] = v.y, tr[u][2] = v.z, tr[u][3] = v.w;
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = k4 + kk;
          const float yk = Ts[mix(k, 32 + j)];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float t = k <= i0 + u ? tr[u][kk] : 0.f;
            z[u] = fmaf(t, yk, z[u]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) Ts[mix(32 + i0 + u, j)] = -z[u];
      named_bar(G.bar_main, 256);
    }
    // T' = T diag(b) -> bf16 64-row K-major tile (rows r, columns j): 16 columns per thread
    {
      const int r = tid >> 2, qc = tid & 3;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        float e[8], tv[8];
        const float4 v0 = *reinterpret_cast<const float4 *>(Ts + mix(r, qc * 16 + ch * 8));
        const float4 v1 = *reinterpret_cast<const float4 *>(Ts + mix(r, qc * 16 + ch * 8 + 4));
        tv[0] = v0.x, tv[1] = v0.y, tv[2] = v0.z, tv[3] = v0.w;
        tv[4] = v1.x, tv[5] = v1.y, tv[6] = v1.z, tv[7] = v1.w;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = qc * 16 + ch * 8 + u;
          e[u] = (j <= r) ? tv[u] * s_b[j] : 0.f;
        }
        *reinterpret_cast<uint4 *>(sm + A_TB + sw128_chunk(r, qc * 2 + ch, 64)) = pack8(e);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  named_bar(G.bar_main, 256);
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
      for (int ch = 0; ch < 4; ++ch) {
        const uint4 hi = pack8(t32 + ch * 8);
        *reinterpret_cast<uint4 *>(dst + sw128_chunk(L, half * 4 + ch, 128)) = hi;
        if (grp == 1) {  // Ut^T: the rounding residue as a second bf16 tile
          float h8[8], lo[8];
          unpack8(hi, h8);
#pragma unroll
          for (int u = 0; u < 8; ++u) lo[u] = t32[ch * 8 + u] - h8[u];
          *reinterpret_cast<uint4 *>(sm + A_UL + sw128_chunk(L, half * 4 + ch, 128)) = pack8(lo);
        }
      }
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
  named_bar(G.bar_main, 256);
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
    // twelve 4 KB staging blocks in regions dead by now: the Qt rows and Kt's second atom
    // column [A_X1 + 8192, A_LA), W^T [A_M, A_M + 16384) and the identity [A_TB, A_TB + 8192);
    // P, Kd and both Ut^T tiles stay intact for GEMMs 3b/4b
    static_assert(A_X1 + 8192 + 6 * 4096 == A_LA && A_TB + 8192 <= A_XT, "staging blocks");
    auto stage_block = [&](int i) -> uint8_t * {
      return sm + (i < 6 ? A_X1 + 8192 + i * 4096
                         : (i < 10 ? A_M + (i - 6) * 4096 : A_TB + (i - 10) * 4096));
    };
    uint8_t *blk = stage_block(grp * 4 + quad);  // (quadrant, atom grp)
    uint8_t *blk2 = stage_block(8 + quad);       // (quadrant, atom 2), shared by grp 0/1
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
    named_bar(G.bar_quad + quad, 64);  // both halves of the atom-2 block are staged
    if (grp == 0 && lane == 0) {
      bulk_s2g(card + CARD_PHIQ + 2 * 16384 + L0 * 128, blk2, 4096);
      bulk_commit();
    }
  }
  tc_fence_before();
  named_bar(G.bar_main, 256);
  tc_fence_after();
  // ---------------- GEMMs 3b/4b on Ut^T: O_intra^T -> [0,64), B_c^T -> [64,192)
  if (tid == 0 && ok) {
    const uint32_t id3 = idesc_bf16(128, 64, 0, 0), id4 = idesc_bf16(128, 128, 0, 1);
    for (int part2 = 0; part2 < 2; ++part2)  // Ut^T = hi + lo
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = desc_kmajor(sb + (part2 ? A_UL : A_V), 128, kk);
        const uint32_t acc = (part2 | kk) > 0;
        mma_bf16(tb + 0, ad, desc_kmajor(sb + A_X1, 64, kk), id3, acc);
        mma_bf16(tb + 64, ad, desc_mnmajor(sb + A_LA, 64, kk), id4, acc);
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
  if (!ok && lane == 0) atomicOr(G.err, kErrTimeout);
  // the card-tile bulk stores have read shared memory (and, when the card is published to
  // another CTA, completed their writes)
  if (lane == 0) bulk_wait_read_all();
  tc_fence_before();
  named_bar(G.bar_main, 256);
  return ok;
}

}  // namespace tcb
}  // namespace kda
