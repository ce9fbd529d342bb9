// Chunked KDA forward on the sm_103a tensor cores (bf16 inputs, dk = dv = 128).
//
// Structure (K3 training overview, zuoshipin.com/article/18261, section 4
// "FlashKDA": per-chunk update cards prepared in parallel; only the state
// hand-off and read-out run in order):
//
// Stage A, kda_card_tc: one CTA per (chunk, head) builds the chunk's update
// card. With G the inclusive running sum of log_alpha inside the chunk,
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
// single tensor-core round trip per chunk.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
constexpr int CARD_STAGE = 82432;  // part copied into shared memory (PhiQ, B_c^T, e^{G_C})

// ---- stage A shared memory (offsets from a 1024-aligned base)
constexpr int A_X1 = 0;         // 32768: [Kt ; Qt] 128-row tile (K-major / MN-major)
constexpr int A_KH = 32768;     // 16384: Kh 64-row tile; during the solve T (fp32); later W^T 128x64
constexpr int A_VS = 49152;     // 16384: V 64-row tile; later Ut^T 128x64
constexpr int A_KD = 65536;     // 16384: Kd 64-row tile
constexpr int A_STG = 81920;    // 32768: input staging (half chunk); later P, T', M
constexpr int A_P = A_STG;            // 8192: P 64-row tile
constexpr int A_TB = A_STG + 8192;    // 8192: T' 64-row tile (and block temporaries during the solve)
constexpr int A_MS = A_STG + 16384;   // 16384: M fp32 64x64 (column-swizzled)
constexpr int A_DYN = 114688 + 1024;  // dynamic shared memory request (with alignment slack)

// ---- stage B shared memory
constexpr int B_STAGE_BYTES = 82944;  // CARD_STAGE rounded up to 1024
constexpr int B_SA = 2 * B_STAGE_BYTES;   // S^T bf16 operand, 128 x 128 K-major (32768)
constexpr int B_DYN = B_SA + 32768 + 1024;

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
__device__ __forceinline__ void put_bf(uint8_t *base, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(base + off) = __float2bfloat16_rn(x);
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

// fp32 64x64 matrix in shared memory, column index XOR-swizzled by row.
__device__ __forceinline__ int mix(int r, int c) { return r * 64 + (c ^ (r & 31)); }

// ===========================================================================
// Stage A: update cards. 128 threads; thread t is key/value channel t in the
// element-wise phase and tensor-memory lane t in the epilogues.
__global__ void __launch_bounds__(128, 2) kda_card_tc(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ la,
    const __nv_bfloat16 *__restrict__ beta, const int32_t *__restrict__ cu, int n_seq,
    int64_t fixed_len, int H, unsigned flags, const ChunkMeta *__restrict__ meta,
    const int *__restrict__ off, uint8_t *__restrict__ cards) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_rk[C], s_rq[C], s_b[C], s_d[DD];

  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (meta->invalid || ci >= meta->total_chunks) return;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);

  const int s = find_seq(off, n_seq, ci);
  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int64_t t0 = ts + (int64_t)(ci - off[s]) * C;
  const int len = (int)min((int64_t)C, ls - (int64_t)(ci - off[s]) * C);
  const size_t row_stride = (size_t)H * DD;  // elements between consecutive tokens
  const bool l2 = (flags & KDA_QK_L2NORM) != 0;
  const bool dbg = (flags & KDA_DEBUG_CHECK) != 0;

  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  if (tid < C) {
    float b = tid < len ? __bfloat162float(beta[(size_t)(t0 + tid) * H + h]) : 0.f;
    if (dbg && tid < len && !(b >= 0.f && b <= 1.f)) set_err(kErrPrecondition);
    s_b[tid] = b;
  }

  // ---------------- element-wise phase, two halves of 32 rows
  float G = 0.f;  // running log-decay of channel tid
  const __nv_bfloat16 *srcs[4] = {k, q, la, v};
  for (int half = 0; half < 2; ++half) {
    const int h0 = half * 32;
    // stage rows [h0, h0 + 32) of k, q, log_alpha, v as raw bf16 rows of 256 bytes
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int idx = tid + 128 * i;
      const int tn = idx >> 9, row = (idx >> 4) & 31, ch = idx & 15;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (h0 + row < len)
        val = *reinterpret_cast<const uint4 *>(srcs[tn] + (size_t)(t0 + h0 + row) * row_stride +
                                               (size_t)h * DD + ch * 8);
      *reinterpret_cast<uint4 *>(sm + A_STG + tn * 8192 + row * 256 + ch * 16) = val;
    }
    __syncthreads();
    // row norms of k and q: four threads per row, 32 channels each
    {
      const int row = tid >> 2, part = tid & 3;
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float a[8], b[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + A_STG + 0 * 8192 + row * 256 +
                                                 (part * 4 + c4) * 16), a);
        unpack8(*reinterpret_cast<const uint4 *>(sm + A_STG + 1 * 8192 + row * 256 +
                                                 (part * 4 + c4) * 16), b);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sk = fmaf(a[e], a[e], sk);
          sq = fmaf(b[e], b[e], sq);
        }
      }
      sk += __shfl_xor_sync(0xffffffffu, sk, 1);
      sk += __shfl_xor_sync(0xffffffffu, sk, 2);
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      if (part == 0) {
        s_rk[h0 + row] = l2 ? rsqrtf(sk + kL2Eps) : 1.f;
        s_rq[h0 + row] = l2 ? rsqrtf(sq + kL2Eps) : 1.f;
      }
    }
    __syncthreads();
    // channel-parallel pass: running decay and the decayed operands
    {
      const int c = tid;
      for (int row = 0; row < 32; ++row) {
        const int r = h0 + row;
        const float l = bf(sm + A_STG + 2 * 8192, row * 256 + c * 2);
        if (dbg && r < len && !(l >= kLogAlphaMin && l <= 0.f)) set_err(kErrPrecondition);
        G += l;
        const float ep = __expf(G), en = __expf(-G);
        const float kn = bf(sm + A_STG, row * 256 + c * 2) * s_rk[r];
        const float qn = bf(sm + A_STG + 8192, row * 256 + c * 2) * s_rq[r];
        const float vv = bf(sm + A_STG + 3 * 8192, row * 256 + c * 2);
        put_bf(sm + A_X1, sw128_off(r, c, 128), kn * ep);
        put_bf(sm + A_X1, sw128_off(64 + r, c, 128), qn * ep);
        put_bf(sm + A_KH, sw128_off(r, c, 64), kn * en);
        put_bf(sm + A_VS, sw128_off(r, c, 64), vv);
      }
    }
    __syncthreads();
  }
  // Kd = Kh * e^{G_C}
  {
    const int c = tid;
    const float eC = __expf(G);
    s_d[c] = eC;
    for (int r = 0; r < C; ++r) put_bf(sm + A_KD, sw128_off(r, c, 64), bf(sm + A_KH, sw128_off(r, c, 64)) * eC);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  uint32_t phase = 0;
  bool ok = true;

  auto wait_mma = [&]() {
    if (!mbar_wait(&bar_mma, phase)) {
      if (lane == 0) set_err(kErrTimeout);
      ok = false;
    }
    phase ^= 1u;
    tc_fence_after();
  };

  // ---------------- GEMM 1: D1[0,64) = [Kt ; Qt] Kh^T  (M=128, N=64, K=128)
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, 64, 0, 0);
    for (int kk = 0; kk < 8; ++kk)
      mma_bf16(tb + 0, desc_kmajor(sb + A_X1, 128, kk), desc_kmajor(sb + A_KH, 64, kk), id,
               kk > 0);
    mma_commit(&bar_mma);
  }
  wait_mma();
  // epilogue 1: lanes 0-63 -> M (fp32, strict lower, beta-scaled rows); lanes 64-127 -> P (bf16)
  {
    const int L = warp * 32 + lane;
    float a[64];
    {
      float t32[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 0), t32);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = t32[i];
      tmem_ld32(tmem_addr(tb, warp * 32, 32), t32);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) a[32 + i] = t32[i];
    }
    float *Ms = reinterpret_cast<float *>(sm + A_MS);
    if (L < 64) {
      const int r = L;
      const float b = s_b[r];
#pragma unroll
      for (int i = 0; i < 64; ++i) Ms[mix(r, i)] = i < r ? b * a[i] : 0.f;
    } else {
      const int r = L - 64;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e[u] = (ch * 8 + u <= r) ? a[ch * 8 + u] : 0.f;
        *reinterpret_cast<uint4 *>(sm + A_P + sw128_chunk(r, ch, 64)) = pack8(e);
      }
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---------------- T = (I + M)^{-1}, blocked by 16; T kept in A_KH (fp32, swizzled)
  {
    const float *Ms = reinterpret_cast<const float *>(sm + A_MS);
    float *Ts = reinterpret_cast<float *>(sm + A_KH);
    float *Xt = reinterpret_cast<float *>(sm + A_TB);  // 3 x 16 x 16 temporaries
    if (tid < 64) {  // diagonal blocks: thread = (block a, column j)
      const int a = tid >> 4, j = tid & 15, o = 16 * a;
      float t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int kx = 0; kx < i; ++kx) acc = fmaf(Ms[mix(o + i, o + kx)], t[kx], acc);
        t[i] = (i == j) ? 1.f : (i < j ? 0.f : -acc);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) Ts[mix(o + i, o + j)] = t[i];
    }
    __syncthreads();
    for (int d = 1; d < 4; ++d) {
      const int nb = 4 - d;
      for (int e = tid; e < nb * 256; e += 128) {
        const int a = e >> 8, i = (e >> 4) & 15, j = e & 15, rb = a + d;
        float acc = 0.f;
        for (int kb = a; kb < rb; ++kb)
#pragma unroll
          for (int kx = 0; kx < 16; ++kx)
            acc = fmaf(Ms[mix(16 * rb + i, 16 * kb + kx)], Ts[mix(16 * kb + kx, 16 * a + j)], acc);
        Xt[e] = acc;
      }
      __syncthreads();
      for (int e = tid; e < nb * 256; e += 128) {
        const int a = e >> 8, i = (e >> 4) & 15, j = e & 15, rb = a + d;
        float acc = 0.f;
#pragma unroll
        for (int kx = 0; kx < 16; ++kx)
          acc = fmaf(Ts[mix(16 * rb + i, 16 * rb + kx)], Xt[(a << 8) + (kx << 4) + j], acc);
        Ts[mix(16 * rb + i, 16 * a + j)] = -acc;
      }
      __syncthreads();
    }
    // T' = T diag(beta) -> bf16 64-row K-major tile (rows r, columns j)
    {
      const int r = tid >> 1, hc = tid & 1;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = hc * 32 + ch * 8 + u;
          e[u] = (j <= r) ? Ts[mix(r, j)] * s_b[j] : 0.f;
        }
        *reinterpret_cast<uint4 *>(sm + A_TB + sw128_chunk(r, hc * 4 + ch, 64)) = pack8(e);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---------------- GEMM 2: W^T -> [64,128), Ut^T -> [128,192)   (M=128, N=64, K=64)
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, 64, 1, 0);
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t bd = desc_kmajor(sb + A_TB, 64, kk);
      mma_bf16(tb + 64, sdesc_sw128(sb + A_X1 + kk * 2048, 128 * 128, 1024), bd, id, kk > 0);
      mma_bf16(tb + 128, sdesc_sw128(sb + A_VS + kk * 2048, 64 * 128, 1024), bd, id, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  wait_mma();
  // epilogue 2: W^T and Ut^T rows (lane = channel) -> bf16 128-row K-major tiles
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const int L = warp * 32 + lane;
    uint8_t *dst = sm + (which == 0 ? A_KH : A_VS);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float t32[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 64 + 64 * which + 32 * half), t32);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(dst + sw128_chunk(L, half * 4 + ch, 128)) = pack8(t32 + ch * 8);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint8_t *card = cards + ((size_t)ci * H + h) * CARD_BYTES;
  // ---------------- GEMMs 3a/4a on W^T: (PW)^T -> [0,64), W^T Kd -> [64,192)
  if (tid == 0) {
    const uint32_t id3 = idesc_bf16(128, 64, 0, 0), id4 = idesc_bf16(128, 128, 0, 1);
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = desc_kmajor(sb + A_KH, 128, kk);
      mma_bf16(tb + 0, ad, desc_kmajor(sb + A_P, 64, kk), id3, kk > 0);
      mma_bf16(tb + 64, ad, desc_mnmajor(sb + A_KD, 64, kk), id4, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  wait_mma();
  {
    const int c = warp * 32 + lane;  // key channel
    // Q'^T[c][r] = Qt[r][c] - (PW)^T[c][r]
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float t32[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 32 * half), t32);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int r = half * 32 + ch * 8 + u;
          e[u] = bf(sm + A_X1, sw128_off(64 + r, c, 128)) - t32[ch * 8 + u];
        }
        *reinterpret_cast<uint4 *>(card + CARD_PHIQ + sw128_chunk(c, 16 + half * 4 + ch, 128)) =
            pack8(e);
      }
    }
    // Phi'^T[c][c'] = -(W^T Kd)[c][c']
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float t32[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 64 + 32 * q4), t32);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) e[u] = -t32[ch * 8 + u];
        *reinterpret_cast<uint4 *>(card + CARD_PHIQ + sw128_chunk(c, q4 * 4 + ch, 128)) = pack8(e);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // ---------------- GEMMs 3b/4b on Ut^T: O_intra^T -> [0,64), B_c^T -> [64,192)
  if (tid == 0) {
    const uint32_t id3 = idesc_bf16(128, 64, 0, 0), id4 = idesc_bf16(128, 128, 0, 1);
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t ad = desc_kmajor(sb + A_VS, 128, kk);
      mma_bf16(tb + 0, ad, desc_kmajor(sb + A_P, 64, kk), id3, kk > 0);
      mma_bf16(tb + 64, ad, desc_mnmajor(sb + A_KD, 64, kk), id4, kk > 0);
    }
    mma_commit(&bar_mma);
  }
  wait_mma();
  {
    const int j = warp * 32 + lane;  // value channel
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float t32[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 32 * half), t32);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(card + CARD_OIT + ((half * 4 + ch) * 128 + j) * 16) =
            pack8(t32 + ch * 8);
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      float t32[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 64 + 32 * q4), t32);
      tmem_wait_ld();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(card + CARD_BCT + ((q4 * 4 + ch) * 128 + j) * 16) =
            pack8(t32 + ch * 8);
    }
    reinterpret_cast<float *>(card + CARD_D)[tid] = s_d[tid];
  }
  (void)ok;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}

// ===========================================================================
// Stage B: the sequential state pass. 128 threads; thread j owns tensor-memory
// lane j = value channel j (row j of S^T). mode 0: prefill; mode 1: segment
// summary on [X | Z] (blockIdx.y = 0: X with entry I; 1: Z with entry 0).
__global__ void __launch_bounds__(128, 1) kda_state_tc(
    int mode, const __nv_bfloat16 *__restrict__ gate, __nv_bfloat16 *__restrict__ out,
    const float *__restrict__ S0, float *__restrict__ S_final, float *__restrict__ X_out,
    float *__restrict__ Z_out, const int32_t *__restrict__ cu, int n_seq, int64_t fixed_len,
    int H, float scale, const ChunkMeta *__restrict__ meta, const int *__restrict__ off,
    const uint8_t *__restrict__ cards) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[2], bar_mma;
  __shared__ uint32_t tmem_base;
  if (meta->invalid) return;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = smem_u32(sm);
  const int chain = blockIdx.x, s = chain / H, h = chain % H, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, j = tid;
  const bool xpart = (mode == 1 && blockIdx.y == 0);
  const bool with_bc = !xpart;
  const bool with_o = (mode == 0 && out != nullptr);

  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int nchunks = (int)((ls + C - 1) / C);
  const int cbase = nchunks > 0 ? off[s] : 0;
  auto card_of = [&](int n) { return cards + ((size_t)(cbase + n) * H + h) * CARD_BYTES; };
  // element (c, j) of the entry state, and of the result
  auto entry = [&](int c) -> float {
    if (mode == 0) return S0 ? S0[(((size_t)s * H + h) * DD + c) * DD + j] : 0.f;
    return (xpart && c == j) ? 1.f : 0.f;
  };
  auto result_ptr = [&](int c) -> float * {
    if (mode == 0) return S_final ? S_final + (((size_t)s * H + h) * DD + c) * DD + j : nullptr;
    if (xpart) return X_out + (((size_t)s * H + h) * DD + c) * DD + j;
    return Z_out + (((size_t)s * H + h) * DD + c) * DD + j;
  };
  if (nchunks == 0) {
    for (int c = 0; c < DD; ++c) {
      float *p = result_ptr(c);
      if (p) *p = entry(c);
    }
    return;
  }

  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_full[0], 1);
    mbar_init(&bar_full[1], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  int loads_issued = 0;
  auto load_card = [&](int n) {  // by thread 0
    uint8_t *dst = sm + (n & 1) * B_STAGE_BYTES;
    const uint8_t *src = card_of(n);
    mbar_arrive_expect_tx(&bar_full[n & 1], CARD_STAGE);
    for (int o = 0; o < CARD_STAGE; o += 16384) {
      const int bytes = min(16384, CARD_STAGE - o);
      bulk_g2s(dst + o, src + o, bytes, &bar_full[n & 1]);
    }
    ++loads_issued;
  };
  if (tid == 0) {
    load_card(0);
    if (nchunks > 1) load_card(1);
  }
  uint32_t full_phase[2] = {0u, 0u}, mma_phase = 0u;
  int loads_done = 0;
  bool ok = true;

  // For the MMA of chunk n: tensor memory [0,128) <- Diag(e^{G_C}) S + B_c (fp32) and the
  // bf16 operand S^T (row j) in shared memory, from one 32-column piece `x` of row j of S^T.
  auto stage_piece = [&](int n, int q4, const float *x) {
    const uint8_t *st = sm + (n & 1) * B_STAGE_BYTES;
    const float *dv = reinterpret_cast<const float *>(st + CARD_D);
    float init[32];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      float bc[8];
      if (with_bc)
        unpack8(*reinterpret_cast<const uint4 *>(st + CARD_BCT + ((q4 * 4 + ch) * 128 + j) * 16),
                bc);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = q4 * 32 + ch * 8 + u;
        init[ch * 8 + u] = dv[c] * x[ch * 8 + u] + (with_bc ? bc[u] : 0.f);
      }
      *reinterpret_cast<uint4 *>(sm + B_SA + sw128_chunk(j, q4 * 4 + ch, 128)) = pack8(x + ch * 8);
    }
    tmem_st32(tmem_addr(tb, warp * 32, 32 * q4), init);
  };
  auto finish_stage = [&]() {
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
  };
  auto issue_mma = [&](int n) {  // by thread 0
    const uint32_t stg = sb + (n & 1) * B_STAGE_BYTES;
    const uint32_t idS = idesc_bf16(128, 128, 0, 1), idO = idesc_bf16(128, 64, 0, 1);
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t ad = desc_kmajor(sb + B_SA, 128, kk);
      const uint64_t bS = sdesc_sw128(stg + CARD_PHIQ + kk * 2048, 128 * 128, 1024);
      mma_bf16(tb + 0, ad, bS, idS, 1u);
      if (with_o) {
        const uint64_t bO = sdesc_sw128(stg + CARD_PHIQ + 2 * 16384 + kk * 2048, 128 * 128, 1024);
        mma_bf16(tb + 128 + 64 * (n & 1), ad, bO, idO, kk > 0);
      }
    }
    mma_commit(&bar_mma);
  };
  auto wait_full = [&](int n) -> bool {
    const bool r = mbar_wait(&bar_full[n & 1], full_phase[n & 1]);
    full_phase[n & 1] ^= 1u;
    if (r) ++loads_done;
    return r;
  };

  // chunk 0: entry state from global memory
  if (!wait_full(0)) ok = false;
  if (ok) {
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
      float x[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) x[u] = entry(q4 * 32 + u);
      stage_piece(0, q4, x);
    }
    finish_stage();
  }
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) issue_mma(0);

  for (int n = 0; n < nchunks && ok; ++n) {
    const int64_t t0 = ts + (int64_t)n * C;
    const int len = (int)min((int64_t)C, ls - (int64_t)n * C);
    if (!mbar_wait(&bar_mma, mma_phase)) {
      ok = false;
      break;
    }
    mma_phase ^= 1u;
    tc_fence_after();
    // the card of chunk n is consumed: refill its stage with chunk n + 2
    if (tid == 0 && n + 2 < nchunks) load_card(n + 2);
    const bool last = (n + 1 == nchunks);
    if (!last && !wait_full(n + 1)) {
      ok = false;
      break;
    }
    // state after chunk n: stage it for chunk n + 1, or write it out
#pragma unroll 1
    for (int q4 = 0; q4 < 4; ++q4) {
      float x[32];
      tmem_ld32(tmem_addr(tb, warp * 32, 32 * q4), x);
      tmem_wait_ld();
      if (last) {
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          float *p = result_ptr(q4 * 32 + u);
          if (p) *p = x[u];
        }
      } else {
        stage_piece(n + 1, q4, x);
      }
    }
    if (!last) {
      finish_stage();
      named_bar(1, 128);
      tc_fence_after();
      if (tid == 0) issue_mma(n + 1);
    }
    // output of chunk n (overlaps the MMA of chunk n + 1)
    if (with_o) {
      const uint8_t *card = card_of(n);
#pragma unroll 1
      for (int hf = 0; hf < 2; ++hf) {
        float t32[32];
        tmem_ld32(tmem_addr(tb, warp * 32, 128 + 64 * (n & 1) + 32 * hf), t32);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          float oi[8];
          unpack8(*reinterpret_cast<const uint4 *>(card + CARD_OIT + ((hf * 4 + ch) * 128 + j) * 16),
                  oi);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = hf * 32 + ch * 8 + u;
            if (r < len) {
              const size_t g = ((size_t)(t0 + r) * H + h) * DD + j;
              const float gv = gate ? __bfloat162float(gate[g]) : 1.f;
              out[g] = __float2bfloat16_rn(scale * gv * (t32[ch * 8 + u] + oi[u]));
            }
          }
        }
      }
      tc_fence_before();
    }
  }
  if (!ok) {
    if (lane == 0) set_err(kErrTimeout);
    // let copies still in flight land (bounded) before shared memory is released
    if (tid == 0)
      for (int n = loads_done; n < loads_issued; ++n)
        if (!mbar_wait(&bar_full[n & 1], full_phase[n & 1], 100000000ull)) break;
        else full_phase[n & 1] ^= 1u;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
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

cudaError_t launch_card_tc(const void *q, const void *k, const void *v, const void *la,
                           const void *beta, const int32_t *cu, int n_seq, int64_t T_total, int H,
                           unsigned flags, const ChunkWs &ws, cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(kda_card_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, A_DYN);
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  kda_card_tc<<<dim3(ws.max_chunks, H), 128, A_DYN, st>>>(
      (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k, (const __nv_bfloat16 *)v,
      (const __nv_bfloat16 *)la, (const __nv_bfloat16 *)beta, cu, n_seq, fixed_len, H, flags,
      ws.meta, ws.seq_chunk_off, ws.cards);
  return cudaGetLastError();
}

cudaError_t launch_state_tc(int mode, const void *gate, void *out, const float *S0,
                            float *S_final, float *X_out, float *Z_out, const int32_t *cu,
                            int n_seq, int64_t T_total, int H, float scale, const ChunkWs &ws,
                            cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(kda_state_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, B_DYN);
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  kda_state_tc<<<dim3(n_seq * H, mode == 0 ? 1 : 2), 128, B_DYN, st>>>(
      mode, (const __nv_bfloat16 *)gate, (__nv_bfloat16 *)out, S0, S_final, X_out, Z_out, cu,
      n_seq, fixed_len, H, scale, ws.meta, ws.seq_chunk_off, ws.cards);
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
