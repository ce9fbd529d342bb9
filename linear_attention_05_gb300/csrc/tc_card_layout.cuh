// Layout of the tensor-core path's per-(chunk, head) update card and device helpers shared
// by the card kernel (kda_card_tc.cu) and the state pass (kda_state_tc.cu).
//
// K3 training overview (zuoshipin.com/article/18261), section 4 "FlashKDA": per-chunk update
// cards are prepared in parallel; only the state hand-off and the output read-out run in
// order. With G the inclusive running sum of log_alpha inside the chunk, Kt = k e^{G},
// Kh = k e^{-G}, Qt = q e^{G}, Kd = k e^{G_C - G} (k, q L2-normalised) and
// W = (I + M)^{-1} diag(b) Kt, Ut = (I + M)^{-1} diag(b) V, M = strict_lower(diag(b) Kt Kh^T),
// P = lower(Qt Kh^T), the card holds Phi' = -Kd^T W, Q' = Qt - P W, B_c = Kd^T Ut,
// O_intra = P Ut and e^{G_C}, so that for the state S entering the chunk
//   S_next = Diag(e^{G_C}) S + Phi' S + B_c,   O = Q' S + O_intra,   o = scale g O.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_common.cuh"

namespace kda {
namespace tcl {

using tc::pack_bf16x2;

constexpr int C = kChunk;  // 64
constexpr int DD = 128;    // dk = dv

// ---- update card (per chunk and head), bytes
constexpr int CARD_PHIQ = 0;       // [Phi'^T | Q'^T]: MN-major tile, 128 rows x 192 cols, 3 atom cols
constexpr int CARD_BCT = 49152;    // B_c^T: [16][128][8] bf16 (8-column chunks, lane-interleaved)
constexpr int CARD_D = 81920;      // e^{G_C}: 128 fp32
constexpr int CARD_OIT = 82432;    // O_intra^T: [8][128][8] bf16
constexpr int CARD_BYTES = 98816;


static __device__ __forceinline__ int find_seq(const int *off, int n_seq, int ci) {
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= ci) lo = mid; else hi = mid - 1;
  }
  return lo;
}

static __device__ __forceinline__ void seq_range(const int32_t *cu, int64_t fixed_len, int s, int64_t *t0,
                                          int64_t *len) {
  if (cu) {
    *t0 = cu[s];
    *len = (int64_t)cu[s + 1] - cu[s];
  } else {
    *t0 = (int64_t)s * fixed_len;
    *len = fixed_len;
  }
}

static __device__ __forceinline__ float bf(const uint8_t *base, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(base + off));
}
static __device__ __forceinline__ uint4 pack8(const float *v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  return u;
}
static __device__ __forceinline__ void unpack8(uint4 u, float *v) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// fp32 64x64 matrix in shared memory with a padded row pitch.

}  // namespace tcl
}  // namespace kda
