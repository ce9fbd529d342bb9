// Internal helpers shared by the libkda translation units (device side).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;
// log 0.5 rounded down by one bf16 ulp: the smallest log-retention the chunked
// kernels accept (64 tokens x 0.6953125 = 44.5, so exp(-Gamma) <= 2^64.2).
constexpr float kLogAlphaMin = -0.6953125f;
constexpr float kL2Eps = 1e-6f;

// Bits of the per-translation-unit device error word.
enum : unsigned {
  kErrPrecondition = 1u,
  kErrTimeout = 2u,
  kErrBadSeqlens = 4u,
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
// 8 consecutive elements (16-byte aligned for bf16, 32-byte for fp32) as fp32
__device__ __forceinline__ void load8(const float *p, float *o) {
  const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *o) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// `bytes` (a multiple of 16, from a 16-byte-aligned address) into L2, asynchronously
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Per-call metadata at the head of the chunk workspace.
struct ChunkMeta {
  int total_chunks;  // sum over sequences of ceil(len / 64)
  int invalid;       // non-zero: cu_seqlens rejected; every kernel exits
  int pad[62];
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

// Gate preparation fused into the kernels' loads (flag KDA_GATE_LOGITS): beta and the output
// gate arrive as logits, log_alpha as the forget gate's pre-activation a.
constexpr float kLogHalf = -0.69314718055994531f;
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }
// log(alpha) = max(-e^a, log 1/2): a negative log-retention with the lower bound alpha >= 1/2
__device__ __forceinline__ float log_alpha_of(float a) { return fmaxf(-expf(a), kLogHalf); }
__device__ __forceinline__ float prep_beta(float x, unsigned flags) {
  return (flags & KDA_GATE_LOGITS) ? sigmoid_f(x) : x;
}
__device__ __forceinline__ float prep_gate(float x, unsigned flags) {
  return (flags & KDA_GATE_LOGITS) ? sigmoid_f(x) : x;
}
__device__ __forceinline__ float prep_log_alpha(float x, unsigned flags) {
  return (flags & KDA_GATE_LOGITS) ? log_alpha_of(x) : x;
}

// Prefix-cache state checkpoints: [n_seq, per_seq, H, dk, dv] fp32; slot (s, i) holds the
// state after the first (i + 1) * every_chunks * 64 tokens of sequence s.
struct CkptOut {
  float *ptr = nullptr;
  int every_chunks = 0;  // boundary spacing in chunks (> 0 when ptr is set)
  int per_seq = 0;       // slots per sequence
};

// Optional exports of the SIMT prep kernel, per (chunk, head) slab, fp32 (used by the
// backward pass): K^ = k e^{-G} [64, dk], diag(b) K~ [64, dk], A = strict_lower(diag(b) K~ K^T)
// [64, 64].
struct PrepSave {
  float *Kh = nullptr, *Bk = nullptr, *A = nullptr;
};
// Optional saves of the SIMT state pass (mode 0), per slab, fp32: the state entering the chunk
// Sb [dk, dv], the corrected values U = U~ - W S [64, dv] and the chunk output before scale and
// gate O = Q~ S + P U [64, dv].
struct StateSave {
  float *Sb = nullptr, *Ub = nullptr, *O = nullptr;
};

// Base of the [dk, dv] checkpoint written after chunk n (0-based) of sequence s, or null when
// that chunk does not end on a checkpoint boundary inside the sequence.
__device__ __forceinline__ float *ckpt_after_chunk(const CkptOut &ck, int s, int n, int64_t len,
                                                   int H, int h, int dk, int dv) {
  if (ck.ptr == nullptr || (n + 1) % ck.every_chunks != 0) return nullptr;
  if ((int64_t)(n + 1) * 64 > len) return nullptr;  // boundary past the sequence end
  const int i = (n + 1) / ck.every_chunks - 1;
  if (i >= ck.per_seq) return nullptr;
  return ck.ptr + (((size_t)s * ck.per_seq + i) * H + h) * dk * dv;
}

}  // namespace kda

// Launchers and error-word accessors defined in the kernel translation units.
namespace kda {

constexpr int kMaxParts = 3;
struct ChunkWs {
  ChunkMeta *meta;
  int *seq_chunk_off;  // [n_seq + 1]
  float *W, *U, *Q, *Kd, *P, *D;  // SIMT path
  uint8_t *cards;                 // tensor-core path: one update card per (chunk, head)
  int max_chunks;
  // Split prefill (tensor-core path): part p < nparts of a sequence with n chunks holds its
  // chunks [floor(n * bound64[p] / 64), floor(n * bound64[p + 1] / 64)), bound64[0] = 0 and
  // bound64[nparts] = 64. seq_chunk_b [nparts - 1][n_seq + 1] holds, for each inner boundary,
  // the running sum over the sequences of floor(n * bound64[p] / 64) (with cu_seqlens); part p
  // leaves its state in mid[p & 1] ([n_seq, H, 128, 128]), where part p + 1 starts.
  // nparts = 0: no split.
  int nparts;
  int bound64[kMaxParts + 1];
  int *seq_chunk_b;
  float *mid[2];
  // tensor-core path: sequences by decreasing chunk count (ties by index) when there are at
  // most kOrderMax of them, else in index order. The state pass takes its chains in this
  // order, so the longest chains start in the first wave of CTAs.
  int *seq_order;
  // persistent prefill (fixed lengths, few chains): one ready flag per (chunk, head) card and the
  // card counter, both cleared at the start of each call
  unsigned *ready;
  int *next;
};
constexpr int kOrderMax = 256;

// Persistent prefill (kda_prefill_fused.cu): eligible shapes have at least kFusedMinChunks
// chunks per sequence and at most kFusedMaxChains (sequence, head) chains, and the device must
// leave at least kFusedMinBuilders SMs to build cards beside the chain owners. Measured on the
// GB300 against the two-kernel schedule: 16 chains x 256 chunks 0.731 vs 0.858 ms, 32 x 128
// 0.410 vs 0.565 ms, 8 x 128 0.384 vs 0.425 ms, 64 x 64 equal (0.39 ms); hence at most 48.
// The chain owners start their chains once the cards of the leading fraction of the chunks
// are claimed, the fraction from the rates kFusedCardUs (one card, one group of the persistent
// kernel) and kFusedStepUs (one chunk step of a chain) -- see fused_switch_chunks.
constexpr int kFusedMinChunks = 16;
constexpr int kFusedMaxChains = 48;
constexpr int kFusedMinBuilders = 48;
constexpr double kFusedCardUs = 20.0;
constexpr double kFusedStepUs = 2.85;
inline size_t fused_flag_bytes(int64_t T_total, int n_seq, int H) {
  const int64_t n_chunks = n_seq > 0 ? (T_total / n_seq + kChunk - 1) / kChunk : 0;
  return align_up(sizeof(unsigned) * (size_t)(n_seq * n_chunks * H), 256) + 256;
}

size_t chunk_ws_bytes(int64_t T_total, int n_seq, int H, int dk, int dv);
ChunkWs chunk_ws_carve(void *ws, int64_t T_total, int n_seq, int H, int dk, int dv);

cudaError_t launch_chunk_table(const int32_t *cu, int n_seq, int64_t T_total,
                               const ChunkWs &ws, cudaStream_t st);
cudaError_t launch_prep(const void *q, const void *k, const void *v,
                        const void *la, const void *beta, const int32_t *cu,
                        int n_seq, int64_t T_total, int H, int dk, int dv,
                        unsigned flags, kda_dtype dt, const ChunkWs &ws,
                        bool need_q, cudaStream_t st, PrepSave save = PrepSave());
// mode 0: forward (out, final); mode 1: segment summary (X_out, Z_out)
cudaError_t launch_state_pass(int mode, unsigned flags, const void *gate, void *out,
                              const float *S0, float *S_final, float *X_out,
                              float *Z_out, const int32_t *cu, int n_seq,
                              int64_t T_total, int H, int dk, int dv,
                              float scale, kda_dtype dt, const ChunkWs &ws,
                              cudaStream_t st, CkptOut ck = CkptOut(),
                              StateSave save = StateSave());
cudaError_t launch_decode(const void *q, const void *k, const void *v,
                          const void *la, const void *beta, const void *gate,
                          void *out, float *state, const int32_t *slot,
                          int n_slots, int N, int H, int dk, int dv,
                          float scale, unsigned flags, kda_dtype dt,
                          cudaStream_t st);
cudaError_t launch_scan_combine(const float *X, const float *Z, int n_seg,
                                int H, int dk, int dv, const float *S_init,
                                float *E_out, float *S_final, cudaStream_t st);

// Tensor-core path (bf16, dk = dv = 128): update cards + state pass.
bool tc_path(int dk, int dv, kda_dtype dt);
// 2D tensor map over `rows` rows of 128 fp32 values: box 32 columns x 128 rows, 128-byte swizzle.
bool make_rows_map_f32(CUtensorMap *m, const void *base, uint64_t rows);
// Split prefill: the number of parts the prefill splits each sequence into (writing their
// boundaries in 64ths to bound64[0 .. parts]), or 0 when the state pass would leave too few
// SMs idle for the cards of the later parts to use.
int tc_split_parts(int64_t T_total, int n_seq, int H, int *bound64 = nullptr);
size_t tc_ws_bytes(int64_t T_total, int n_seq, int H);
ChunkWs tc_ws_carve(void *ws, int64_t T_total, int n_seq, int H);
// part -1: every chunk; p >= 0: part p of a split prefill (ws.nparts > 0). The state pass of
// part p leaves its state in ws.mid[p & 1], where part p + 1 starts.
cudaError_t launch_card_tc(const void *q, const void *k, const void *v, const void *la,
                           const void *beta, const int32_t *cu, int n_seq, int64_t T_total,
                           int H, unsigned flags, const ChunkWs &ws, cudaStream_t st,
                           int part = -1);
cudaError_t launch_state_tc(int mode, unsigned flags, const void *gate, void *out, const float *S0,
                            float *S_final, float *X_out, float *Z_out, const int32_t *cu,
                            int n_seq, int64_t T_total, int H, float scale, const ChunkWs &ws,
                            cudaStream_t st, CkptOut ck = CkptOut(), int part = -1);
// Persistent prefill: shape eligibility (no device query), the grid for the current device (0:
// not possible there), the launch (clears the flags first) and its error word.
bool fused_shape(int64_t T_total, int n_seq, int H);
int fused_ctas(int n_seq, int H);
int fused_switch_chunks(int n_chunks, int n_chains, int grid);
cudaError_t launch_prefill_fused(const void *q, const void *k, const void *v, const void *la,
                                 const void *beta, const void *gate, void *out, const float *S0,
                                 float *S_final, int n_seq, int64_t T_total, int H, float scale,
                                 unsigned flags, const ChunkWs &ws, CkptOut ck, int grid,
                                 cudaStream_t st);
cudaError_t fused_take_error(unsigned *bits);
cudaError_t tc_take_error(unsigned *bits);        // card and state-pass words together
cudaError_t state_tc_take_error(unsigned *bits);  // the state pass's word alone

// chunked backward pass (kda_bwd.cu)
size_t chunk_bwd_ws_bytes(int64_t T_total, int n_seq, int H, int dk, int dv);
cudaError_t launch_chunk_bwd(const void *q, const void *k, const void *v, const void *la,
                             const void *beta, const void *gate, const float *S0,
                             const void *d_out, const float *dSf, void *dq, void *dk, void *dv,
                             void *dla, void *dbeta, void *dgate, float *dS0, const int32_t *cu,
                             int n_seq, int64_t T_total, int H, int dk_, int dv_, float scale,
                             unsigned flags, kda_dtype dt, void *ws, cudaStream_t st);

// The library's second stream on the current device (created once, non-blocking).
cudaError_t side_stream(cudaStream_t *out);

// Sets the calling thread's kda_last_error_string() message; returns `st`.
kda_status api_fail(kda_status st, const char *fmt, ...);

// Read-and-clear of each translation unit's device error word.
cudaError_t chunk_take_error(unsigned *bits);
cudaError_t decode_take_error(unsigned *bits);
cudaError_t scan_take_error(unsigned *bits);
cudaError_t bwd_take_error(unsigned *bits);
cudaError_t selftest_take_error(unsigned *bits);

}  // namespace kda
