// libkda C ABI: argument validation, workspace carving and launches.
// Every check here runs before any launch, so a rejected call has no effect.
#include <cuda_runtime.h>
#include <stdarg.h>

#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "../../include/kda.h"
#include "kda_common.cuh"

namespace {

thread_local char g_msg[512] = "no error";

// caller-owned events recorded around each launch (tracing), per host thread
constexpr int kMaxTrace = 8;
thread_local cudaEvent_t g_tr_begin[kMaxTrace], g_tr_end[kMaxTrace];
thread_local int g_tr_n = 0;

// Records begin/end events around the idx-th launch of an entry point.
struct Tracer {
  cudaStream_t st;
  int idx = 0;
  explicit Tracer(cudaStream_t s) : st(s) {}
  template <typename F>
  cudaError_t operator()(F &&launch) {
    return at(st, launch);
  }
  // a launch on another stream than the entry point's: its events go on that stream
  template <typename F>
  cudaError_t at(cudaStream_t on_stream, F &&launch) {
    const int i = idx++;
    const bool on = i < g_tr_n;
    if (on) cudaEventRecord(g_tr_begin[i], on_stream);
    cudaError_t e = launch();
    if (on) cudaEventRecord(g_tr_end[i], on_stream);
    return e;
  }
};

kda_status fail(kda_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

kda_status cuda_status(cudaError_t e, const char *where) {
  if (e == cudaSuccess) return KDA_OK;
  return fail(KDA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

bool shape_ok(int dk, int dv) { return (dk == 64 || dk == 128) && (dv == 64 || dv == 128); }

#define KDA_REQUIRE(cond, st, ...) \
  do {                             \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

kda_status check_ptr(const void *p, const char *name, bool required) {
  if (p == nullptr) {
    if (required) return fail(KDA_ERR_INVALID_ARG, "%s must not be NULL", name);
    return KDA_OK;
  }
  if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return KDA_OK;
}

#define KDA_CHECK_PTR(p, req)                       \
  do {                                              \
    kda_status s_ = check_ptr((p), #p, (req));      \
    if (s_ != KDA_OK) return s_;                    \
  } while (0)

kda_status common_checks(int64_t T_total, int n_seq, int H, int dk, int dv, int chunk,
                         kda_dtype dtype, const int32_t *cu) {
  KDA_REQUIRE(T_total >= 0 && n_seq >= 0 && H > 0, KDA_ERR_INVALID_ARG,
              "negative size (T_total=%lld n_seq=%d H=%d)", (long long)T_total, n_seq, H);
  KDA_REQUIRE(dtype == KDA_DTYPE_F32 || dtype == KDA_DTYPE_BF16, KDA_ERR_UNSUPPORTED,
              "dtype %d not supported", (int)dtype);
  KDA_REQUIRE(shape_ok(dk, dv), KDA_ERR_UNSUPPORTED, "dk=%d dv=%d: only 64 or 128", dk, dv);
  KDA_REQUIRE(chunk == kda::kChunk, KDA_ERR_UNSUPPORTED, "chunk=%d: only 64", chunk);
  KDA_REQUIRE(T_total < (int64_t)INT32_MAX, KDA_ERR_UNSUPPORTED, "T_total too large");
  KDA_REQUIRE((int64_t)n_seq * H < (int64_t)INT32_MAX / 4, KDA_ERR_UNSUPPORTED, "too many chains");
  if (cu == nullptr && n_seq > 0)
    KDA_REQUIRE(T_total % n_seq == 0, KDA_ERR_INVALID_ARG,
                "cu_seqlens is NULL but T_total=%lld is not a multiple of n_seq=%d",
                (long long)T_total, n_seq);
  if (cu == nullptr && n_seq == 0)
    KDA_REQUIRE(T_total == 0, KDA_ERR_INVALID_ARG, "n_seq=0 with T_total>0");
  return KDA_OK;
}

}  // namespace

namespace kda {
// Library-owned stream (one per device): the trailing cards of a split prefill, and the
// backward's work beside its forward replay.
cudaError_t side_stream(cudaStream_t *out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static cudaStream_t streams[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (streams[dev] == nullptr) {
    cudaStream_t s = nullptr;
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
    streams[dev] = s;
  }
  *out = streams[dev];
  return cudaSuccess;
}

// Sets this thread's kda_last_error_string() message and returns `st`.
kda_status api_fail(kda_status st, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}
}  // namespace kda

constexpr unsigned kKnownFlags = KDA_QK_L2NORM | KDA_DEBUG_CHECK | KDA_GATE_LOGITS;

extern "C" {

const char *kda_version(void) { return "libkda 0.1 sm_103a"; }

const char *kda_last_error_string(void) { return g_msg; }

size_t kda_chunk_fwd_workspace_size(int64_t T_total, int n_seq, int H, int dk, int dv,
                                    int chunk, kda_dtype dtype) {
  if (common_checks(T_total, n_seq, H, dk, dv, chunk, dtype, (const int32_t *)1) != KDA_OK)
    return 0;
  if (kda::tc_path(dk, dv, dtype)) return kda::tc_ws_bytes(T_total, n_seq, H);
  return kda::chunk_ws_bytes(T_total, n_seq, H, dk, dv);
}

int kda_chunk_fwd_launches(int64_t T_total, int n_seq, int H, int dk, int dv, int chunk,
                           kda_dtype dtype, int varlen) {
  if (common_checks(T_total, n_seq, H, dk, dv, chunk, dtype, (const int32_t *)1) != KDA_OK)
    return 0;
  if (n_seq == 0) return 0;
  const bool tc = kda::tc_path(dk, dv, dtype);
  if (tc && !varlen && kda::fused_shape(T_total, n_seq, H) && kda::fused_ctas(n_seq, H) > 0)
    return 1;  // the persistent prefill
  const int table = (!tc || varlen) ? 1 : 0;
  const int parts = tc ? kda::tc_split_parts(T_total, n_seq, H) : 0;
  return table + (parts > 1 ? 2 * parts : 2);
}

size_t kda_segment_summary_workspace_size(int64_t T_total, int n_seg, int H, int dk, int dv,
                                          int chunk, kda_dtype dtype) {
  return kda_chunk_fwd_workspace_size(T_total, n_seg, H, dk, dv, chunk, dtype);
}

}  // extern "C"

// Tensor-core prefill split into ws.nparts parts per sequence, after the chunk table. For three:
//   stream s:     cards 0 -> state pass 0 -> state pass 1 -> state pass 2
//   card stream:              cards 1        cards 2
// Part p's cards run beside the state pass over part p - 1. They wait for the state pass over
// part p - 2, so that they become ready together with the pass over part p - 1, which is
// enqueued first: the pass's CTAs are placed on the SMs the earlier pass leaves before the
// cards take the rest. Events fork the card stream off s and join it back, so the call stays
// ordered on s (and can be captured).
static kda_status split_prefill(const void *q, const void *k, const void *v,
                                const void *log_alpha, const void *beta, const void *gate,
                                void *out, const float *initial_state, float *final_state,
                                kda::CkptOut ck, const int32_t *cu_seqlens, int n_seq,
                                int64_t T_total, int H, float scale, unsigned flags,
                                const kda::ChunkWs &ws, cudaStream_t s, Tracer &tr) {
  cudaStream_t side = nullptr;
  kda_status st = cuda_status(kda::side_stream(&side), "card stream");
  if (st != KDA_OK) return st;
  const int K = ws.nparts;
  // per part: its cards are built (card_ev) and its state pass is done (pass_ev); the join
  cudaEvent_t card_ev[kda::kMaxParts] = {}, pass_ev[kda::kMaxParts] = {}, join_ev = nullptr;
  auto make = [&](cudaEvent_t *e) {
    return cuda_status(cudaEventCreateWithFlags(e, cudaEventDisableTiming), "event");
  };
  for (int p = 0; p < K && st == KDA_OK; ++p) {
    st = make(&card_ev[p]);
    if (st == KDA_OK && p + 2 < K) st = make(&pass_ev[p]);
  }
  if (st == KDA_OK) st = make(&join_ev);
  auto cards = [&](int part, cudaStream_t on) {
    return cuda_status(tr.at(on, [&] {
                         return kda::launch_card_tc(q, k, v, log_alpha, beta, cu_seqlens, n_seq,
                                                    T_total, H, flags, ws, on, part);
                       }),
                       "chunk prep");
  };
  auto state = [&](int part) {
    return cuda_status(tr([&] {
                         return kda::launch_state_tc(0, flags, gate, out, initial_state,
                                                     final_state, nullptr, nullptr, cu_seqlens,
                                                     n_seq, T_total, H, scale, ws, s, ck, part);
                       }),
                       "state pass");
  };
  auto record = [&](cudaEvent_t e, cudaStream_t on) {
    return cuda_status(cudaEventRecord(e, on), "event record");
  };
  auto wait = [&](cudaStream_t on, cudaEvent_t e) {
    return cuda_status(cudaStreamWaitEvent(on, e, 0), "stream wait");
  };
  bool forked = false;
  if (st == KDA_OK) st = cards(0, s);
  if (st == KDA_OK) st = record(card_ev[0], s);
  if (st == KDA_OK) st = state(0);
  if (st == KDA_OK) {
    st = wait(side, card_ev[0]);
    forked = st == KDA_OK;
  }
  for (int p = 1; p < K && st == KDA_OK; ++p) {
    if (p >= 2) st = wait(side, pass_ev[p - 2]);
    if (st == KDA_OK) st = cards(p, side);
    if (st == KDA_OK) st = record(card_ev[p], side);
    if (st == KDA_OK && p + 1 < K) st = record(pass_ev[p - 1], s);
    if (st == KDA_OK) st = wait(s, card_ev[p]);
    if (st == KDA_OK) st = state(p);
  }
  if (forked && st != KDA_OK) {  // join the card stream back into s after a failed step
    kda_status j = record(join_ev, side);
    if (j == KDA_OK) wait(s, join_ev);
  }
  for (cudaEvent_t e : card_ev)
    if (e) cudaEventDestroy(e);
  for (cudaEvent_t e : pass_ev)
    if (e) cudaEventDestroy(e);
  if (join_ev) cudaEventDestroy(join_ev);
  return st;
}

// kda_chunk_fwd and kda_chunk_fwd_checkpoints: one path, the checkpoint output optional.
static kda_status chunk_fwd_impl(const void *q, const void *k, const void *v,
                                 const void *log_alpha, const void *beta, const void *gate,
                                 void *out, const float *initial_state, float *final_state,
                                 kda::CkptOut ck, const int32_t *cu_seqlens, int n_seq,
                                 int64_t T_total, int H, int dk, int dv, int chunk, float scale,
                                 unsigned flags, kda_dtype dtype, void *workspace,
                                 size_t workspace_bytes, kda_stream_t stream) {
  kda_status st = common_checks(T_total, n_seq, H, dk, dv, chunk, dtype, cu_seqlens);
  if (st != KDA_OK) return st;
  KDA_REQUIRE((flags & ~kKnownFlags) == 0, KDA_ERR_INVALID_ARG,
              "unknown flag bits 0x%x", flags);
  const bool tokens = T_total > 0;
  KDA_CHECK_PTR(q, tokens);
  KDA_CHECK_PTR(k, tokens);
  KDA_CHECK_PTR(v, tokens);
  KDA_CHECK_PTR(log_alpha, tokens);
  KDA_CHECK_PTR(beta, false);
  KDA_REQUIRE(!tokens || beta != nullptr, KDA_ERR_INVALID_ARG, "beta must not be NULL");
  KDA_CHECK_PTR(gate, false);
  KDA_CHECK_PTR(out, tokens);
  KDA_CHECK_PTR(initial_state, false);
  KDA_CHECK_PTR(final_state, false);
  KDA_REQUIRE(cu_seqlens == nullptr || ((uintptr_t)cu_seqlens & 3u) == 0, KDA_ERR_INVALID_ARG,
              "cu_seqlens is not 4-byte aligned");
  if (n_seq == 0) return KDA_OK;
  const bool tc = kda::tc_path(dk, dv, dtype);
  const size_t need = tc ? kda::tc_ws_bytes(T_total, n_seq, H)
                         : kda::chunk_ws_bytes(T_total, n_seq, H, dk, dv);
  KDA_REQUIRE(workspace != nullptr && workspace_bytes >= need, KDA_ERR_WORKSPACE,
              "workspace %zu bytes, need %zu", workspace_bytes, need);
  KDA_REQUIRE(((uintptr_t)workspace & 255u) == 0, KDA_ERR_INVALID_ARG,
              "workspace is not 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  Tracer tr(s);
  kda::ChunkWs ws = tc ? kda::tc_ws_carve(workspace, T_total, n_seq, H)
                       : kda::chunk_ws_carve(workspace, T_total, n_seq, H, dk, dv);
  // fixed lengths, few chains: cards and state pass in one persistent launch; if the device
  // cannot run it (too few SMs, no cooperative launch), the split schedule below
  if (tc && cu_seqlens == nullptr && kda::fused_shape(T_total, n_seq, H)) {
    const int grid = kda::fused_ctas(n_seq, H);
    if (grid > 0) {
      cudaError_t e = tr([&] {
        return kda::launch_prefill_fused(q, k, v, log_alpha, beta, gate, out, initial_state,
                                         final_state, n_seq, T_total, H, scale, flags, ws, ck,
                                         grid, s);
      });
      if (e == cudaSuccess) return KDA_OK;
      if (e != cudaErrorCooperativeLaunchTooLarge) return cuda_status(e, "persistent prefill");
      cudaGetLastError();  // not resident at once on this device: take the split schedule
      tr.idx = 0;
    }
  }
  // the tensor-core kernels index fixed-length batches (no cu_seqlens) without the chunk table
  if (!tc || cu_seqlens != nullptr) {
    st = cuda_status(
        tr([&] { return kda::launch_chunk_table(cu_seqlens, n_seq, T_total, ws, s); }),
        "chunk table");
    if (st != KDA_OK) return st;
  }
  if (tc && ws.nparts > 1)
    return split_prefill(q, k, v, log_alpha, beta, gate, out, initial_state, final_state, ck,
                         cu_seqlens, n_seq, T_total, H, scale, flags, ws, s, tr);
  st = cuda_status(tr([&] {
                     return tc ? kda::launch_card_tc(q, k, v, log_alpha, beta, cu_seqlens, n_seq,
                                                     T_total, H, flags, ws, s)
                               : kda::launch_prep(q, k, v, log_alpha, beta, cu_seqlens, n_seq,
                                                  T_total, H, dk, dv, flags, dtype, ws, true, s);
                   }),
                   "chunk prep");
  if (st != KDA_OK) return st;
  return cuda_status(tr([&] {
                       return tc ? kda::launch_state_tc(0, flags, gate, out, initial_state, final_state,
                                                        nullptr, nullptr, cu_seqlens, n_seq,
                                                        T_total, H, scale, ws, s, ck)
                                 : kda::launch_state_pass(0, flags, gate, out, initial_state,
                                                          final_state, nullptr, nullptr,
                                                          cu_seqlens, n_seq, T_total, H, dk, dv,
                                                          scale, dtype, ws, s, ck);
                     }),
                     "state pass");
}

extern "C" {

kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const void *log_alpha,
                         const void *beta, const void *gate, void *out,
                         const float *initial_state, float *final_state,
                         const int32_t *cu_seqlens, int n_seq, int64_t T_total, int H, int dk,
                         int dv, int chunk, float scale, unsigned flags, kda_dtype dtype,
                         void *workspace, size_t workspace_bytes, kda_stream_t stream) {
  return chunk_fwd_impl(q, k, v, log_alpha, beta, gate, out, initial_state, final_state,
                        kda::CkptOut(), cu_seqlens, n_seq, T_total, H, dk, dv, chunk, scale,
                        flags, dtype, workspace, workspace_bytes, stream);
}

kda_status kda_chunk_fwd_checkpoints(
    const void *q, const void *k, const void *v, const void *log_alpha, const void *beta,
    const void *gate, void *out, const float *initial_state, float *final_state,
    float *checkpoints, int64_t checkpoint_every, int checkpoints_per_seq,
    const int32_t *cu_seqlens, int n_seq, int64_t T_total, int H, int dk, int dv, int chunk,
    float scale, unsigned flags, kda_dtype dtype, void *workspace, size_t workspace_bytes,
    kda_stream_t stream) {
  KDA_REQUIRE(checkpoint_every > 0 && chunk > 0 && checkpoint_every % chunk == 0 &&
                  checkpoint_every / chunk <= (int64_t)INT32_MAX,
              KDA_ERR_INVALID_ARG, "checkpoint_every=%lld: a positive multiple of chunk=%d",
              (long long)checkpoint_every, chunk);
  KDA_REQUIRE(checkpoints_per_seq >= 0, KDA_ERR_INVALID_ARG, "checkpoints_per_seq=%d < 0",
              checkpoints_per_seq);
  KDA_CHECK_PTR(checkpoints, checkpoints_per_seq > 0);
  kda::CkptOut ck;
  if (checkpoints_per_seq > 0) {
    ck.ptr = checkpoints;
    ck.every_chunks = (int)(checkpoint_every / chunk);
    ck.per_seq = checkpoints_per_seq;
  }
  return chunk_fwd_impl(q, k, v, log_alpha, beta, gate, out, initial_state, final_state, ck,
                        cu_seqlens, n_seq, T_total, H, dk, dv, chunk, scale, flags, dtype,
                        workspace, workspace_bytes, stream);
}

size_t kda_chunk_bwd_workspace_size(int64_t T_total, int n_seq, int H, int dk, int dv,
                                    int chunk, kda_dtype dtype) {
  if (common_checks(T_total, n_seq, H, dk, dv, chunk, dtype, (const int32_t *)1) != KDA_OK)
    return 0;
  return kda::chunk_bwd_ws_bytes(T_total, n_seq, H, dk, dv);
}

kda_status kda_chunk_bwd(const void *q, const void *k, const void *v, const void *log_alpha,
                         const void *beta, const void *gate, const float *initial_state,
                         const void *d_out, const float *d_final_state, void *d_q, void *d_k,
                         void *d_v, void *d_log_alpha, void *d_beta, void *d_gate,
                         float *d_initial_state, const int32_t *cu_seqlens, int n_seq,
                         int64_t T_total, int H, int dk, int dv, int chunk, float scale,
                         unsigned flags, kda_dtype dtype, void *workspace,
                         size_t workspace_bytes, kda_stream_t stream) {
  kda_status st = common_checks(T_total, n_seq, H, dk, dv, chunk, dtype, cu_seqlens);
  if (st != KDA_OK) return st;
  KDA_REQUIRE((flags & ~kKnownFlags) == 0, KDA_ERR_INVALID_ARG,
              "unknown flag bits 0x%x", flags);
  const bool tokens = T_total > 0;
  KDA_CHECK_PTR(q, tokens);
  KDA_CHECK_PTR(k, tokens);
  KDA_CHECK_PTR(v, tokens);
  KDA_CHECK_PTR(log_alpha, tokens);
  KDA_REQUIRE(!tokens || beta != nullptr, KDA_ERR_INVALID_ARG, "beta must not be NULL");
  KDA_CHECK_PTR(gate, false);
  KDA_CHECK_PTR(initial_state, false);
  KDA_CHECK_PTR(d_out, tokens);
  KDA_CHECK_PTR(d_final_state, false);
  KDA_CHECK_PTR(d_q, tokens);
  KDA_CHECK_PTR(d_k, tokens);
  KDA_CHECK_PTR(d_v, tokens);
  KDA_CHECK_PTR(d_log_alpha, tokens);
  KDA_REQUIRE(!tokens || d_beta != nullptr, KDA_ERR_INVALID_ARG, "d_beta must not be NULL");
  KDA_CHECK_PTR(d_gate, false);
  KDA_REQUIRE(gate != nullptr || d_gate == nullptr, KDA_ERR_INVALID_ARG,
              "d_gate given without gate");
  KDA_CHECK_PTR(d_initial_state, false);
  KDA_REQUIRE(cu_seqlens == nullptr || ((uintptr_t)cu_seqlens & 3u) == 0, KDA_ERR_INVALID_ARG,
              "cu_seqlens is not 4-byte aligned");
  if (n_seq == 0) return KDA_OK;
  const size_t need = kda::chunk_bwd_ws_bytes(T_total, n_seq, H, dk, dv);
  KDA_REQUIRE(workspace != nullptr && workspace_bytes >= need, KDA_ERR_WORKSPACE,
              "workspace %zu bytes, need %zu", workspace_bytes, need);
  KDA_REQUIRE(((uintptr_t)workspace & 255u) == 0, KDA_ERR_INVALID_ARG,
              "workspace is not 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  Tracer tr(s);
  return cuda_status(tr([&] {
                       return kda::launch_chunk_bwd(
                           q, k, v, log_alpha, beta, gate, initial_state, d_out, d_final_state,
                           d_q, d_k, d_v, d_log_alpha, d_beta, d_gate, d_initial_state,
                           cu_seqlens, n_seq, T_total, H, dk, dv, scale, flags, dtype, workspace,
                           s);
                     }),
                     "backward");
}

kda_status kda_decode_step(const void *q, const void *k, const void *v, const void *log_alpha,
                           const void *beta, const void *gate, void *out, float *state,
                           const int32_t *state_slot, int n_slots, int N, int H, int dk, int dv,
                           float scale, unsigned flags, kda_dtype dtype, kda_stream_t stream) {
  KDA_REQUIRE(N >= 0 && H > 0 && n_slots >= 0, KDA_ERR_INVALID_ARG,
              "negative size (N=%d H=%d n_slots=%d)", N, H, n_slots);
  KDA_REQUIRE(dtype == KDA_DTYPE_F32 || dtype == KDA_DTYPE_BF16, KDA_ERR_UNSUPPORTED,
              "dtype %d not supported", (int)dtype);
  KDA_REQUIRE(shape_ok(dk, dv), KDA_ERR_UNSUPPORTED, "dk=%d dv=%d: only 64 or 128", dk, dv);
  KDA_REQUIRE((flags & ~kKnownFlags) == 0, KDA_ERR_INVALID_ARG,
              "unknown flag bits 0x%x", flags);
  KDA_REQUIRE((int64_t)N * H < (int64_t)INT32_MAX, KDA_ERR_UNSUPPORTED, "N*H too large");
  if (N == 0) return KDA_OK;
  KDA_REQUIRE(state_slot != nullptr || n_slots >= N, KDA_ERR_INVALID_ARG,
              "n_slots=%d < N=%d without a slot map", n_slots, N);
  KDA_CHECK_PTR(q, true);
  KDA_CHECK_PTR(k, true);
  KDA_CHECK_PTR(v, true);
  KDA_CHECK_PTR(log_alpha, true);
  KDA_REQUIRE(beta != nullptr, KDA_ERR_INVALID_ARG, "beta must not be NULL");
  KDA_CHECK_PTR(gate, false);
  KDA_CHECK_PTR(out, true);
  KDA_CHECK_PTR(state, true);
  KDA_REQUIRE(state_slot == nullptr || ((uintptr_t)state_slot & 3u) == 0, KDA_ERR_INVALID_ARG,
              "state_slot is not 4-byte aligned");
  Tracer tr((cudaStream_t)stream);
  return cuda_status(tr([&] {
                       return kda::launch_decode(q, k, v, log_alpha, beta, gate, out, state,
                                                 state_slot, n_slots, N, H, dk, dv, scale, flags,
                                                 dtype, (cudaStream_t)stream);
                     }),
                     "decode");
}

kda_status kda_segment_summary(const void *k, const void *v, const void *log_alpha,
                               const void *beta, const int32_t *cu_segs, int n_seg,
                               int64_t T_total, int H, int dk, int dv, int chunk, unsigned flags,
                               kda_dtype dtype, float *X_out, float *Z_out, void *workspace,
                               size_t workspace_bytes, kda_stream_t stream) {
  kda_status st = common_checks(T_total, n_seg, H, dk, dv, chunk, dtype, cu_segs);
  if (st != KDA_OK) return st;
  KDA_REQUIRE((flags & ~kKnownFlags) == 0, KDA_ERR_INVALID_ARG,
              "unknown flag bits 0x%x", flags);
  const bool tokens = T_total > 0;
  KDA_CHECK_PTR(k, tokens);
  KDA_CHECK_PTR(v, tokens);
  KDA_CHECK_PTR(log_alpha, tokens);
  KDA_REQUIRE(!tokens || beta != nullptr, KDA_ERR_INVALID_ARG, "beta must not be NULL");
  KDA_CHECK_PTR(X_out, n_seg > 0);
  KDA_CHECK_PTR(Z_out, n_seg > 0);
  KDA_REQUIRE(cu_segs == nullptr || ((uintptr_t)cu_segs & 3u) == 0, KDA_ERR_INVALID_ARG,
              "cu_segs is not 4-byte aligned");
  if (n_seg == 0) return KDA_OK;
  const bool tc = kda::tc_path(dk, dv, dtype);
  const size_t need = tc ? kda::tc_ws_bytes(T_total, n_seg, H)
                         : kda::chunk_ws_bytes(T_total, n_seg, H, dk, dv);
  KDA_REQUIRE(workspace != nullptr && workspace_bytes >= need, KDA_ERR_WORKSPACE,
              "workspace %zu bytes, need %zu", workspace_bytes, need);
  KDA_REQUIRE(((uintptr_t)workspace & 255u) == 0, KDA_ERR_INVALID_ARG,
              "workspace is not 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  Tracer tr(s);
  kda::ChunkWs ws = tc ? kda::tc_ws_carve(workspace, T_total, n_seg, H)
                       : kda::chunk_ws_carve(workspace, T_total, n_seg, H, dk, dv);
  st = cuda_status(tr([&] { return kda::launch_chunk_table(cu_segs, n_seg, T_total, ws, s); }),
                   "chunk table");
  if (st != KDA_OK) return st;
  st = cuda_status(tr([&] {
                     return tc ? kda::launch_card_tc(k, k, v, log_alpha, beta, cu_segs, n_seg,
                                                     T_total, H, flags, ws, s)
                               : kda::launch_prep(k, k, v, log_alpha, beta, cu_segs, n_seg,
                                                  T_total, H, dk, dv, flags, dtype, ws, false, s);
                   }),
                   "chunk prep");
  if (st != KDA_OK) return st;
  return cuda_status(tr([&] {
                       return tc ? kda::launch_state_tc(1, flags, nullptr, nullptr, nullptr, nullptr,
                                                        X_out, Z_out, cu_segs, n_seg, T_total, H,
                                                        1.0f, ws, s)
                                 : kda::launch_state_pass(1, flags, nullptr, nullptr, nullptr, nullptr,
                                                          X_out, Z_out, cu_segs, n_seg, T_total,
                                                          H, dk, dv, 1.0f, dtype, ws, s);
                     }),
                     "summary state pass");
}

size_t kda_segmented_fwd_workspace_size(int64_t T_total, int n_seg, int H, int dk, int dv,
                                        int chunk, kda_dtype dtype) {
  const size_t base = kda_chunk_fwd_workspace_size(T_total, n_seg, H, dk, dv, chunk, dtype);
  if (base == 0) return 0;
  const size_t per = (size_t)n_seg * H;
  return base + kda::align_up(sizeof(float) * per * dk * dk, 256) +
         2 * kda::align_up(sizeof(float) * per * dk * dv, 256);
}

kda_status kda_segmented_fwd(const void *q, const void *k, const void *v, const void *log_alpha,
                             const void *beta, const void *gate, void *out,
                             const float *initial_state, float *final_state,
                             float *segment_entry_states, const int32_t *cu_segs, int n_seg,
                             int64_t T_total, int H, int dk, int dv, int chunk, float scale,
                             unsigned flags, kda_dtype dtype, void *workspace,
                             size_t workspace_bytes, kda_stream_t stream) {
  kda_status st = common_checks(T_total, n_seg, H, dk, dv, chunk, dtype, cu_segs);
  if (st != KDA_OK) return st;
  KDA_REQUIRE(n_seg >= 1, KDA_ERR_INVALID_ARG, "n_seg=%d: at least one segment", n_seg);
  KDA_REQUIRE((flags & ~kKnownFlags) == 0, KDA_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  const bool tokens = T_total > 0;
  KDA_CHECK_PTR(q, tokens);
  KDA_CHECK_PTR(k, tokens);
  KDA_CHECK_PTR(v, tokens);
  KDA_CHECK_PTR(log_alpha, tokens);
  KDA_REQUIRE(!tokens || beta != nullptr, KDA_ERR_INVALID_ARG, "beta must not be NULL");
  KDA_CHECK_PTR(gate, false);
  KDA_CHECK_PTR(out, tokens);
  KDA_CHECK_PTR(initial_state, false);
  KDA_CHECK_PTR(final_state, false);
  KDA_CHECK_PTR(segment_entry_states, false);
  KDA_REQUIRE(cu_segs == nullptr || ((uintptr_t)cu_segs & 3u) == 0, KDA_ERR_INVALID_ARG,
              "cu_segs is not 4-byte aligned");
  const size_t need = kda_segmented_fwd_workspace_size(T_total, n_seg, H, dk, dv, chunk, dtype);
  KDA_REQUIRE(workspace != nullptr && workspace_bytes >= need, KDA_ERR_WORKSPACE,
              "workspace %zu bytes, need %zu", workspace_bytes, need);
  KDA_REQUIRE(((uintptr_t)workspace & 255u) == 0, KDA_ERR_INVALID_ARG,
              "workspace is not 256-byte aligned");
  cudaStream_t s = (cudaStream_t)stream;
  Tracer tr(s);
  const bool tc = kda::tc_path(dk, dv, dtype);
  const size_t base = tc ? kda::tc_ws_bytes(T_total, n_seg, H)
                         : kda::chunk_ws_bytes(T_total, n_seg, H, dk, dv);
  kda::ChunkWs ws = tc ? kda::tc_ws_carve(workspace, T_total, n_seg, H)
                       : kda::chunk_ws_carve(workspace, T_total, n_seg, H, dk, dv);
  const size_t per = (size_t)n_seg * H;
  float *X = (float *)((char *)workspace + kda::align_up(base, 256));
  float *Z = (float *)((char *)X + kda::align_up(sizeof(float) * per * dk * dk, 256));
  float *E = segment_entry_states
                 ? segment_entry_states
                 : (float *)((char *)Z + kda::align_up(sizeof(float) * per * dk * dv, 256));
  st = cuda_status(tr([&] { return kda::launch_chunk_table(cu_segs, n_seg, T_total, ws, s); }),
                   "chunk table");
  if (st != KDA_OK) return st;
  // one set of update cards serves both the summaries and the re-run
  st = cuda_status(tr([&] {
                     return tc ? kda::launch_card_tc(q, k, v, log_alpha, beta, cu_segs, n_seg,
                                                     T_total, H, flags, ws, s)
                               : kda::launch_prep(q, k, v, log_alpha, beta, cu_segs, n_seg,
                                                  T_total, H, dk, dv, flags, dtype, ws, true, s);
                   }),
                   "chunk prep");
  if (st != KDA_OK) return st;
  st = cuda_status(tr([&] {
                     return tc ? kda::launch_state_tc(1, flags, nullptr, nullptr, nullptr, nullptr,
                                                      X, Z, cu_segs, n_seg, T_total, H, 1.0f, ws,
                                                      s)
                               : kda::launch_state_pass(1, flags, nullptr, nullptr, nullptr,
                                                        nullptr, X, Z, cu_segs, n_seg, T_total,
                                                        H, dk, dv, 1.0f, dtype, ws, s);
                   }),
                   "segment summaries");
  if (st != KDA_OK) return st;
  st = cuda_status(tr([&] {
                     return kda::launch_scan_combine(X, Z, n_seg, H, dk, dv, initial_state, E,
                                                     final_state, s);
                   }),
                   "scan combine");
  if (st != KDA_OK) return st;
  return cuda_status(tr([&] {
                       return tc ? kda::launch_state_tc(0, flags, gate, out, E, nullptr, nullptr,
                                                        nullptr, cu_segs, n_seg, T_total, H,
                                                        scale, ws, s)
                                 : kda::launch_state_pass(0, flags, gate, out, E, nullptr,
                                                          nullptr, nullptr, cu_segs, n_seg,
                                                          T_total, H, dk, dv, scale, dtype, ws,
                                                          s);
                     }),
                     "segment re-run");
}

kda_status kda_scan_combine(const float *X, const float *Z, int n_seg, int H, int dk, int dv,
                            const float *S_init, float *S_entry_out, float *S_final_out,
                            kda_stream_t stream) {
  KDA_REQUIRE(n_seg >= 0 && H > 0, KDA_ERR_INVALID_ARG, "negative size (n_seg=%d H=%d)", n_seg,
              H);
  KDA_REQUIRE(shape_ok(dk, dv), KDA_ERR_UNSUPPORTED, "dk=%d dv=%d: only 64 or 128", dk, dv);
  KDA_CHECK_PTR(X, n_seg > 0);
  KDA_CHECK_PTR(Z, n_seg > 0);
  KDA_CHECK_PTR(S_init, false);
  KDA_CHECK_PTR(S_entry_out, false);
  KDA_CHECK_PTR(S_final_out, false);
  if (S_entry_out == nullptr && S_final_out == nullptr) return KDA_OK;
  Tracer tr((cudaStream_t)stream);
  return cuda_status(tr([&] {
                       return kda::launch_scan_combine(X, Z, n_seg, H, dk, dv, S_init,
                                                       S_entry_out, S_final_out,
                                                       (cudaStream_t)stream);
                     }),
                     "scan combine");
}

kda_status kda_trace_events(void *const *begin, void *const *end, int n) {
  KDA_REQUIRE(n >= 0 && n <= kMaxTrace, KDA_ERR_INVALID_ARG, "n=%d: 0..%d events", n, kMaxTrace);
  KDA_REQUIRE(n == 0 || (begin != nullptr && end != nullptr), KDA_ERR_INVALID_ARG,
              "begin/end must not be NULL");
  for (int i = 0; i < n; ++i) {
    KDA_REQUIRE(begin[i] != nullptr && end[i] != nullptr, KDA_ERR_INVALID_ARG,
                "event %d is NULL", i);
    g_tr_begin[i] = (cudaEvent_t)begin[i];
    g_tr_end[i] = (cudaEvent_t)end[i];
  }
  g_tr_n = n;
  return KDA_OK;
}

kda_status kda_get_error(kda_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "stream synchronize");
  unsigned a = 0, b = 0, c = 0, d = 0, f = 0, g = 0, r = 0;
  if ((e = kda::chunk_take_error(&a)) != cudaSuccess) return cuda_status(e, "error word");
  if ((e = kda::decode_take_error(&b)) != cudaSuccess) return cuda_status(e, "error word");
  if ((e = kda::tc_take_error(&c)) != cudaSuccess) return cuda_status(e, "error word");
  if ((e = kda::scan_take_error(&d)) != cudaSuccess) return cuda_status(e, "error word");
  if ((e = kda::selftest_take_error(&f)) != cudaSuccess) return cuda_status(e, "error word");
  if ((e = kda::fused_take_error(&g)) != cudaSuccess) return cuda_status(e, "error word");
  if ((e = kda::bwd_take_error(&r)) != cudaSuccess) return cuda_status(e, "error word");
  const unsigned bits = a | b | c | d | f | g | r;
  if (bits & kda::kErrTimeout) return fail(KDA_ERR_TIMEOUT, "a bounded device wait ran out");
  if (bits & kda::kErrBadSeqlens)
    return fail(KDA_ERR_INVALID_ARG, "malformed cu_seqlens / cu_segs or state_slot on device");
  if (bits & kda::kErrPrecondition)
    return fail(KDA_ERR_PRECONDITION, "log_alpha < -0.6953125 or beta outside [0,1]");
  return KDA_OK;
}

}  // extern "C"
