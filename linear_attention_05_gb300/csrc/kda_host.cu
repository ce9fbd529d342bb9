// kda_chunk_fwd_host: the chunked prefill on host-resident (page-locked) buffers, the copies
// over the host link overlapped with the compute, one sequence at a time.
//
// Sequence s's inputs go to the device on the library's copy-in stream; its kda_chunk_fwd call
// runs on the caller's stream once they are there; its outputs come back on the copy-out stream
// once the call is done. So sequence s + 1 is copied in while s is computed and s - 1 copied
// back. The last sequence is computed in time slices, each starting from the state the slice
// before left (the fp32 hand-over is exact, so the bits do not change), so that only one
// slice's compute and copy back are left after the last copy in. On a GB300 the host link
// moves about 211 GB/s in and 193 GB/s out, 342 GB/s both ways at once: the copies in bound a
// call.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_common.cuh"

namespace {

constexpr int kMaxTailSlices = 16;

size_t elem_bytes(kda_dtype dt) { return dt == KDA_DTYPE_BF16 ? 2 : 4; }

// Device buffer: per tensor one 256-byte aligned slot per sequence (so every pointer handed
// to kda_chunk_fwd is aligned whatever the sequence length), the states, the two states
// handed between the last sequence's slices, then one sequence's workspace.
struct HostLayout {
  int64_t len;                    // tokens per sequence
  size_t stride_k, stride_v, stride_b;  // bytes of one sequence's slot: rows of dk, dv, 1
  size_t q, k, v, la, beta, gate, out, s0, fs, mid[2], ws, ws_bytes, total;
};

bool shape_supported(int dk, int dv, int chunk, kda_dtype dt) {
  return (dk == 64 || dk == 128) && (dv == 64 || dv == 128) && chunk == 64 &&
         (dt == KDA_DTYPE_BF16 || dt == KDA_DTYPE_F32);
}

// false: an invalid problem (the shape is checked before)
bool host_layout(int64_t T_total, int n_seq, int H, int dk, int dv, int chunk, kda_dtype dt,
                 int tail_slices, HostLayout *L) {
  if (n_seq <= 0 || H <= 0 || T_total < 0 || T_total % n_seq != 0) return false;
  if (tail_slices < 1 || tail_slices > kMaxTailSlices) return false;
  const int64_t len = T_total / n_seq;
  if (tail_slices > 1 && len % ((int64_t)chunk * tail_slices) != 0) return false;
  const size_t e = elem_bytes(dt), th = (size_t)len * H;
  const size_t st = (size_t)H * dk * dv * sizeof(float);
  L->len = len;
  L->stride_k = kda::align_up(th * dk * e, 256);
  L->stride_v = kda::align_up(th * dv * e, 256);
  L->stride_b = kda::align_up(th * e, 256);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += kda::align_up(bytes, 256);
    return o;
  };
  L->q = take(L->stride_k * n_seq);
  L->k = take(L->stride_k * n_seq);
  L->v = take(L->stride_v * n_seq);
  L->la = take(L->stride_k * n_seq);
  L->beta = take(L->stride_b * n_seq);
  L->gate = take(L->stride_v * n_seq);
  L->out = take(L->stride_v * n_seq);
  L->s0 = take(st * n_seq);
  L->fs = take(st * n_seq);
  L->mid[0] = take(st);
  L->mid[1] = take(st);
  const size_t w1 = kda_chunk_fwd_workspace_size(len, 1, H, dk, dv, chunk, dt);
  const size_t w2 = kda_chunk_fwd_workspace_size(len / tail_slices, 1, H, dk, dv, chunk, dt);
  if (w1 == 0 || w2 == 0) return false;
  L->ws_bytes = w1 > w2 ? w1 : w2;
  L->ws = take(L->ws_bytes);
  L->total = off;
  return true;
}

// page-locked host memory (pinned by cudaHostAlloc or registered by cudaHostRegister)
bool page_locked(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// Library-owned copy streams (one pair per device, for the process's lifetime).
cudaError_t copy_streams(cudaStream_t *in, cudaStream_t *out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static cudaStream_t s_in[kMaxDev] = {}, s_out[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  for (cudaStream_t *s : {&s_in[dev], &s_out[dev]}) {
    if (*s != nullptr) continue;
    e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *in = s_in[dev];
  *out = s_out[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t kda_chunk_fwd_host_buffer_size(int64_t T_total, int n_seq, int H, int dk, int dv,
                                      int chunk, kda_dtype dtype, int tail_slices) {
  HostLayout L;
  if (!shape_supported(dk, dv, chunk, dtype) ||
      !host_layout(T_total, n_seq, H, dk, dv, chunk, dtype, tail_slices, &L))
    return 0;
  return L.total;
}

kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v, const void *log_alpha,
                              const void *beta, const void *gate, void *out,
                              const float *initial_state, float *final_state, int n_seq,
                              int64_t T_total, int H, int dk, int dv, int chunk, float scale,
                              unsigned flags, kda_dtype dtype, int tail_slices,
                              void *device_buffer, size_t device_bytes, kda_stream_t stream) {
  using kda::api_fail;
  if (!shape_supported(dk, dv, chunk, dtype))
    return api_fail(KDA_ERR_UNSUPPORTED, "kda_chunk_fwd_host: dk=%d dv=%d chunk=%d dtype=%d", dk,
                    dv, chunk, (int)dtype);
  HostLayout L;
  if (!host_layout(T_total, n_seq, H, dk, dv, chunk, dtype, tail_slices, &L))
    return api_fail(KDA_ERR_INVALID_ARG,
                    "kda_chunk_fwd_host: n_seq=%d T_total=%lld H=%d tail_slices=%d: needs "
                    "n_seq > 0 sequences of equal length, tail_slices in 1..%d and, for "
                    "tail_slices > 1, lengths a multiple of 64 * tail_slices",
                    n_seq, (long long)T_total, H, tail_slices, kMaxTailSlices);
  if (device_buffer == nullptr || device_bytes < L.total)
    return api_fail(KDA_ERR_WORKSPACE, "kda_chunk_fwd_host: device buffer %zu bytes, need %zu",
                    device_bytes, L.total);
  if (((uintptr_t)device_buffer & 255u) != 0)
    return api_fail(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_host: device buffer not 256-byte aligned");
  const bool tokens = T_total > 0;
  const struct {
    const void *p;
    const char *name;
    bool required;
  } host[] = {{q, "q", tokens},       {k, "k", tokens},        {v, "v", tokens},
              {log_alpha, "log_alpha", tokens}, {beta, "beta", tokens}, {gate, "gate", false},
              {out, "out", tokens},   {initial_state, "initial_state", false},
              {final_state, "final_state", false}};
  for (const auto &h : host) {
    if (h.p == nullptr) {
      if (h.required) return api_fail(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_host: %s is NULL", h.name);
      continue;
    }
    if (!page_locked(h.p))
      return api_fail(KDA_ERR_INVALID_ARG, "kda_chunk_fwd_host: %s is not page-locked host memory",
                      h.name);
  }

  cudaStream_t s = (cudaStream_t)stream, s_in = nullptr, s_out = nullptr;
  cudaError_t ce = copy_streams(&s_in, &s_out);
  if (ce != cudaSuccess)
    return api_fail(KDA_ERR_CUDA, "kda_chunk_fwd_host: copy streams: %s", cudaGetErrorString(ce));
  // events: the call's start (on s), the two joins, then per slice "inputs in" and "computed"
  const int n_slices = n_seq - 1 + tail_slices;
  std::vector<cudaEvent_t> ev((size_t)3 + 2 * n_slices, nullptr);
  kda_status st = KDA_OK;
  auto ok = [&](cudaError_t e, const char *what) {
    if (st == KDA_OK && e != cudaSuccess)
      st = api_fail(KDA_ERR_CUDA, "kda_chunk_fwd_host: %s: %s", what, cudaGetErrorString(e));
    return st == KDA_OK;
  };
  for (cudaEvent_t &e : ev)
    if (!ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "event")) break;
  auto ev_in = [&](int i) { return ev[3 + 2 * (size_t)i]; };
  auto ev_done = [&](int i) { return ev[4 + 2 * (size_t)i]; };

  char *d = static_cast<char *>(device_buffer);
  const size_t e = elem_bytes(dtype), sb = (size_t)H * dk * dv * sizeof(float);
  bool forked = false;
  if (st == KDA_OK && ok(cudaEventRecord(ev[0], s), "event record") &&
      ok(cudaStreamWaitEvent(s_in, ev[0], 0), "stream wait") &&
      ok(cudaStreamWaitEvent(s_out, ev[0], 0), "stream wait"))
    forked = true;
  int slice = 0;
  for (int sq = 0; sq < n_seq && st == KDA_OK; ++sq) {
    const int parts = sq == n_seq - 1 ? tail_slices : 1;
    const int64_t tl = L.len / parts;
    for (int p = 0; p < parts && st == KDA_OK; ++p, ++slice) {
      // token-heads of the slice: host offset (packed) and device offset (sequence slot)
      const size_t h0 = ((size_t)sq * L.len + (size_t)p * tl) * H, dh0 = (size_t)p * tl * H;
      const size_t n = (size_t)tl * H;
      auto dev = [&](size_t base, size_t stride, size_t row) {
        return d + base + (size_t)sq * stride + dh0 * row * e;
      };
      auto copy_in = [&](size_t base, size_t stride, const void *hp, size_t row) {
        if (st != KDA_OK) return false;
        if (hp == nullptr || n == 0) return true;
        return ok(cudaMemcpyAsync(dev(base, stride, row), (const char *)hp + h0 * row * e,
                                  n * row * e, cudaMemcpyHostToDevice, s_in),
                  "copy in");
      };
      if (p == 0 && initial_state)
        ok(cudaMemcpyAsync(d + L.s0 + sq * sb, (const char *)initial_state + sq * sb, sb,
                           cudaMemcpyHostToDevice, s_in),
           "copy in");
      copy_in(L.q, L.stride_k, q, dk) && copy_in(L.k, L.stride_k, k, dk) &&
          copy_in(L.v, L.stride_v, v, dv) && copy_in(L.la, L.stride_k, log_alpha, dk) &&
          copy_in(L.beta, L.stride_b, beta, 1) && copy_in(L.gate, L.stride_v, gate, dv);
      if (!ok(cudaEventRecord(ev_in(slice), s_in), "event record") ||
          !ok(cudaStreamWaitEvent(s, ev_in(slice), 0), "stream wait"))
        break;
      // compute the slice on the caller's stream
      const float *entry = p == 0 ? (initial_state ? (const float *)(d + L.s0 + sq * sb) : nullptr)
                                  : (const float *)(d + L.mid[(p - 1) & 1]);
      float *exit = p == parts - 1 ? (float *)(d + L.fs + sq * sb) : (float *)(d + L.mid[p & 1]);
      const kda_status cs = kda_chunk_fwd(
          dev(L.q, L.stride_k, dk), dev(L.k, L.stride_k, dk), dev(L.v, L.stride_v, dv),
          dev(L.la, L.stride_k, dk), dev(L.beta, L.stride_b, 1),
          gate ? dev(L.gate, L.stride_v, dv) : nullptr, dev(L.out, L.stride_v, dv), entry, exit,
          nullptr, 1, tl, H, dk, dv, chunk, scale, flags, dtype, d + L.ws, L.ws_bytes, stream);
      if (cs != KDA_OK) {  // kda_chunk_fwd has set the message
        st = cs;
        break;
      }
      if (!ok(cudaEventRecord(ev_done(slice), s), "event record") ||
          !ok(cudaStreamWaitEvent(s_out, ev_done(slice), 0), "stream wait"))
        break;
      // copy the slice's output (and after the last slice the final state) back
      if (n > 0)
        ok(cudaMemcpyAsync((char *)out + h0 * dv * e, dev(L.out, L.stride_v, dv), n * dv * e,
                           cudaMemcpyDeviceToHost, s_out),
           "copy back");
      if (p == parts - 1 && final_state)
        ok(cudaMemcpyAsync((char *)final_state + sq * sb, d + L.fs + sq * sb, sb,
                           cudaMemcpyDeviceToHost, s_out),
           "copy back");
    }
  }
  // join both copy streams back into the caller's stream, also after a failed step
  if (forked) {
    for (int i = 0; i < 2; ++i) {
      cudaStream_t c = i == 0 ? s_in : s_out;
      cudaError_t je = cudaEventRecord(ev[1 + i], c);
      if (je == cudaSuccess) je = cudaStreamWaitEvent(s, ev[1 + i], 0);
      ok(je, "join");
    }
  }
  for (cudaEvent_t x : ev)
    if (x) cudaEventDestroy(x);
  return st;
}

}  // extern "C"
