// kda_chunk_fwd_noalloc: chunked prefill whose scratch space is a fixed,
// file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// mixer: host frameworks that reserve the whole device heap up front and hand a
// kernel only its inputs and outputs, plugin interfaces with no workspace
// argument, and code paths that must not call cudaMalloc / cudaFree because
// those can synchronise the device. This entry point serves them. It runs the
// same kernels as kda_chunk_fwd; only the origin of the scratch differs.
//
// Limits and sharing rules:
//  - The scratch is kNoAllocScratchBytes (64 MiB) per device, reserved for as
//    long as the library stays loaded on every device that loads it.
//  - Problems whose scratch need (kda_chunk_fwd_workspace_size) exceeds that are
//    rejected with KDA_ERR_WORKSPACE before anything is launched.
//  - Every call on a device uses the same array and leaves its contents behind.
//    No byte of it is assumed to be zero: each call writes every scratch byte it
//    later reads. Calls whose kernels overlap on the GPU (different streams with
//    no ordering between them) race on the array and give wrong results; order
//    such calls on one stream or with events.
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, under a lock). That first call
//    should come before any stream capture.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
cudaError_t scratch_address(void **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(
    const void *q, const void *k, const void *v, const void *log_alpha, const void *beta,
    const void *gate, void *out, const float *initial_state, float *final_state,
    const int32_t *cu_seqlens, int n_seq, int64_t T_total, int H, int dk, int dv, int chunk,
    float scale, unsigned flags, kda_dtype dtype, kda_stream_t stream) {
  const size_t need = kda_chunk_fwd_workspace_size(T_total, n_seq, H, dk, dv, chunk, dtype);
  if (need > kNoAllocScratchBytes) {
    // Argument errors keep their own status: with no workspace the regular entry
    // point validates everything and stops before its first launch.
    kda_status st = kda_chunk_fwd(q, k, v, log_alpha, beta, gate, out, initial_state,
                                  final_state, cu_seqlens, n_seq, T_total, H, dk, dv, chunk,
                                  scale, flags, dtype, nullptr, 0, stream);
    if (st != KDA_ERR_WORKSPACE) return st;
    return kda::api_fail(KDA_ERR_WORKSPACE,
                         "kda_chunk_fwd_noalloc: this problem needs %zu bytes of scratch; the "
                         "static scratch holds %zu bytes",
                         need, kNoAllocScratchBytes);
  }
  void *scratch = nullptr;
  if (need > 0) {
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
      return kda::api_fail(KDA_ERR_CUDA, "kda_chunk_fwd_noalloc: scratch address lookup: %s",
                           cudaGetErrorString(e));
  }
  return kda_chunk_fwd(q, k, v, log_alpha, beta, gate, out, initial_state, final_state,
                       cu_seqlens, n_seq, T_total, H, dk, dv, chunk, scale, flags, dtype, scratch,
                       kNoAllocScratchBytes, stream);
}
