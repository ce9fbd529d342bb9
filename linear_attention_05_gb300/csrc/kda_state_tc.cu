// Stage B of the chunked KDA forward on the sm_103a tensor cores (bf16 inputs,
// dk = dv = 128): the sequential state pass, one CTA per (sequence, head). The pass itself is
// state_body (tc_state_body.cuh, which also describes it); this file launches it.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_card_layout.cuh"
#include "tc_common.cuh"
#include "tc_state_body.cuh"

namespace kda {

__device__ unsigned g_state_tc_err;

namespace {

using namespace tc;
using namespace tcl;
using namespace tsb;

// One CTA per (sequence, head) chain (the prefill pass; a grid y index of 1 would select the X /
// Z part of a summary pass, which kda_summary_tc now walks in one CTA).
template <bool SUMMARY>
__global__ void __launch_bounds__(kThreads, 1) kda_state_tc(const __grid_constant__ StateIn p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[Geo<SUMMARY>::NST], bar_mma, bar_ofull[2], bar_ofree[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  const StateShared sh{(uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023), bar_full,
                       &bar_mma, bar_ofull, bar_ofree, &tmem_base, &s_fail, &g_state_tc_err};
  state_body<SUMMARY>(p, sh, blockIdx.x, blockIdx.y, threadIdx.x, true, nullptr);
}

// Segment summaries: one CTA per (segment, head) walks X and Z together.
__global__ void __launch_bounds__(kThreads, 1) kda_summary_tc(const __grid_constant__ StateIn p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[kSumNst], bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  const SummaryShared sh{(uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023), bar_full,
                         &bar_mma, &tmem_base, &s_fail, &g_state_tc_err};
  summary_body(p, sh, blockIdx.x, threadIdx.x);
}

}  // namespace

cudaError_t launch_state_tc(int mode, unsigned flags, const void *gate, void *out, const float *S0,
                            float *S_final, float *X_out, float *Z_out, const int32_t *cu,
                            int n_seq, int64_t T_total, int H, float scale, const ChunkWs &ws,
                            cudaStream_t st, CkptOut ck, int part) {
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  auto launch = [&](auto kernel, int dyn) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
    if (e != cudaSuccess) return e;
    // part p of a split prefill starts from mid[(p - 1) & 1] and leaves its state in mid[p & 1]
    const bool split = part >= 0;
    const StateIn p{mode, flags, (const __nv_bfloat16 *)gate, (__nv_bfloat16 *)out, S0, S_final,
                    X_out, Z_out, cu, n_seq, fixed_len, H, scale, ws.meta, ws.seq_chunk_off,
                    ws.cards, ck, part, split ? ws.bound64[part] : 0,
                    split ? ws.bound64[part + 1] : 64,
                    split && part > 0 ? ws.mid[(part - 1) & 1] : nullptr,
                    split && part + 1 < ws.nparts ? ws.mid[part & 1] : nullptr, ws.seq_order};
    kernel<<<dim3(n_seq * H, 1), kThreads, dyn, st>>>(p);
    return cudaSuccess;
  };
  // mode 1 (segment summaries): X and Z of a chain in one CTA
  cudaError_t e = mode == 0 ? launch(kda_state_tc<false>, Geo<false>::DYN)
                            : launch(kda_summary_tc, kSumDyn);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t state_tc_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_state_tc_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_state_tc_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

}  // namespace kda
