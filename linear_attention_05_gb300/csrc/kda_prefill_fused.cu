// One persistent launch for a fixed-length tensor-core prefill (bf16, dk = dv = 128): the update
// cards and the sequential state pass overlap inside a single cooperative grid of one CTA per
// SM.
//
// K3 training analysis (lotamate.com/blog/posts/kimi-k3-training-analysis.html), section 4:
// FlashKDA overlaps the intra-chunk computation with the cross-chunk state propagation. K3
// training overview (zuoshipin.com/article/18261), section 4 "FlashKDA": the per-chunk update
// cards are independent and prepared in parallel; only the state hand-off runs in order.
//
// Schedule. Every CTA starts as two card-building groups of 256 threads (card_body,
// tc_card_body.cuh) that take cards from one counter in chunk-major order: chunk 0 of every
// (sequence, head) chain, then chunk 1, and so on. The first n_chains CTAs own one chain
// each: once the counter passes switch_at they finish the card in hand and walk their chain
// with the state pass (state_body, tc_state_body.cuh), reading each card after its ready flag
// is up. The other CTAs keep building cards until none is left. So the whole GPU builds the
// leading cards, and the state pass then runs beside the remaining ones, which it reads
// shortly after they are written (mostly from L2).
//
// Progress. No CTA waits on the state pass, and a card builder waits only on its own copies
// and MMAs, so every card is eventually built; a chain owner waits only on flags of cards that
// builders will raise. The cooperative launch guarantees that all CTAs are resident at once.
// Every wait is bounded: a flag that does not come up within 2 s records KDA_ERR_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_card_body.cuh"
#include "tc_card_layout.cuh"
#include "tc_common.cuh"
#include "tc_state_body.cuh"

namespace kda {

__device__ unsigned g_fused_err;

namespace {

using namespace tc;
using namespace tcl;

constexpr int kFusedThreads = 512;
constexpr int kFusedDyn = 2 * tcb::A_BODY + 1024;  // two card groups (the state pass needs less)
static_assert(tsb::Geo<false>::DYN <= kFusedDyn, "the state pass fits the card groups' memory");
static_assert(tsb::kThreads == kFusedThreads, "one CTA shape for both roles");
static_assert(tcb::A_BODY % 1024 == 0, "the second group's region stays 1024-byte aligned");

struct FusedArgs {
  tsb::StateIn st;   // the state pass (mode 0, fixed lengths, no split)
  const __nv_bfloat16 *beta;
  int n_chunks;      // chunks per sequence
  int total;         // cards: n_chunks * n_seq * H
  int switch_at;     // a chain owner stops building cards after claiming this card or a later one
  unsigned *ready;   // [n_seq * n_chunks * H] card flags, zero on entry
  int *next;         // the card counter, zero on entry
};

// One card-building group's loop: claim the next card, build it, publish its flag; a chain
// owner's groups stop once they claimed a card at or past switch_at. Both groups run this one
// copy of the code (one copy per group would double the card code's instruction footprint,
// which measured about 60 % slower per card).
__device__ __forceinline__ void build_cards(int grp, const CUtensorMap &tm_k,
                                            const CUtensorMap &tm_q, const CUtensorMap &tm_la,
                                            const CUtensorMap &tm_v, const FusedArgs &a,
                                            uint8_t *sm, const uint32_t *tmem_base,
                                            uint64_t *c_bar_tma, uint64_t *c_bar_mma,
                                            float (*s_rk)[C], float (*s_rq)[C], float (*s_b)[C],
                                            float (*s_d)[DD], int *s_item, bool owner,
                                            int n_chains) {
  const int gt = threadIdx.x - 256 * grp;
  const int H = a.st.H;
  const tcb::CardIn in{&tm_k, &tm_q, &tm_la, &tm_v, a.beta, H, a.st.flags,
                       const_cast<uint8_t *>(a.st.cards)};
  const tcb::CardGroup G{sm + grp * tcb::A_BODY, tmem_base, 256u * grp, &c_bar_tma[grp],
                         &c_bar_mma[grp], s_rk[grp], s_rq[grp], s_b[grp], s_d[grp],
                         &g_fused_err, gt, 1 + 5 * grp, 2 + 5 * grp};
  const int64_t L = a.st.fixed_len;
  uint32_t parity = 0;
  unsigned *pending = nullptr;  // flag of the last card built, raised once its stores complete
  for (;;) {
    if (gt == 0) s_item[grp] = atomicAdd(a.next, 1);
    named_bar(G.bar_main, 256);
    const int i = s_item[grp];
    if (i >= a.total) break;
    const int jc = i / n_chains, chain = i - jc * n_chains;
    const int s = chain / H, h = chain - s * H;
    const int ci = s * a.n_chunks + jc;
    const int64_t t0 = (int64_t)s * L + (int64_t)jc * C;
    const int len = (int)min((int64_t)C, L - (int64_t)jc * C);
    if (gt == 0) tcb::card_issue_loads(in, G, h, t0);
    // the previous card is published while this card's inputs are in flight
    bool ok = tcb::card_body(in, G, ci, h, t0, len, parity, pending);
    parity ^= 1u;
    pending = nullptr;
    ok = named_bar_and(G.bar_main, 256, ok);
    if (!ok) break;  // recorded in the error word; the chain owner's wait runs out too
    pending = a.ready + (size_t)ci * H + h;
    if (owner && i >= a.switch_at) break;
  }
  tcb::card_publish(G, pending);
}

__global__ void __launch_bounds__(kFusedThreads, 1) kda_prefill_fused(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ FusedArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t c_bar_tma[2], c_bar_mma[2];
  __shared__ float s_rk[2][C], s_rq[2][C], s_b[2][C], s_d[2][DD];
  __shared__ int s_item[2];
  __shared__ uint64_t bar_full[tsb::Geo<false>::NST], bar_mma, bar_ofull[2], bar_ofree[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.st.H;
  const int n_chains = a.st.n_seq * H;
  const bool owner = (int)blockIdx.x < n_chains;

  // 512 tensor-memory columns for the CTA: 256 per card group, all 512 for the state pass
  if (warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int g = 0; g < 2; ++g) {
      mbar_init(&c_bar_tma[g], 1);
      mbar_init(&c_bar_mma[g], 1);
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- cards, chunk-major, by two independent groups (named barriers 1-5 and 6-10)
  build_cards(tid >> 8, tm_k, tm_q, tm_la, tm_v, a, sm, &tmem_base, c_bar_tma, c_bar_mma, s_rk,
              s_rq, s_b, s_d, s_item, owner, n_chains);
  tc_fence_before();
  __syncthreads();  // both groups are done with their shared memory and tensor memory
  tc_fence_after();
  if (owner) {
    const tsb::StateShared sh{sm, bar_full, &bar_mma, bar_ofull, bar_ofree, &tmem_base, &s_fail,
                              &g_fused_err};
    // the pass index is blockIdx.y, 0 on this one-dimensional grid: given a literal 0 the
    // compiler folds the summary branches differently and spills ~250 bytes a thread
    tsb::state_body<false>(a.st, sh, blockIdx.x, blockIdx.y, tid, false, a.ready);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tmem_base, 512);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
  }();
  return fn;
}

// [T_total, H, 128] bf16; box = 64 channels x 1 head x 64 tokens, 128-byte swizzle (the
// tensor-core tile layout), zero fill past T_total.
bool token_map(CUtensorMap *m, const void *base, int64_t T_total, int H) {
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

}  // namespace

// Chunk rows (one chunk of every chain) that all SMs build before the chain owners switch to
// their chains. After the switch, the grid - n_chains builder CTAs (two groups each) make
// P = 2 (grid - n_chains) / kFusedCardUs cards a microsecond while the chains take
// Q = n_chains / kFusedStepUs. If P >= Q the owners can start after the first row; otherwise
// the chains must start with a lead of n_chunks (1 - P / Q) rows so that the last cards are
// ready when the chains reach them. (Measured best: 1 of 16 rows for 16 and 32 chains, 9-10 of
// 16 for 64, on 152 SMs.)
int fused_switch_chunks(int n_chunks, int n_chains, int grid) {
  const double p_over_q = 2.0 * kFusedStepUs * (grid - n_chains) / (kFusedCardUs * n_chains);
  const double lead = p_over_q >= 1.0 ? 0.0 : 1.0 - p_over_q;
  const int rows = (int)(n_chunks * lead + 0.5);
  return rows < 1 ? 1 : (rows > n_chunks ? n_chunks : rows);
}

int fused_ctas(int n_seq, int H) {
  int dev = 0, sms = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (!coop || (int64_t)n_seq * H + kFusedMinBuilders > sms) return 0;
  return sms;
}

bool fused_shape(int64_t T_total, int n_seq, int H) {
  if (n_seq <= 0 || T_total % n_seq != 0) return false;
  const int64_t n_chunks = (T_total / n_seq + C - 1) / C;
  return n_chunks >= kFusedMinChunks && (int64_t)n_seq * H <= kFusedMaxChains;
}

cudaError_t launch_prefill_fused(const void *q, const void *k, const void *v, const void *la,
                                 const void *beta, const void *gate, void *out, const float *S0,
                                 float *S_final, int n_seq, int64_t T_total, int H, float scale,
                                 unsigned flags, const ChunkWs &ws, CkptOut ck, int grid,
                                 cudaStream_t st) {
  CUtensorMap mk, mq, mla, mv;
  if (!token_map(&mk, k, T_total, H) || !token_map(&mq, q, T_total, H) ||
      !token_map(&mla, la, T_total, H) || !token_map(&mv, v, T_total, H))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kda_prefill_fused,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedDyn);
  if (e != cudaSuccess) return e;
  const int64_t L = T_total / n_seq;
  const int n_chunks = (int)((L + C - 1) / C);
  const int n_chains = n_seq * H;
  FusedArgs a;
  a.st = tsb::StateIn{0, flags, (const __nv_bfloat16 *)gate, (__nv_bfloat16 *)out, S0, S_final,
                      nullptr, nullptr, nullptr, n_seq, L, H, scale, ws.meta, ws.seq_chunk_off,
                      ws.cards, ck, -1, 0, 64, nullptr, nullptr, nullptr};
  a.beta = (const __nv_bfloat16 *)beta;
  a.n_chunks = n_chunks;
  a.total = n_chunks * n_chains;
  a.switch_at = fused_switch_chunks(n_chunks, n_chains, grid) * n_chains;
  a.ready = ws.ready;
  a.next = ws.next;
  // flags and counter start at zero (stream-ordered, so a graph capture records them too)
  e = cudaMemsetAsync(ws.ready, 0, fused_flag_bytes(T_total, n_seq, H), st);
  if (e != cudaSuccess) return e;
  void *args[] = {&mk, &mq, &mla, &mv, &a};
  return cudaLaunchCooperativeKernel((const void *)kda_prefill_fused, dim3(grid),
                                     dim3(kFusedThreads), args, kFusedDyn, st);
}

cudaError_t fused_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_fused_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_fused_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

}  // namespace kda
