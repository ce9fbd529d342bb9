// Stage A of the chunked KDA forward on the sm_103a tensor cores (bf16 inputs,
// dk = dv = 128): the update cards, one CTA per (chunk, head), two per SM. The card itself is
// built by card_body (tc_card_body.cuh, which also states the algebra); this file maps CTAs to
// chunks and sizes the workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "tc_card_body.cuh"
#include "tc_card_layout.cuh"
#include "tc_common.cuh"

namespace kda {

__device__ unsigned g_tc_err;

namespace {

using namespace tc;
using namespace tcl;
using namespace tcb;

// One CTA (256 threads, two per SM) per (chunk, head).
__global__ void __launch_bounds__(256, 2) kda_card_tc(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
    const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16 *__restrict__ beta, const int32_t *__restrict__ cu, int n_seq,
    int64_t fixed_len, int H, unsigned flags, const ChunkMeta *__restrict__ meta,
    const int *__restrict__ off, int chunk_part, int b_lo, int b_hi,
    const int *__restrict__ off_blo, const int *__restrict__ off_bhi, uint8_t *__restrict__ cards) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_tma, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ float s_rk[C], s_rq[C], s_b[C], s_d[DD];

  const int h = blockIdx.y, tid = threadIdx.x;
  // global chunk ci of this CTA, its sequence s and its chunk jc within s: all chunks
  // (chunk_part < 0), or the x-th chunk of part chunk_part of the sequences, in sequence order.
  // A part of a sequence with n chunks holds its chunks [n * b_lo / 64, n * b_hi / 64). Without
  // cu_seqlens every sequence has n chunks and the chunk table is not used; with them, off_blo
  // and off_bhi hold the running sums over the sequences of the part's first and end chunk
  // (off_blo == nullptr: the first part, which starts at 0; off_bhi == off: the last part).
  int ci = blockIdx.x, s, jc;
  if (cu == nullptr) {
    const int n = (int)((fixed_len + C - 1) / C);
    const int lo = chunk_part < 0 ? 0 : (int)((int64_t)n * b_lo / 64);
    const int per = (chunk_part < 0 ? n : (int)((int64_t)n * b_hi / 64)) - lo;
    if (per == 0 || ci >= n_seq * per) return;
    s = ci / per;
    jc = ci - s * per + lo;
    ci = s * n + jc;
  } else {
    if (meta->invalid) return;
    if (chunk_part >= 0) {
      // part-local offset of sequence t: its part's chunks in all earlier sequences
      auto pre = [&](int t) { return off_bhi[t] - (off_blo ? off_blo[t] : 0); };
      if (ci >= pre(n_seq)) return;
      int lo = 0, hi = n_seq - 1;  // largest s whose part starts at or before ci
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre(mid) <= ci) lo = mid; else hi = mid - 1;
      }
      s = lo;
      jc = (off_blo ? off_blo[s + 1] - off_blo[s] : 0) + (ci - pre(s));
      ci = off[s] + jc;
    } else {
      if (ci >= meta->total_chunks) return;
      s = find_seq(off, n_seq, ci);
      jc = ci - off[s];
    }
  }
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int64_t t0 = ts + (int64_t)jc * C;
  const int len = (int)min((int64_t)C, ls - (int64_t)jc * C);
  const CardIn in{&tm_k, &tm_q, &tm_la, &tm_v, beta, H, flags, cards};
  const CardGroup G{sm, &tmem_base, 0u, &bar_tma, &bar_mma, s_rk, s_rq, s_b, s_d, &g_tc_err,
                    tid, 0, 2};
  if (tid == 0) {
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    card_issue_loads(in, G, h, t0);
  }
  if ((tid >> 5) == 1) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  card_body(in, G, ci, h, t0, len, 0u);
  if ((tid >> 5) == 1) tmem_dealloc(tmem_base, 256);
}


}  // namespace

bool tc_path(int dk, int dv, kda_dtype dt) {
  return dt == KDA_DTYPE_BF16 && dk == DD && dv == DD;
}

// The state pass runs one CTA per (sequence, head). With at most 112 of them (three
// quarters of a 152-SM GPU's SMs) and at least 16 chunks per sequence on average, the cards of
// each sequence's later part are built on the idle SMs while the state pass walks the earlier
// one. Measured on the prefill workload (4 x 4096 tokens, 16 heads), in 64ths of each
// sequence's chunks: a boundary at 47 took 0.3600 ms, at 45/46/48/49/50 0.3618/0.3610/0.3623/
// 0.3655/0.3682 ms; three parts (boundaries 41-45 and 56-59) 0.371-0.385 ms, their short state
// passes paying the pass's start-up (about 9 us) once more.
int tc_split_parts(int64_t T_total, int n_seq, int H, int *bound64) {
  constexpr int kParts = 2;
  constexpr int kBound[kParts + 1] = {0, 47, 64};
  if (n_seq <= 0 || (int64_t)n_seq * H > 112 || T_total < (int64_t)16 * C * n_seq) return 0;
  if (bound64)
    for (int i = 0; i <= kParts; ++i) bound64[i] = kBound[i];
  return kParts;
}

size_t tc_ws_bytes(int64_t T_total, int n_seq, int H) {
  const size_t mc = (size_t)(T_total / C) + (size_t)n_seq + 1;
  size_t b = align_up(sizeof(ChunkMeta), 256);
  b += 2 * align_up(sizeof(int) * (size_t)(n_seq + 1), 256);
  const int parts = tc_split_parts(T_total, n_seq, H);
  if (parts > 1) {
    b += align_up(sizeof(int) * (size_t)(parts - 1) * (n_seq + 1), 256);
    b += (parts > 2 ? 2 : 1) * align_up(sizeof(float) * (size_t)n_seq * H * DD * DD, 256);
  }
  if (fused_shape(T_total, n_seq, H)) b += fused_flag_bytes(T_total, n_seq, H);
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
  w.seq_order = (int *)p;
  p += align_up(sizeof(int) * (size_t)(n_seq + 1), 256);
  w.nparts = tc_split_parts(T_total, n_seq, H, w.bound64);
  if (w.nparts > 1) {
    w.seq_chunk_b = (int *)p;
    p += align_up(sizeof(int) * (size_t)(w.nparts - 1) * (n_seq + 1), 256);
    const size_t mb = align_up(sizeof(float) * (size_t)n_seq * H * DD * DD, 256);
    w.mid[0] = (float *)p;
    p += mb;
    if (w.nparts > 2) {
      w.mid[1] = (float *)p;
      p += mb;
    }
  }
  if (fused_shape(T_total, n_seq, H)) {
    const size_t fb = fused_flag_bytes(T_total, n_seq, H);
    w.ready = (unsigned *)p;
    w.next = (int *)(p + fb - 256);
    p += fb;
  }
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

bool make_rows_map_f32(CUtensorMap *m, const void *base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)DD, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)DD * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_card_tc(const void *q, const void *k, const void *v, const void *la,
                           const void *beta, const int32_t *cu, int n_seq, int64_t T_total, int H,
                           unsigned flags, const ChunkWs &ws, cudaStream_t st, int part) {
  if (T_total == 0) return cudaSuccess;  // no chunk has tokens
  CUtensorMap mk, mq, mla, mv;
  if (!make_token_map(&mk, k, T_total, H) || !make_token_map(&mq, q, T_total, H) ||
      !make_token_map(&mla, la, T_total, H) || !make_token_map(&mv, v, T_total, H))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(kda_card_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, A_DYN);
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  // CTAs beyond a part's chunk count (known on the device only) return at once. A part spanning
  // the 64ths [b_lo, b_hi) holds at most that fraction of all chunks plus one per sequence.
  int grid = ws.max_chunks, b_lo = 0, b_hi = 64;
  const int *off_blo = nullptr, *off_bhi = ws.seq_chunk_off;
  if (part >= 0) {
    b_lo = ws.bound64[part];
    b_hi = ws.bound64[part + 1];
    if (part > 0) off_blo = ws.seq_chunk_b + (size_t)(part - 1) * (n_seq + 1);
    if (part + 1 < ws.nparts) off_bhi = ws.seq_chunk_b + (size_t)part * (n_seq + 1);
    grid = (int)std::min<int64_t>(ws.max_chunks,
                                  (int64_t)ws.max_chunks * (b_hi - b_lo) / 64 + n_seq + 1);
  }
  kda_card_tc<<<dim3(grid, H), 256, A_DYN, st>>>(
      mk, mq, mla, mv, (const __nv_bfloat16 *)beta, cu, n_seq, fixed_len, H, flags, ws.meta,
      ws.seq_chunk_off, part, b_lo, b_hi, off_blo, off_bhi, ws.cards);
  return cudaGetLastError();
}

cudaError_t tc_take_error(unsigned *bits) {
  unsigned v = 0, z = 0, w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_tc_err, &z, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = state_tc_take_error(&w);  // the state pass's word
  *bits = v | w;
  return e;
}

}  // namespace kda
