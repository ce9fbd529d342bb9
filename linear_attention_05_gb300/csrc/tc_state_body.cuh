// The sequential state pass of one (sequence, head) chain on the sm_103a tensor cores, as a
// device function run by a CTA of 512 threads: the state-pass kernel (kda_state_tc.cu) and the
// persistent prefill kernel (kda_prefill_fused.cu) both walk their chains with it.
//
// K3 training overview (zuoshipin.com/article/18261), section 4 "FlashKDA": only the state
// hand-off and the output read-out run in order. The fp32 state lives in tensor memory as
// S^T (lane = value channel). Per chunk the CTA pre-loads Diag(e^{G_C}) S + B_c into tensor
// memory and issues one group of MMAs, bf16(S^T) x [Phi'^T | Q'^T] (card layout in
// tc_card_layout.cuh), accumulating onto it, so the serial path has a single tensor-core round
// trip per chunk; two warpgroups stage the state and two more turn the output accumulators
// into o while the next chunk's MMAs run.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"
#include "tc_card_layout.cuh"
#include "tc_common.cuh"

namespace kda {
namespace tsb {

using namespace tc;
using namespace tcl;

// ---- stage B shared memory
// 8 state warps + 8 output warps; launched at 128 registers a thread, split by setmaxnreg
constexpr int kThreads = 512;
constexpr int kStateRegs = 160, kOutRegs = 96;
static_assert(2 * 128 * kStateRegs + 2 * 128 * kOutRegs <= kThreads * 128,
              "the register split must fit the launch's allocation");
// Card ring geometry. The prefill pass copies [Phi'^T | Q'^T] and e^{G_C} into each stage,
// three stages deep; the summary pass needs no Q'^T, so its stages are a third smaller and
// four fit (no output tile either).
template <bool SUMMARY>
struct Geo {
  static constexpr int NST = SUMMARY ? 4 : 3;             // card ring depth
  static constexpr int PHIQ = SUMMARY ? 32768 : CARD_BCT;  // card bytes of the MMA's B operand
  static constexpr int TX = PHIQ + 512;                    // then e^{G_C}
  static constexpr int STAGE = (TX + 1023) / 1024 * 1024;
  static constexpr int SA = NST * STAGE;  // S^T bf16 operand, 128 x 128 K-major (32768)
  static constexpr int OT = SA + 32768;   // output tile: 64 tokens x (128 + 4) fp32
  static constexpr int DYN = OT + (SUMMARY ? 0 : 64 * (DD + 4) * 4) + 1024;
};

// Acquire-load of a 32-bit flag (gpu scope) until it is non-zero, for at most limit_ns. With
// bulk, a proxy fence then orders the caller's later bulk copies (async proxy) behind it.
__device__ __forceinline__ bool wait_flag(const unsigned *f, bool bulk,
                                          uint64_t limit_ns = 2000000000ull) {
  auto ld = [&]() {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
  };
  bool ok = ld() != 0u;
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    while (!(ok = ld() != 0u)) {
      __nanosleep(64);
      if (globaltimer_ns() - t0 > limit_ns) break;
    }
  }
  if (bulk) asm volatile("fence.proxy.async.global;" ::: "memory");
  return ok;
}

// The arguments of a state pass (those of the kernel).
struct StateIn {
  int mode;  // 0: prefill (out, S_final); 1: segment summary (X_out, Z_out)
  unsigned flags;
  const __nv_bfloat16 *gate;
  __nv_bfloat16 *out;
  const float *S0;
  float *S_final, *X_out, *Z_out;
  const int32_t *cu;
  int n_seq;
  int64_t fixed_len;
  int H;
  float scale;
  const ChunkMeta *meta;
  const int *off;
  const uint8_t *cards;
  CkptOut ck;
  // split prefill: part >= 0 walks each sequence's chunks [n * b_lo / 64, n * b_hi / 64),
  // starting from mid_in (else S0) and leaving its state in mid_out (else S_final)
  int part, b_lo, b_hi;
  const float *mid_in;
  float *mid_out;
  const int *seq_order;
};

// Shared-memory objects of the CTA running the pass.
struct StateShared {
  uint8_t *sm;  // Geo<SUMMARY>::DYN - 1024 bytes, 1024-byte aligned
  uint64_t *bar_full, *bar_mma, *bar_ofull, *bar_ofree;
  uint32_t *tmem_base;
  int *s_fail;
  unsigned *err;  // device error word
};

// ===========================================================================
// Stage B: the sequential state pass, one CTA per (sequence, head), 512 threads.
// Warps 0-7 (state group, kStateRegs registers a thread) carry the serial path: warp w serves
// tensor-memory lanes 32*(w%4).. (lane j = value channel j, i.e. row j of S^T) and the key
// columns [64*(w/4), 64*(w/4) + 64) of that row. Warps 8-15 (two output warpgroups, kOutRegs
// registers a thread, one per 32-token half of the chunk) read the chunk outputs from the same
// lanes, apply scale and gate and store o, off the serial path. mode 0: prefill; mode 1:
// segment summary on [X | Z] (blockIdx.y = 0: X with entry I; 1: Z with entry 0), no output.
//
// Tensor memory holds two accumulator sets, chunk n using set n % 2: columns
// [256b, 256b+128) the fp32 state S^T, [256b+128, 256b+192) the output block.
// Before the MMAs of chunk n the set is pre-loaded with Diag(e^{G_C}) S + B_c
// (state group) and O_intra^T (output group), so one N = 192 MMA chain per chunk
// produces both the next state and the chunk output.
// mbarriers: bar_full[G::NST] card stages landed; bar_mma chunk MMAs done (state
// group); bar_ofull[2] output block written (output group); bar_ofree[2]
// output block read and re-seeded (MMA issuer).
// chain: the CTA's chain index; yblk: 0/1 = X/Z part of a summary pass; own_tmem: allocate
// (and free) the 512 tensor-memory columns here, else they are allocated already at
// *sh.tmem_base; ready: null, or one flag per (chunk, head) card that another CTA raises
// once the card is complete in global memory.
template <bool SUMMARY>
__device__ __forceinline__ void state_body(const StateIn &p, const StateShared &sh, int chain,
                                           int yblk, int tid, bool own_tmem,
                                           const unsigned *ready) {
  const int mode = p.mode;
  const unsigned flags = p.flags;
  const __nv_bfloat16 *__restrict__ gate = p.gate;
  __nv_bfloat16 *__restrict__ out = p.out;
  const float *__restrict__ S0 = p.S0;
  float *__restrict__ S_final = p.S_final;
  float *__restrict__ X_out = p.X_out;
  float *__restrict__ Z_out = p.Z_out;
  const int32_t *__restrict__ cu = p.cu;
  const int64_t fixed_len = p.fixed_len;
  const int H = p.H;
  const float scale = p.scale;
  const ChunkMeta *__restrict__ meta = p.meta;
  const int *__restrict__ off = p.off;
  const uint8_t *__restrict__ cards = p.cards;
  const CkptOut &ck = p.ck;
  const int part = p.part;
  const int *__restrict__ seq_order = p.seq_order;
  using G = Geo<SUMMARY>;
  constexpr int B_NSTAGE = G::NST;
  uint64_t *bar_full = sh.bar_full, *bar_ofull = sh.bar_ofull, *bar_ofree = sh.bar_ofree;
  uint64_t &bar_mma = *sh.bar_mma;
  uint32_t &tmem_base = *sh.tmem_base;
  int &s_fail = *sh.s_fail;
  // without cu_seqlens the chunk table is not used: chains in index order, n chunks a sequence
  if (cu != nullptr && meta->invalid) return;
  uint8_t *sm = sh.sm;
  const uint32_t sb = smem_u32(sm);
  // CTAs take the sequences longest first (the order the chunk table computed)
  const int h = chain % H;
  const int s = cu ? seq_order[chain / H] : chain / H;
  const int warp = tid >> 5, lane = tid & 31;
  const bool state_grp = warp < 8;
  const int quad = warp & 3;           // lane quadrant of this warp
  const int j = quad * 32 + lane;      // tensor-memory lane / value channel
  const int half = (warp >> 2) & 1;    // state group: which 64 key columns
  const bool xpart = (mode == 1 && yblk == 0);
  const bool with_bc = !xpart;
  const bool with_o = (mode == 0 && out != nullptr);

  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int64_t ls_seq = ls;
  int nchunks = (int)((ls + C - 1) / C);
  const int seq_off = cu ? off[s] : s * nchunks;  // first global chunk of the sequence
  // a split prefill walks the sequence in parts, each a range of its chunks, handing the state
  // from one part to the next through a buffer; chunk n below is chunk n_lo + n of the sequence
  int n_lo = 0;
  if (part >= 0) {
    const int lo = (int)((int64_t)nchunks * p.b_lo / 64), hi = (int)((int64_t)nchunks * p.b_hi / 64);
    n_lo = lo;
    ls = min(ls, (int64_t)hi * C) - (int64_t)lo * C;
    ts += (int64_t)lo * C;
    nchunks = hi - lo;
  }
  const int cbase = nchunks > 0 ? seq_off + n_lo : 0;
  auto card_of = [&](int n) { return cards + ((size_t)(cbase + n) * H + h) * CARD_BYTES; };
  // With ready flags (cards built by other CTAs of the same launch) the loader thread acquires
  // card n's flag, bounded, before it copies the card; a flag that never comes up is recorded
  // as a timeout. The other state threads read card n with plain loads only after a barrier
  // that follows the loader's acquire (card n + 3 is acquired before the barrier of chunk n),
  // so they need no acquire of their own; the output warps, which share no barrier with the
  // loader, acquire the flag themselves.
  auto card_ready = [&](int n, bool bulk) -> bool {
    if (ready == nullptr) return true;
    if (wait_flag(ready + (size_t)(cbase + n) * H + h, bulk)) return true;
    atomicOr(sh.err, kErrTimeout);
    return false;
  };
  const float *S_entry = p.mid_in ? p.mid_in : S0;
  float *S_exit = p.mid_out ? p.mid_out : S_final;
  // element (c, j) of the entry state, and where element (c, j) of the result goes
  auto entry = [&](int c) -> float {
    if (mode == 0) return S_entry ? S_entry[(((size_t)s * H + h) * DD + c) * DD + j] : 0.f;
    return (xpart && c == j) ? 1.f : 0.f;
  };
  auto result_ptr = [&](int c) -> float * {
    if (mode == 0) return S_exit ? S_exit + (((size_t)s * H + h) * DD + c) * DD + j : nullptr;
    if (xpart) return X_out + (((size_t)s * H + h) * DD + c) * DD + j;
    return Z_out + (((size_t)s * H + h) * DD + c) * DD + j;
  };
  // prefix-cache checkpoint after chunk n (mode 0): this thread's 64 rows of column j
  auto save_ckpt = [&](int n, const float *x0, const float *x1) {
    if (mode != 0) return;
    float *cp = ckpt_after_chunk(ck, s, n_lo + n, ls_seq, H, h, DD, DD);
    if (cp == nullptr) return;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      cp[(size_t)(64 * half + u) * DD + j] = x0[u];
      cp[(size_t)(64 * half + 32 + u) * DD + j] = x1[u];
    }
  };
  if (nchunks == 0) {
    if (state_grp)
      for (int c = 64 * half; c < 64 * half + 64; ++c) {
        float *p = result_ptr(c);
        if (p) *p = entry(c);
      }
    return;
  }

  if (own_tmem && warp == 0) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < B_NSTAGE; ++i) mbar_init(&bar_full[i], 1);
    mbar_init(&bar_mma, 1);
    mbar_init(&bar_ofull[0], 1);
    mbar_init(&bar_ofull[1], 1);
    mbar_init(&bar_ofree[0], 256);
    mbar_init(&bar_ofree[1], 256);
    fence_mbar_init();
    s_fail = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = tmem_base;
  auto set_col = [](int n) { return 256 * (n & 1); };
  // register split of the launch's kThreads x 128: the two state warpgroups take 168 per
  // thread, the two output warpgroups 88 (2 x 128 x 168 + 2 x 128 x 88 = 512 x 128)
  if (state_grp) setmaxnreg_inc<kStateRegs>();
  else setmaxnreg_dec<kOutRegs>();
  if (state_grp) {
    int loads_issued = 0, loads_done = 0;
    uint32_t full_phase[B_NSTAGE] = {}, mma_phase = 0u;
    bool ok = true;
    const bool loader = (tid == 32);  // issues the card copies, off the MMA issuer's path
    auto stage_of = [](int n) { return n % B_NSTAGE; };
    // card n -> stage n % 3: [Phi'^T | Q'^T] and e^{G_C}
    auto load_card = [&](int n) {
      const int st = stage_of(n);
      uint8_t *dst = sm + st * G::STAGE;
      const uint8_t *src = card_of(n);
      if (!card_ready(n, true)) return;  // no copy: the wait on its stage runs out and reports it
      mbar_arrive_expect_tx(&bar_full[st], G::TX);
      for (int o = 0; o < G::PHIQ; o += 16384) bulk_g2s(dst + o, src + o, 16384, &bar_full[st]);
      bulk_g2s(dst + G::PHIQ, src + CARD_D, 512, &bar_full[st]);
      ++loads_issued;
    };
    auto wait_full = [&](int n) -> bool {
      const int st = stage_of(n);
      const bool r = mbar_wait(&bar_full[st], full_phase[st]);
      full_phase[st] ^= 1u;
      if (r) ++loads_done;
      return r;
    };
    // this thread's 64 columns of B_c^T row j of chunk n, straight from the card in global
    // memory (lane-interleaved: a warp reads 512 contiguous bytes per 8-column chunk). The pass
    // is the card's only reader, so the loads carry the last-use hint: the lines leave L2
    // early, making room for the cards prefetched ahead (0.1361 -> 0.1340 ms for the leading
    // pass of the prefill workload, with the same hint on the O_intra^T loads below)
    uint4 bcr[8];
    auto fetch_bc = [&](int n) {
      if (!with_bc || n >= nchunks) return;
      const uint8_t *src = card_of(n) + CARD_BCT;
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8)
        bcr[c8] = __ldlu(reinterpret_cast<const uint4 *>(src + ((8 * half + c8) * 128 + j) * 16));
    };
    // Pre-load for chunk n: tensor memory <- Diag(e^{G_C}) S + B_c (fp32) and the bf16
    // operand S^T (row j) in shared memory, from the 32 key columns 64*half + 32*qq.
    auto stage_piece = [&](int n, int qq, const float *x) {
      const float *dv =
          reinterpret_cast<const float *>(sm + stage_of(n) * G::STAGE + G::PHIQ);
      const int q4 = 2 * half + qq;
      float init[32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float bc[8];
        if (with_bc) unpack8(bcr[qq * 4 + ch], bc);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int c = q4 * 32 + ch * 8 + u;
          init[ch * 8 + u] = dv[c] * x[ch * 8 + u] + (with_bc ? bc[u] : 0.f);
        }
        *reinterpret_cast<uint4 *>(sm + G::SA + sw128_chunk(j, q4 * 4 + ch, 128)) =
            pack8(x + ch * 8);
      }
      tmem_st32(tmem_addr(tb, quad * 32, set_col(n) + 32 * q4), init);
    };
    auto finish_stage = [&]() {
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
    };
    auto issue_mma = [&](int n) -> bool {  // by thread 0
      // the output block of set n % 2 is read and zeroed (prologue, then chunk n - 2)
      if (with_o && !mbar_wait(&bar_ofree[n & 1], (n >> 1) & 1)) return false;
      tc_fence_after();
      const uint32_t stg = sb + stage_of(n) * G::STAGE;
      const uint32_t id = idesc_bf16(128, with_o ? 192 : 128, 0, 1);
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tb + set_col(n), desc_kmajor(sb + G::SA, 128, kk),
                 sdesc_sw128(stg + CARD_PHIQ + kk * 2048, 128 * 128, 1024), id, 1u);
      mma_commit(&bar_mma);
      if (with_o) mma_commit(&bar_ofull[n & 1]);
      return true;
    };

    // card n into L2 as its [Phi'^T | Q'^T] part is bulk-copied: the plain loads of its B_c^T
    // and O_intra^T come two chunks later. (Prefetching 1, 2, 3 or 6 chunks further ahead was
    // measured slower: 0.189, 0.190, 0.192 and 0.216 ms per pass against 0.1885.)
    auto prefetch_card = [&](int n) {
      if (n >= nchunks) return;
      const uint8_t *src = card_of(n);
      for (int o = 0; o < CARD_BYTES; o += 32768)
        prefetch_l2(src + o, min(32768, CARD_BYTES - o));
    };
    if (loader)
      for (int n = 0; n < B_NSTAGE && n < nchunks; ++n) {
        load_card(n);
        prefetch_card(n);
      }
    if (ready != nullptr) named_bar(1, 256);  // the loader has acquired cards 0-2
    fetch_bc(0);
    // chunk 0: entry state from global memory
    if (!wait_full(0)) ok = false;
    if (ok) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        float x[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) x[u] = entry(64 * half + 32 * qq + u);
        stage_piece(0, qq, x);
      }
      finish_stage();
    }
    // all state threads agree on `ok`, so none is left waiting at a later barrier
    ok = named_bar_and(1, 256, ok);
    tc_fence_after();
    if (tid == 0 && ok && !issue_mma(0)) s_fail = 1;
    fetch_bc(1);

    for (int n = 0; n < nchunks && ok; ++n) {
      // a timed-out wait only clears `good`; the group votes on it at the barrier below
      bool good = mbar_wait(&bar_mma, mma_phase);
      mma_phase ^= 1u;
      tc_fence_after();
      // the card of chunk n is consumed: refill its stage with chunk n + 3
      if (good && loader && n + B_NSTAGE < nchunks) {
        load_card(n + B_NSTAGE);
        prefetch_card(n + B_NSTAGE);
      }
      const bool last = (n + 1 == nchunks);
      if (good && !last) good = wait_full(n + 1);
      // state after chunk n: stage it for chunk n + 1, or write it out
      float x0[32], x1[32];
      if (good) {
        tmem_ld32(tmem_addr(tb, quad * 32, set_col(n) + 64 * half), x0);
        tmem_ld32(tmem_addr(tb, quad * 32, set_col(n) + 64 * half + 32), x1);
        tmem_wait_ld();
      }
      if (last) {
        if (good)
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            float *p0 = result_ptr(64 * half + u), *p1 = result_ptr(64 * half + 32 + u);
            if (p0) *p0 = x0[u];
            if (p1) *p1 = x1[u];
          }
        else
          ok = false;
        if (good) save_ckpt(n, x0, x1);
      } else {
        if (good) {
          stage_piece(n + 1, 0, x0);
          stage_piece(n + 1, 1, x1);
          finish_stage();
        }
        ok = named_bar_and(1, 256, good);
        tc_fence_after();
        if (!ok) break;
        if (tid == 0 && !issue_mma(n + 1)) s_fail = 1;
        save_ckpt(n, x0, x1);  // off the serial path: the next chunk's MMAs are in flight
        fetch_bc(n + 2);
      }
    }
    if (!ok || s_fail) {
      if (lane == 0) atomicOr(sh.err, kErrTimeout);
      // let copies still in flight land (bounded) before shared memory is released
      if (loader)
        for (int n = loads_done; n < loads_issued; ++n) {
          const int st = stage_of(n);
          if (!mbar_wait(&bar_full[st], full_phase[st], 100000000ull)) break;
          full_phase[st] ^= 1u;
        }
    }
  } else if (with_o) {
    // output warpgroups: o = scale * g * (Q' S + O_intra) for chunk n; warpgroup og takes tokens
    // [32 og, 32 og + 32). The output block of chunk n starts as O_intra^T (seeded two chunks
    // ahead from the card), so the MMA leaves Q' S + O_intra in it. The warps copy their lane
    // quadrants (channels) into a [32 tokens][128 channels] fp32 half-tile; then each thread
    // takes 4 tokens x 8 channels, so that a warp's gate loads and output stores cover two
    // whole 256-byte rows per instruction. The gate of the next chunk is loaded (same mapping)
    // as this one is used.
    constexpr int LDT = DD + 4;  // tile row pitch (floats)
    const int og = (warp - 8) >> 2;             // output warpgroup: token half
    const int bar_id = 2 + og;                  // its named barrier (128 threads)
    float *tile = reinterpret_cast<float *>(sm + G::OT) + og * 32 * LDT;
    const int ot = tid - 256 - 128 * og;        // thread of the warpgroup, 0..127
    const int c8 = ot & 15, r0 = ot >> 4;       // store phase: channels 8*c8.., tokens r0 + 8m
    const bool logits = gate && (flags & KDA_GATE_LOGITS);
    // this lane's O_intra^T row (this half's 32 tokens, bf16) of chunk c, from the card
    auto load_oi = [&](int c, uint4 *oi) {
      const uint8_t *card = card_of(c);
      if (c < nchunks && !card_ready(c, false)) c = nchunks;  // reported; the seed is then zero
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        oi[ch] = c < nchunks  // last use of these card lines (see fetch_bc)
                     ? __ldlu(reinterpret_cast<const uint4 *>(card + CARD_OIT + ((4 * og + ch) * 128 + j) * 16))
                     : make_uint4(0u, 0u, 0u, 0u);
    };
    auto seed = [&](int c, const uint4 *oi) {
      float x[32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) unpack8(oi[ch], x + ch * 8);
      tmem_st32(tmem_addr(tb, quad * 32, set_col(c) + 128 + 32 * og), x);
    };
    // gate of tokens 32 og + r0 + 8m, channels 8*c8 .. 8*c8 + 7 of chunk c (1.0 when absent)
    auto load_gate = [&](int c, uint4 *gq) {
      const int64_t tc0 = ts + (int64_t)c * C;
      const int lc = (int)min((int64_t)C, ls - (int64_t)c * C);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = 32 * og + r0 + 8 * m;
        gq[m] = (gate && c < nchunks && r < lc)
                    ? *reinterpret_cast<const uint4 *>(gate + ((size_t)(tc0 + r) * H + h) * DD + c8 * 8)
                    : make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
      }
    };
    {
      uint4 oi[4];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        load_oi(b, oi);
        seed(b, oi);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bar_ofree[0]);
    mbar_arrive(&bar_ofree[1]);
    uint32_t ofull_phase[2] = {0u, 0u};
    uint4 gq[4];
    load_gate(0, gq);
    bool ok = true;
    for (int n = 0; n < nchunks; ++n) {
      const int64_t t0 = ts + (int64_t)n * C;
      const int len = (int)min((int64_t)C, ls - (int64_t)n * C);
      uint4 oi[4];
      load_oi(n + 2, oi);  // its latency overlaps the wait below
      // every thread of the warpgroup takes the same branch, so a timeout strands none of them
      ok = named_bar_and(bar_id, 128, mbar_wait(&bar_ofull[n & 1], ofull_phase[n & 1]));
      if (!ok) break;
      ofull_phase[n & 1] ^= 1u;
      tc_fence_after();
      // this half into the half-tile (token row, this lane's channel), 16 tokens at a time
      // (the registers of the 88-register budget that oi and gq leave)
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        float t[16];
        tmem_ld16(tmem_addr(tb, quad * 32, set_col(n) + 128 + 32 * og + 16 * q), t);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 16; ++u) tile[(16 * q + u) * LDT + j] = t[u];
      }
      // the half is read: seed it with O_intra^T of chunk n + 2, hand it back to the issuer
      seed(n + 2, oi);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar_ofree[n & 1]);
      named_bar(bar_id, 128);  // half-tile complete
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int rr = r0 + 8 * m, r = 32 * og + rr;
        const float4 a = *reinterpret_cast<const float4 *>(tile + rr * LDT + c8 * 8);
        const float4 b = *reinterpret_cast<const float4 *>(tile + rr * LDT + c8 * 8 + 4);
        float g8[8], e[8];
        unpack8(gq[m], g8);
        const float x8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int u = 0; u < 8; ++u)
          e[u] = scale * (logits ? sigmoid_approx(g8[u]) : g8[u]) * x8[u];
        if (r < len)
          *reinterpret_cast<uint4 *>(out + ((size_t)(t0 + r) * H + h) * DD + c8 * 8) = pack8(e);
      }
      load_gate(n + 1, gq);  // the next chunk's gate, while its MMAs run
      named_bar(bar_id, 128);  // half-tile consumed before the next chunk overwrites it
    }
    if (!ok && ot == 0) atomicOr(sh.err, kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (own_tmem && warp == 0) tmem_dealloc(tb, 512);
}

// ===========================================================================
// Segment summary of one (segment, head) chain: the transition X (entry I, no B_c) and the
// zero-entry state Z (entry 0) walked by one CTA, so that a summary needs one CTA instead of
// two and shares each card copy between them. Warps 0-7 carry X, warps 8-15 Z; each group is
// laid out as the state warps of state_body (lane quadrant = warp % 4, 64 key columns per
// warpgroup half) and works 32 key columns at a time to stay within 128 registers. Tensor
// memory: per accumulator set b (chunk n uses b = n % 2) X^T at [256b, 256b + 128) and Z^T at
// [256b + 128, 256b + 256). Per chunk, thread 0 issues the two chains' MMA groups (eight
// M = 128, N = 128, K = 16 steps each, the same card operand) once both groups have staged;
// every step is the one state_body's summary pass takes for its chain, so the results are the
// same bits.
constexpr int kSumNst = 4;                          // card ring depth
constexpr int kSumStage = 33792;                    // Phi'^T (32768) + e^{G_C} (512), 1 KB rounded
constexpr int kSumSA = kSumNst * kSumStage;         // bf16 X^T operand, then Z^T's at +32768
constexpr int kSumDyn = kSumSA + 2 * 32768 + 1024;  // with alignment slack

struct SummaryShared {
  uint8_t *sm;  // kSumDyn - 1024 bytes, 1024-byte aligned
  uint64_t *bar_full, *bar_mma;  // [kSumNst], [1]
  uint32_t *tmem_base;
  int *s_fail;
  unsigned *err;
};

__device__ __forceinline__ void summary_body(const StateIn &p, const SummaryShared &sh, int chain,
                                             int tid) {
  const int32_t *__restrict__ cu = p.cu;
  const int H = p.H;
  if (cu != nullptr && p.meta->invalid) return;
  uint8_t *sm = sh.sm;
  const uint32_t sb = smem_u32(sm);
  const int h = chain % H;
  const int s = cu ? p.seq_order[chain / H] : chain / H;
  const int warp = tid >> 5, lane = tid & 31;
  const int zg = warp >> 3;              // 0: X, 1: Z
  const int quad = warp & 3;             // lane quadrant
  const int j = quad * 32 + lane;        // tensor-memory lane / column of X or Z
  const int half = (warp >> 2) & 1;      // which 64 key columns
  int64_t ts, ls;
  seq_range(cu, p.fixed_len, s, &ts, &ls);
  const int nchunks = (int)((ls + C - 1) / C);
  const int cbase = nchunks > 0 ? (cu ? p.off[s] : s * nchunks) : 0;
  auto card_of = [&](int n) { return p.cards + ((size_t)(cbase + n) * H + h) * CARD_BYTES; };
  float *res = (zg ? p.Z_out : p.X_out) + ((size_t)s * H + h) * DD * DD;
  if (nchunks == 0) {  // X = I, Z = 0
    for (int c = 64 * half; c < 64 * half + 64; ++c) res[(size_t)c * DD + j] = (!zg && c == j);
    return;
  }
  if (warp == 0) {
    tmem_alloc(sh.tmem_base, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kSumNst; ++i) mbar_init(&sh.bar_full[i], 1);
    mbar_init(sh.bar_mma, 1);
    fence_mbar_init();
    *sh.s_fail = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *sh.tmem_base;
  auto set_col = [](int n) { return 256 * (n & 1); };
  int loads_issued = 0, loads_done = 0;
  uint32_t full_phase[kSumNst] = {}, mma_phase = 0u;
  bool ok = true;
  const bool loader = (tid == 32);
  auto load_card = [&](int n) {
    const int st = n % kSumNst;
    uint8_t *dst = sm + st * kSumStage;
    const uint8_t *src = card_of(n);
    mbar_arrive_expect_tx(&sh.bar_full[st], 32768 + 512);
    bulk_g2s(dst, src + CARD_PHIQ, 16384, &sh.bar_full[st]);
    bulk_g2s(dst + 16384, src + CARD_PHIQ + 16384, 16384, &sh.bar_full[st]);
    bulk_g2s(dst + 32768, src + CARD_D, 512, &sh.bar_full[st]);
    // B_c^T (read by the Z group with plain loads two chunks later) into L2
    prefetch_l2(src + CARD_BCT, 32768);
    ++loads_issued;
  };
  auto wait_full = [&](int n) -> bool {
    const int st = n % kSumNst;
    const bool r = mbar_wait(&sh.bar_full[st], full_phase[st]);
    full_phase[st] ^= 1u;
    if (r) ++loads_done;
    return r;
  };
  // Z group: this thread's 64 columns of B_c^T row j of chunk n (lane-interleaved in the card)
  uint4 bcr[8];
  auto fetch_bc = [&](int n) {
    if (!zg || n >= nchunks) return;
    const uint8_t *src = card_of(n) + CARD_BCT;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      bcr[c8] = *reinterpret_cast<const uint4 *>(src + ((8 * half + c8) * 128 + j) * 16);
  };
  uint8_t *sa = sm + kSumSA + zg * 32768;  // this group's bf16 operand tile
  // accumulator <- Diag(e^{G_C}) S + B_c (Z) and the bf16 operand from the 32 key columns
  // 64 * half + 32 * qq of this thread's row, for chunk n
  auto stage_piece = [&](int n, int qq, const float *x) {
    const float *dv = reinterpret_cast<const float *>(sm + (n % kSumNst) * kSumStage + 32768);
    const int q4 = 2 * half + qq;
    float init[32];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      float bc[8];
      if (zg) unpack8(bcr[qq * 4 + ch], bc);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = q4 * 32 + ch * 8 + u;
        init[ch * 8 + u] = dv[c] * x[ch * 8 + u] + (zg ? bc[u] : 0.f);
      }
      *reinterpret_cast<uint4 *>(sa + sw128_chunk(j, q4 * 4 + ch, 128)) = pack8(x + ch * 8);
    }
    tmem_st32(tmem_addr(tb, quad * 32, set_col(n) + 128 * zg + 32 * q4), init);
  };
  auto issue_mma = [&](int n) {  // by thread 0
    const uint32_t stg = sb + (n % kSumNst) * kSumStage;
    const uint32_t id = idesc_bf16(128, 128, 0, 1);
    for (int g = 0; g < 2; ++g)
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16(tb + set_col(n) + 128 * g, desc_kmajor(sb + kSumSA + g * 32768, 128, kk),
                 sdesc_sw128(stg + kk * 2048, 128 * 128, 1024), id, 1u);
    mma_commit(sh.bar_mma);
  };
  if (loader)
    for (int n = 0; n < kSumNst && n < nchunks; ++n) load_card(n);
  fetch_bc(0);
  if (!wait_full(0)) ok = false;
  if (ok) {
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
      float x[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) x[u] = (!zg && 64 * half + 32 * qq + u == j) ? 1.f : 0.f;
      stage_piece(0, qq, x);
    }
    tmem_wait_st();
    fence_async_smem();
    tc_fence_before();
  }
  ok = named_bar_and(1, 512, ok);
  tc_fence_after();
  if (tid == 0 && ok) issue_mma(0);
  fetch_bc(1);
  for (int n = 0; n < nchunks && ok; ++n) {
    bool good = mbar_wait(sh.bar_mma, mma_phase);
    mma_phase ^= 1u;
    tc_fence_after();
    if (good && loader && n + kSumNst < nchunks) load_card(n + kSumNst);
    const bool last = (n + 1 == nchunks);
    if (good && !last) good = wait_full(n + 1);
    if (good) {
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        float x[32];
        tmem_ld32(tmem_addr(tb, quad * 32, set_col(n) + 128 * zg + 64 * half + 32 * qq), x);
        tmem_wait_ld();
        if (last) {
#pragma unroll
          for (int u = 0; u < 32; ++u) res[(size_t)(64 * half + 32 * qq + u) * DD + j] = x[u];
        } else {
          stage_piece(n + 1, qq, x);
        }
      }
    }
    if (last) {
      if (!good) ok = false;
      break;
    }
    if (good) {
      tmem_wait_st();
      fence_async_smem();
      tc_fence_before();
    }
    ok = named_bar_and(1, 512, good);
    tc_fence_after();
    if (!ok) break;
    if (tid == 0) issue_mma(n + 1);
    fetch_bc(n + 2);
  }
  if (!ok) {
    if (lane == 0) atomicOr(sh.err, kErrTimeout);
    if (loader)  // copies still in flight land (bounded) before shared memory is released
      for (int n = loads_done; n < loads_issued; ++n) {
        const int st = n % kSumNst;
        if (!mbar_wait(&sh.bar_full[st], full_phase[st], 100000000ull)) break;
        full_phase[st] ^= 1u;
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace tsb
}  // namespace kda
