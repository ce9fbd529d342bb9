// Chunked KDA forward, SIMT fp32 path.
//
// The chunked form follows from the recurrence S_t = (I - b k k^T) Diag(a) S + b k v^T
// (K3 training overview, zuoshipin.com/article/18261, section 2 "KDA") and the
// FlashKDA split the same page describes in section 4: per-chunk "update cards"
// are prepared in parallel, and only the state hand-off and read-out run in
// order. For a 64-token chunk with entry state S, G_r the inclusive running sum
// of log_alpha inside the chunk, Kt = k*e^{G}, Kh = k*e^{-G}, Qt = q*e^{G},
// Kd = k*e^{G_C - G}:
//   M  = strict_lower(diag(b) Kt Kh^T),   P = lower(Qt Kh^T)
//   (I + M) [W | Ut] = [diag(b) Kt | diag(b) V]            (forward substitution)
//   U  = Ut - W S
//   O  = Qt S + P U,        o = scale * g * O
//   S' = Diag(e^{G_C}) S + Kd^T U
// Stage A (kda_prep_simt) runs over all (chunk, head) pairs at once and writes
// W, Ut, Qt, Kd, P and e^{G_C}; stage B (kda_state_simt) walks the chunks of
// one (sequence, head) in order for a slice of value columns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"

namespace kda {

__device__ unsigned g_chunk_err;

namespace {

constexpr int C = kChunk;

__device__ __forceinline__ void set_err(unsigned bits) { atomicOr(&g_chunk_err, bits); }

// Find the sequence owning global chunk `ci`: largest s with off[s] <= ci.
__device__ __forceinline__ int find_seq(const int *off, int n_seq, int ci) {
  int lo = 0, hi = n_seq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= ci) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void seq_range(const int32_t *cu, int64_t fixed_len, int s,
                                          int64_t *t0, int64_t *len) {
  if (cu) {
    *t0 = cu[s];
    *len = (int64_t)cu[s + 1] - cu[s];
  } else {
    *t0 = (int64_t)s * fixed_len;
    *len = fixed_len;
  }
}

// Exclusive prefix sum of `local` over the block (1024 threads), in thread order.
__device__ int block_exclusive_scan(int local, int *warp_tot) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, w = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();  // warp_tot may still be read from a previous scan
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = (lane < (nt >> 5)) ? warp_tot[lane] : 0;
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += y;
    }
    warp_tot[lane] = xi - x;  // exclusive
  }
  __syncthreads();
  return warp_tot[w] + incl - local;
}

// One block: validate cu_seqlens and build per-sequence chunk offsets. For a split prefill
// with nb inner part boundaries (bound64[0 .. nb), in 64ths of each sequence's chunks), also
// the running sums over the sequences of floor(n_s * bound64[i] / 64), one [n_seq + 1] array
// per boundary in off_b.
__global__ void __launch_bounds__(1024) kda_chunk_table(const int32_t *cu, int n_seq,
                                                        int64_t T_total, ChunkMeta *meta,
                                                        int *off, int nb, int4 bound64,
                                                        int *off_b, int *order) {
  __shared__ int warp_tot[32];
  __shared__ int bad;
  __shared__ int s_chunks[kOrderMax];
  const int tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) bad = 0;
  __syncthreads();
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  // contiguous range of sequences per thread
  const int per = (n_seq + nt - 1) / nt;
  const int s_lo = min(n_seq, tid * per), s_hi = min(n_seq, s_lo + per);
  auto chunks_of = [&](int s) -> int {
    const int64_t len = cu ? (int64_t)cu[s + 1] - cu[s] : fixed_len;
    return len < 0 ? 0 : (int)((len + C - 1) / C);
  };
  int local = 0;
  for (int s = s_lo; s < s_hi; ++s) {
    if (cu && (int64_t)cu[s + 1] - cu[s] < 0) bad = 1;
    local += chunks_of(s);
  }
  if (cu && tid == 0 && (cu[0] != 0 || (int64_t)cu[n_seq] != T_total)) bad = 1;
  int run = block_exclusive_scan(local, warp_tot);
  for (int s = s_lo; s < s_hi; ++s) {
    off[s] = run;
    run += chunks_of(s);
  }
  if (s_hi == n_seq && s_lo < s_hi) off[n_seq] = run;
  for (int i = 0; i < nb; ++i) {  // nb is uniform: every thread takes part in each scan
    const int b = i == 0 ? bound64.x : bound64.y;
    auto lead = [&](int s) { return (int)((int64_t)chunks_of(s) * b / 64); };
    int local_b = 0;
    for (int s = s_lo; s < s_hi; ++s) local_b += lead(s);
    int *ob = off_b + (size_t)i * (n_seq + 1);
    int run_b = block_exclusive_scan(local_b, warp_tot);
    for (int s = s_lo; s < s_hi; ++s) {
      ob[s] = run_b;
      run_b += lead(s);
    }
    if (s_hi == n_seq && s_lo < s_hi) ob[n_seq] = run_b;
    if (n_seq == 0 && tid == 0) ob[0] = 0;
  }
  if (n_seq == 0 && tid == 0) off[0] = 0;
  if (order) {
    // longest first: rank = sequences with more chunks, or as many and a lower index
    if (n_seq <= kOrderMax) {
      for (int s = tid; s < n_seq; s += nt) s_chunks[s] = chunks_of(s);
      __syncthreads();
      for (int s = tid; s < n_seq; s += nt) {
        const int c = s_chunks[s];
        int r = 0;
        for (int t = 0; t < n_seq; ++t) r += (s_chunks[t] > c) || (s_chunks[t] == c && t < s);
        order[r] = s;
      }
    } else {
      for (int s = tid; s < n_seq; s += nt) order[s] = s;
    }
  }
  __syncthreads();
  if (tid == 0) {
    meta->invalid = bad;
    meta->total_chunks = bad ? 0 : off[n_seq];
    if (bad) set_err(kErrBadSeqlens);
  }
}

// ---------------------------------------------------------------------------
// Stage A: per (chunk, head) preparation. 256 threads, one CTA per (chunk, head), two CTAs per
// SM (115,456 bytes of shared memory at dk = dv = 128), so that one CTA's global loads and
// stores overlap the other's arithmetic.
// The [64][d] fp32 tiles are stored without padding, the 16-byte chunk x of row r at x ^ (r & 7):
// a warp reading four channels of eight different rows, or one channel of a row per lane, hits
// every bank once. The products read their operands as 16-byte vectors (one shared-memory
// instruction per four FMAs of a thread). V takes the tile of Qt once the Gram products have
// read it; the log-alpha partial sums of the decay take the Gram tile before it is written.
template <int DK, int DV>
struct PrepLayout {
  static constexpr int DQV = DK > DV ? DK : DV;
  static constexpr int KT = 0, KH = KT + C * DK, QV = KH + C * DK, A = QV + C * DQV,
                       B = A + C * C, GC = B + C;
  static constexpr int FLOATS = GC + DK;
  static_assert(256 <= C * C, "the decay's partial sums fit in the Gram tile");
};

// element (r, c) of a swizzled tile with D floats per row; v4: the 16-byte chunk holding c
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
  return r * D + ((((c >> 2) ^ (r & 7)) << 2) | (c & 3));
}
__device__ __forceinline__ float4 lds4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void sts4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float4 mul4(float4 x, float b) {
  return make_float4(x.x * b, x.y * b, x.z * b, x.w * b);
}

template <int DK, int DV, typename Tin>
__global__ void __launch_bounds__(256, 2) kda_prep_simt(
    const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
    const Tin *__restrict__ la, const Tin *__restrict__ beta, const int32_t *__restrict__ cu,
    int n_seq, int64_t fixed_len, int H, unsigned flags, const ChunkMeta *__restrict__ meta,
    const int *__restrict__ off, float *__restrict__ Wg, float *__restrict__ Ug,
    float *__restrict__ Qg, float *__restrict__ Kdg, float *__restrict__ Pg,
    float *__restrict__ Dg, int need_q, PrepSave save) {
  using Ly = PrepLayout<DK, DV>;
  extern __shared__ __align__(16) float smem[];
  float *sKt = smem + Ly::KT;  // [C][DK]  log alpha, then k*e^{G}, then b*Kt, then W
  float *sKh = smem + Ly::KH;  // [C][DK]  k, then k*e^{-G}
  float *sQV = smem + Ly::QV;  // [C][DK]  q, then q*e^{G}; then [C][DV] b*v, then Ut
  float *sA = smem + Ly::A;    // [C][C]   strict-lower diag(b) Kt Kh^T (first: partial sums)
  float *sB = smem + Ly::B;    // [C]      beta
  float *sGC = smem + Ly::GC;  // [DK]     e^{G_C}

  const int ci = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  if (meta->invalid || ci >= meta->total_chunks) return;
  const int s = find_seq(off, n_seq, ci);
  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int j = ci - off[s];
  const int64_t t0 = ts + (int64_t)j * C;
  const int len = (int)min((int64_t)C, ls - (int64_t)j * C);
  const size_t slab = (size_t)ci * H + h;

  // load q, k, log alpha and beta (rows >= len are zero: no write, no read-out, no decay),
  // every load issued before any use. Each row of q and k is held by DK / 8 consecutive lanes,
  // so the L2 norms are reduced in registers.
  {
    constexpr int NVK = C * DK / 8 / 256, LPR = DK / 8;
    float kv[NVK][8], qv[NVK][8], lv[NVK][8];
    float b = 0.f;
    if (tid < len) b = to_f32(beta[(size_t)(t0 + tid) * H + h]);
#pragma unroll
    for (int m = 0; m < NVK; ++m) {
      const int e = 8 * (tid + 256 * m), r = e / DK, c = e % DK;
      if (r < len) {
        const size_t g = ((size_t)(t0 + r) * H + h) * DK + c;
        load8(k + g, kv[m]);
        load8(q + g, qv[m]);
        load8(la + g, lv[m]);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) kv[m][u] = qv[m][u] = lv[m][u] = 0.f;
      }
    }
    if (tid < C) {
      b = tid < len ? prep_beta(b, flags) : 0.f;
      if ((flags & KDA_DEBUG_CHECK) && tid < len && !(b >= 0.f && b <= 1.f)) set_err(kErrPrecondition);
      sB[tid] = b;
    }
    if (flags & KDA_QK_L2NORM) {  // rows >= len are zero and stay zero
#pragma unroll
      for (int m = 0; m < NVK; ++m) {
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          sk = fmaf(kv[m][u], kv[m][u], sk);
          sq = fmaf(qv[m][u], qv[m][u], sq);
        }
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) {
          sk += __shfl_xor_sync(0xffffffffu, sk, o);
          sq += __shfl_xor_sync(0xffffffffu, sq, o);
        }
        const float rk = rsqrtf(sk + kL2Eps), rq = rsqrtf(sq + kL2Eps);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          kv[m][u] *= rk;
          qv[m][u] *= rq;
        }
      }
    }
#pragma unroll
    for (int m = 0; m < NVK; ++m) {
      const int e = 8 * (tid + 256 * m), r = e / DK, c = e % DK;
      float l[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        l[u] = 0.f;
        if (r < len) {
          l[u] = prep_log_alpha(lv[m][u], flags);
          if ((flags & KDA_DEBUG_CHECK) && !(l[u] >= kLogAlphaMin && l[u] <= 0.f)) set_err(kErrPrecondition);
        }
      }
#pragma unroll
      for (int h4 = 0; h4 < 8; h4 += 4) {
        const int o = swz<DK>(r, c + h4);
        sts4(sKh + o, make_float4(kv[m][h4], kv[m][h4 + 1], kv[m][h4 + 2], kv[m][h4 + 3]));
        sts4(sQV + o, make_float4(qv[m][h4], qv[m][h4 + 1], qv[m][h4 + 2], qv[m][h4 + 3]));
        sts4(sKt + o, make_float4(l[h4], l[h4 + 1], l[h4 + 2], l[h4 + 3]));
      }
    }
  }
  __syncthreads();

  // running log-decay G per key channel and the decayed operands: TPC threads per channel,
  // each over RPT consecutive rows, offset by the sums of the rows before them
  {
    constexpr int TPC = 256 / DK, RPT = C / TPC;
    const int c = tid % DK, part = tid / DK, rb = part * RPT;
    float *sPart = sA;
    float sum = 0.f;
#pragma unroll 8
    for (int r = rb; r < rb + RPT; ++r) sum += sKt[swz<DK>(r, c)];
    sPart[part * DK + c] = sum;
    __syncthreads();
    float G = 0.f;
    for (int p = 0; p < part; ++p) G += sPart[p * DK + c];
#pragma unroll 4
    for (int r = rb; r < rb + RPT; ++r) {
      const int o = swz<DK>(r, c);
      G += sKt[o];  // log_alpha (0 on padded rows)
      const float ep = expf(G), en = expf(-G);
      const float kn = sKh[o];
      sKt[o] = kn * ep;
      sKh[o] = kn * en;
      sQV[o] *= ep;
    }
    if (part == TPC - 1) sGC[c] = expf(G);
  }
  __syncthreads();

  // Gram blocks: A = strict_lower(diag(b) Kt Kh^T), P = lower(Qt Kh^T). Thread (rg, cg) owns
  // rows rg + 16 i and columns cg + 16 j (i, j < 4); a step reads four channels of each row.
  {
    const int rg = tid >> 4, cg = tid & 15;
    float a[4][4] = {}, p[4][4] = {};
#pragma unroll 2
    for (int c = 0; c < DK; c += 4) {
      float4 kt[4], qt[4], kh[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kt[i] = lds4(sKt + swz<DK>(rg + 16 * i, c));
        qt[i] = lds4(sQV + swz<DK>(rg + 16 * i, c));
        kh[i] = lds4(sKh + swz<DK>(cg + 16 * i, c));
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          a[i][jj] = fmaf(kt[i].x, kh[jj].x, a[i][jj]);
          a[i][jj] = fmaf(kt[i].y, kh[jj].y, a[i][jj]);
          a[i][jj] = fmaf(kt[i].z, kh[jj].z, a[i][jj]);
          a[i][jj] = fmaf(kt[i].w, kh[jj].w, a[i][jj]);
          p[i][jj] = fmaf(qt[i].x, kh[jj].x, p[i][jj]);
          p[i][jj] = fmaf(qt[i].y, kh[jj].y, p[i][jj]);
          p[i][jj] = fmaf(qt[i].z, kh[jj].z, p[i][jj]);
          p[i][jj] = fmaf(qt[i].w, kh[jj].w, p[i][jj]);
        }
    }
    float *Pout = Pg + slab * C * C;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int r = rg + 16 * i, c2 = cg + 16 * jj;
        sA[r * C + c2] = c2 < r ? sB[r] * a[i][jj] : 0.f;
        Pout[r * C + c2] = c2 <= r ? p[i][jj] : 0.f;
      }
  }
  __syncthreads();

  // v is loaded while Qt, Kd = Kh * e^{G_C}, e^{G_C} and the save of Kh are written and the
  // right-hand side Kt is scaled by beta; once every read of Qt is done, b*v takes its tile
  {
    constexpr int NVV = C * DV / 8 / 256, NK4 = C * DK / 4 / 256;
    float vv[NVV][8];
#pragma unroll
    for (int m = 0; m < NVV; ++m) {
      const int e = 8 * (tid + 256 * m), r = e / DV, c = e % DV;
      if (r < len) {
        load8(v + ((size_t)(t0 + r) * H + h) * DV + c, vv[m]);
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) vv[m][u] = 0.f;
      }
    }
    float *Qout = Qg + slab * C * DK, *Kdout = Kdg + slab * C * DK;
#pragma unroll
    for (int m = 0; m < NK4; ++m) {
      const int e = 4 * (tid + 256 * m), r = e / DK, c = e % DK, o = swz<DK>(r, c);
      const float4 kh = lds4(sKh + o), g = lds4(sGC + c);
      sts4(Kdout + e, make_float4(kh.x * g.x, kh.y * g.y, kh.z * g.z, kh.w * g.w));
      if (save.Kh) sts4(save.Kh + slab * C * DK + e, kh);
      if (need_q) sts4(Qout + e, lds4(sQV + o));
      sts4(sKt + o, mul4(lds4(sKt + o), sB[r]));
    }
    if (tid < DK) Dg[slab * DK + tid] = sGC[tid];
    __syncthreads();  // Qt is read
#pragma unroll
    for (int m = 0; m < NVV; ++m) {
      const int e = 8 * (tid + 256 * m), r = e / DV, c = e % DV;
      const float b = sB[r];
#pragma unroll
      for (int h4 = 0; h4 < 8; h4 += 4)
        sts4(sQV + swz<DV>(r, c + h4),
             make_float4(vv[m][h4] * b, vv[m][h4 + 1] * b, vv[m][h4 + 2] * b, vv[m][h4 + 3] * b));
    }
  }
  __syncthreads();

  // (I + A) X = [b Kt | b V], forward substitution: one thread per column, the column in
  // registers (indices fixed at compile time), each row's dot product in four partial sums
  // (column i into sum i mod 4), the row of A read as 16-byte vectors. The saved b*Kt column
  // is written from the registers it is solved in.
  if (tid < DK + DV) {
    const bool kcol = tid < DK;
    const int c = kcol ? tid : tid - DK, D = kcol ? DK : DV;
    float *base = kcol ? sKt : sQV;
    int coff[8];  // swizzled offset of column c in a row r with r & 7 = i
#pragma unroll
    for (int i = 0; i < 8; ++i) coff[i] = (((c >> 2) ^ i) << 2) | (c & 3);
    float x[C];
#pragma unroll
    for (int r = 0; r < C; ++r) x[r] = base[r * D + coff[r & 7]];
    if (save.Bk && kcol) {
      float *bk = save.Bk + slab * C * DK + c;
#pragma unroll
      for (int r = 0; r < C; ++r) bk[r * DK] = x[r];
    }
#pragma unroll
    for (int r = 1; r < C; ++r) {
      const float *Ar = sA + r * C;
      float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < r; i += 4) {
        const float4 a4 = lds4(Ar + i);
        p[0] = fmaf(a4.x, x[i], p[0]);
        if (i + 1 < r) p[1] = fmaf(a4.y, x[i + 1], p[1]);
        if (i + 2 < r) p[2] = fmaf(a4.z, x[i + 2], p[2]);
        if (i + 3 < r) p[3] = fmaf(a4.w, x[i + 3], p[3]);
      }
      x[r] -= (p[0] + p[1]) + (p[2] + p[3]);
    }
#pragma unroll
    for (int r = 1; r < C; ++r) base[r * D + coff[r & 7]] = x[r];
  }
  __syncthreads();

  // write W, Ut and the save of A
  {
    float *Wout = Wg + slab * C * DK, *Uout = Ug + slab * C * DV;
    constexpr int NK4 = C * DK / 4 / 256, NV4 = C * DV / 4 / 256, NA4 = C * C / 4 / 256;
#pragma unroll
    for (int m = 0; m < NK4; ++m) {
      const int e = 4 * (tid + 256 * m);
      sts4(Wout + e, lds4(sKt + swz<DK>(e / DK, e % DK)));
    }
#pragma unroll
    for (int m = 0; m < NV4; ++m) {
      const int e = 4 * (tid + 256 * m);
      sts4(Uout + e, lds4(sQV + swz<DV>(e / DV, e % DV)));
    }
    if (save.A)
#pragma unroll
      for (int m = 0; m < NA4; ++m) {
        const int e = 4 * (tid + 256 * m);
        sts4(save.A + slab * C * C + e, lds4(sA + e));
      }
  }
}

// ---------------------------------------------------------------------------
// Stage B: sequential state pass for one (sequence, head) and BV value columns.
// mode 0: prefill (reads Qt/P, writes out and the final state)
// mode 1: segment summary on the augmented state [X | Z]: columns < DK carry X
//         (entry = identity, no value input), the rest carry Z (entry = 0).
constexpr int BV = 32;

template <int DK, int DV, typename Tout>
__global__ void __launch_bounds__(256) kda_state_simt(
    int mode, unsigned flags, const Tout *__restrict__ gate, Tout *__restrict__ out,
    const float *__restrict__ S0, float *__restrict__ S_final, float *__restrict__ X_out,
    float *__restrict__ Z_out, const int32_t *__restrict__ cu, int n_seq, int64_t fixed_len,
    int H, float scale, const ChunkMeta *__restrict__ meta, const int *__restrict__ off,
    const float *__restrict__ Wg, const float *__restrict__ Ug, const float *__restrict__ Qg,
    const float *__restrict__ Kdg, const float *__restrict__ Pg, const float *__restrict__ Dg,
    CkptOut ck, StateSave save) {
  // Register-tiled: thread (rg, cg) = (tid >> 3, tid & 7) owns value columns 4cg..4cg+3 of
  // this slice, rows 2rg, 2rg+1 of U and O and key rows 4rg..4rg+3 of S. Operands are read
  // from shared memory as 8- and 16-byte vectors; W, Q~ and P are stored transposed.
  constexpr int LS = BV + 4, LK = DK + 4, LT = C + 2;
  extern __shared__ __align__(16) float smem[];
  // Q~^T and P^T come last: without an output they are not allocated (two blocks per SM)
  float *sS = smem;            // [DK][LS]  state slice
  float *sU = sS + DK * LS;    // [C][LS]   U~, then U
  float *sWt = sU + C * LS;    // [DK][LT]  W^T
  float *sKd = sWt + DK * LT;  // [C][LK]   K_d
  float *sD = sKd + C * LK;    // [DK]
  float *sQt = sD + DK;        // [DK][LT]  Q~^T   (with an output only)
  float *sPt = sQt + DK * LT;  // [C][LT]   P^T    (with an output only)

  if (meta->invalid) return;
  const int chain = blockIdx.x, s = chain / H, h = chain % H, tid = threadIdx.x;
  const int j0 = blockIdx.y * BV;
  const int cg = tid & 7, rg = tid >> 3, jl = 4 * cg, r0 = 2 * rg;
  const bool s_rows = rg < DK / 4;
  bool xpart = false;
  int vcol0 = j0;  // first value column of this slice (mode 0 / Z part)
  if (mode == 1) {
    xpart = j0 < DK;
    vcol0 = j0 - DK;
  }
  // entry state
  for (int e = tid; e < DK * BV; e += 256) {
    const int c = e / BV, jj = e % BV;
    float x = 0.f;
    if (mode == 0) {
      if (S0) x = S0[(((size_t)s * H + h) * DK + c) * DV + j0 + jj];
    } else if (xpart) {
      x = (c == j0 + jj) ? 1.f : 0.f;
    }
    sS[c * LS + jj] = x;
  }
  int64_t ts, ls;
  seq_range(cu, fixed_len, s, &ts, &ls);
  const int nchunks = (int)((ls + C - 1) / C);
  const bool write_o = (mode == 0) && out != nullptr;
  const bool need_o = write_o || (mode == 0 && save.O != nullptr);
  __syncthreads();

  for (int jc = 0; jc < nchunks; ++jc) {
    const size_t slab = (size_t)(off[s] + jc) * H + h;
    if (tid == 0 && blockIdx.y == 0 && jc + 1 < nchunks) {  // the next chunk's operands into L2
      const size_t sn = slab + H;                             // chunk jc + 1, same head
      prefetch_l2_bulk(Wg + sn * C * DK, C * DK * 4);
      prefetch_l2_bulk(Kdg + sn * C * DK, C * DK * 4);
      prefetch_l2_bulk(Ug + sn * C * DV, C * DV * 4);
      if (need_o) {
        prefetch_l2_bulk(Qg + sn * C * DK, C * DK * 4);
        prefetch_l2_bulk(Pg + sn * C * C, C * C * 4);
      }
    }
    const int64_t t0 = ts + (int64_t)jc * C;
    const int len = (int)min((int64_t)C, ls - (int64_t)jc * C);
    const float *W = Wg + slab * C * DK, *Kd = Kdg + slab * C * DK;
    if (mode == 0 && save.Sb)  // state entering chunk jc
      for (int e = tid; e < DK * BV; e += 256) {
        const int c = e / BV, jj = e % BV;
        save.Sb[(slab * DK + c) * DV + j0 + jj] = sS[c * LS + jj];
      }
    // operands of chunk jc: 16-byte loads, each batch issued before any of its stores
    {
      constexpr int NK = C * DK / 4 / 256;  // float4 per thread of a [C, DK] matrix
      float4 rw[NK], rk[NK];
#pragma unroll
      for (int m = 0; m < NK; ++m) {
        rw[m] = *reinterpret_cast<const float4 *>(W + 4 * (tid + 256 * m));
        rk[m] = *reinterpret_cast<const float4 *>(Kd + 4 * (tid + 256 * m));
      }
#pragma unroll
      for (int m = 0; m < NK; ++m) {
        const int e = 4 * (tid + 256 * m), r = e / DK, c = e % DK;
        sWt[(c + 0) * LT + r] = rw[m].x; sWt[(c + 1) * LT + r] = rw[m].y;
        sWt[(c + 2) * LT + r] = rw[m].z; sWt[(c + 3) * LT + r] = rw[m].w;
        *reinterpret_cast<float4 *>(sKd + r * LK + c) = rk[m];
      }
      if (need_o) {
        const float *Q = Qg + slab * C * DK, *P = Pg + slab * C * C;
        constexpr int NP = C * C / 4 / 256;
        float4 rp[NP];
#pragma unroll
        for (int m = 0; m < NK; ++m) rw[m] = *reinterpret_cast<const float4 *>(Q + 4 * (tid + 256 * m));
#pragma unroll
        for (int m = 0; m < NP; ++m) rp[m] = *reinterpret_cast<const float4 *>(P + 4 * (tid + 256 * m));
#pragma unroll
        for (int m = 0; m < NK; ++m) {
          const int e = 4 * (tid + 256 * m), r = e / DK, c = e % DK;
          sQt[(c + 0) * LT + r] = rw[m].x; sQt[(c + 1) * LT + r] = rw[m].y;
          sQt[(c + 2) * LT + r] = rw[m].z; sQt[(c + 3) * LT + r] = rw[m].w;
        }
#pragma unroll
        for (int m = 0; m < NP; ++m) {
          const int e = 4 * (tid + 256 * m), r = e / C, i = e % C;
          sPt[(i + 0) * LT + r] = rp[m].x; sPt[(i + 1) * LT + r] = rp[m].y;
          sPt[(i + 2) * LT + r] = rp[m].z; sPt[(i + 3) * LT + r] = rp[m].w;
        }
      }
      constexpr int NU = C * BV / 4 / 256;
#pragma unroll
      for (int m = 0; m < NU; ++m) {
        const int e = 4 * (tid + 256 * m), r = e / BV, jj = e % BV;
        const float4 x = xpart ? make_float4(0.f, 0.f, 0.f, 0.f)
                               : *reinterpret_cast<const float4 *>(
                                     Ug + slab * C * DV + (size_t)r * DV + vcol0 + jj);
        *reinterpret_cast<float4 *>(sU + r * LS + jj) = x;
      }
      if (tid < DK) sD[tid] = Dg[slab * DK + tid];
    }
    __syncthreads();

    // U = U~ - W S   (rows r0, r0 + 1)
    float u0[4], u1[4];
    {
      const float4 a = *reinterpret_cast<const float4 *>(sU + r0 * LS + jl);
      const float4 b = *reinterpret_cast<const float4 *>(sU + (r0 + 1) * LS + jl);
      u0[0] = a.x; u0[1] = a.y; u0[2] = a.z; u0[3] = a.w;
      u1[0] = b.x; u1[1] = b.y; u1[2] = b.z; u1[3] = b.w;
    }
#pragma unroll 4
    for (int c = 0; c < DK; ++c) {
      const float2 w = *reinterpret_cast<const float2 *>(sWt + c * LT + r0);
      const float4 x = *reinterpret_cast<const float4 *>(sS + c * LS + jl);
      u0[0] = fmaf(-w.x, x.x, u0[0]); u0[1] = fmaf(-w.x, x.y, u0[1]);
      u0[2] = fmaf(-w.x, x.z, u0[2]); u0[3] = fmaf(-w.x, x.w, u0[3]);
      u1[0] = fmaf(-w.y, x.x, u1[0]); u1[1] = fmaf(-w.y, x.y, u1[1]);
      u1[2] = fmaf(-w.y, x.z, u1[2]); u1[3] = fmaf(-w.y, x.w, u1[3]);
    }
    __syncthreads();  // every thread has read U~
    *reinterpret_cast<float4 *>(sU + r0 * LS + jl) = make_float4(u0[0], u0[1], u0[2], u0[3]);
    *reinterpret_cast<float4 *>(sU + (r0 + 1) * LS + jl) = make_float4(u1[0], u1[1], u1[2], u1[3]);
    if (mode == 0 && save.Ub) {
      *reinterpret_cast<float4 *>(save.Ub + (slab * C + r0) * DV + j0 + jl) =
          make_float4(u0[0], u0[1], u0[2], u0[3]);
      *reinterpret_cast<float4 *>(save.Ub + (slab * C + r0 + 1) * DV + j0 + jl) =
          make_float4(u1[0], u1[1], u1[2], u1[3]);
    }
    __syncthreads();

    if (need_o) {
      // O = Q~ S + P U   (P[r][i] = 0 for i > r)
      float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int c = 0; c < DK; ++c) {
        const float2 q = *reinterpret_cast<const float2 *>(sQt + c * LT + r0);
        const float4 x = *reinterpret_cast<const float4 *>(sS + c * LS + jl);
        o0[0] = fmaf(q.x, x.x, o0[0]); o0[1] = fmaf(q.x, x.y, o0[1]);
        o0[2] = fmaf(q.x, x.z, o0[2]); o0[3] = fmaf(q.x, x.w, o0[3]);
        o1[0] = fmaf(q.y, x.x, o1[0]); o1[1] = fmaf(q.y, x.y, o1[1]);
        o1[2] = fmaf(q.y, x.z, o1[2]); o1[3] = fmaf(q.y, x.w, o1[3]);
      }
      for (int i = 0; i <= r0 + 1; ++i) {
        const float2 p = *reinterpret_cast<const float2 *>(sPt + i * LT + r0);
        const float4 x = *reinterpret_cast<const float4 *>(sU + i * LS + jl);
        o0[0] = fmaf(p.x, x.x, o0[0]); o0[1] = fmaf(p.x, x.y, o0[1]);
        o0[2] = fmaf(p.x, x.z, o0[2]); o0[3] = fmaf(p.x, x.w, o0[3]);
        o1[0] = fmaf(p.y, x.x, o1[0]); o1[1] = fmaf(p.y, x.y, o1[1]);
        o1[2] = fmaf(p.y, x.z, o1[2]); o1[3] = fmaf(p.y, x.w, o1[3]);
      }
      const float *orow[2] = {o0, o1};
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        const int r = r0 + v;
        if (save.O)
          *reinterpret_cast<float4 *>(save.O + (slab * C + r) * DV + j0 + jl) =
              make_float4(orow[v][0], orow[v][1], orow[v][2], orow[v][3]);
        if (write_o && r < len)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const size_t g = ((size_t)(t0 + r) * H + h) * DV + j0 + jl + q;
            const float gv = gate ? prep_gate(to_f32(gate[g]), flags) : 1.f;
            out[g] = from_f32<Tout>(scale * gv * orow[v][q]);
          }
      }
    }

    // S = Diag(e^{G_C}) S + K_d^T U   (rows 4rg .. 4rg + 3)
    float ns[4][4];
    if (s_rows) {
      const int c0 = 4 * rg;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 x = *reinterpret_cast<const float4 *>(sS + (c0 + v) * LS + jl);
        const float d = sD[c0 + v];
        ns[v][0] = d * x.x; ns[v][1] = d * x.y; ns[v][2] = d * x.z; ns[v][3] = d * x.w;
      }
#pragma unroll 4
      for (int i = 0; i < C; ++i) {
        const float4 k4 = *reinterpret_cast<const float4 *>(sKd + i * LK + c0);
        const float4 x = *reinterpret_cast<const float4 *>(sU + i * LS + jl);
        const float ka[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          ns[v][0] = fmaf(ka[v], x.x, ns[v][0]); ns[v][1] = fmaf(ka[v], x.y, ns[v][1]);
          ns[v][2] = fmaf(ka[v], x.z, ns[v][2]); ns[v][3] = fmaf(ka[v], x.w, ns[v][3]);
        }
      }
    }
    __syncthreads();
    if (s_rows) {
#pragma unroll
      for (int v = 0; v < 4; ++v)
        *reinterpret_cast<float4 *>(sS + (4 * rg + v) * LS + jl) =
            make_float4(ns[v][0], ns[v][1], ns[v][2], ns[v][3]);
      if (mode == 0)
        if (float *cp = ckpt_after_chunk(ck, s, jc, ls, H, h, DK, DV))
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<float4 *>(cp + (size_t)(4 * rg + v) * DV + j0 + jl) =
                make_float4(ns[v][0], ns[v][1], ns[v][2], ns[v][3]);
    }
    __syncthreads();
  }

  // final state
  for (int e = tid; e < DK * BV; e += 256) {
    const int c = e / BV, jj = e % BV;
    const float x = sS[c * LS + jj];
    if (mode == 0) {
      if (S_final) S_final[(((size_t)s * H + h) * DK + c) * DV + j0 + jj] = x;
    } else if (xpart) {
      X_out[(((size_t)s * H + h) * DK + c) * DK + j0 + jj] = x;
    } else {
      Z_out[(((size_t)s * H + h) * DK + c) * DV + vcol0 + jj] = x;
    }
  }
}

template <int DK, int DV>
constexpr size_t prep_smem() {
  return sizeof(float) * PrepLayout<DK, DV>::FLOATS;
}
// shared memory of the state pass: without an output (segment summaries, the backward's
// forward replay) the Q~^T and P^T buffers are left out
template <int DK>
constexpr size_t state_smem(bool with_o) {
  return sizeof(float) * (DK * (BV + 4) + C * (BV + 4) + DK * (C + 2) + C * (DK + 4) + DK +
                          (with_o ? DK * (C + 2) + C * (C + 2) : 0));
}

template <int DK, int DV, typename Tin>
cudaError_t launch_prep_t(const void *q, const void *k, const void *v, const void *la,
                          const void *beta, const int32_t *cu, int n_seq, int64_t T_total,
                          int H, unsigned flags, const ChunkWs &ws, bool need_q,
                          cudaStream_t st, PrepSave save) {
  auto kern = kda_prep_simt<DK, DV, Tin>;
  constexpr size_t sm = prep_smem<DK, DV>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  // two CTAs per SM need the largest shared-memory carveout
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  dim3 grid(ws.max_chunks, H);
  kern<<<grid, 256, sm, st>>>((const Tin *)q, (const Tin *)k, (const Tin *)v, (const Tin *)la,
                              (const Tin *)beta, cu, n_seq, fixed_len, H, flags, ws.meta,
                              ws.seq_chunk_off, ws.W, ws.U, ws.Q, ws.Kd, ws.P, ws.D,
                              need_q ? 1 : 0, save);
  return cudaGetLastError();
}

template <int DK, int DV, typename Tout>
cudaError_t launch_state_t(int mode, unsigned flags, const void *gate, void *out, const float *S0,
                           float *S_final, float *X_out, float *Z_out, const int32_t *cu,
                           int n_seq, int64_t T_total, int H, float scale, const ChunkWs &ws,
                           cudaStream_t st, CkptOut ck, StateSave save) {
  auto kern = kda_state_simt<DK, DV, Tout>;
  const bool with_o = mode == 0 && (out != nullptr || save.O != nullptr);
  const size_t sm = state_smem<DK>(with_o);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)state_smem<DK>(true));
  if (e != cudaSuccess) return e;
  const int64_t fixed_len = (cu == nullptr && n_seq > 0) ? T_total / n_seq : 0;
  const int ncols = mode == 0 ? DV : DK + DV;
  dim3 grid(n_seq * H, ncols / BV);
  kern<<<grid, 256, sm, st>>>(mode, flags, (const Tout *)gate, (Tout *)out, S0, S_final, X_out, Z_out,
                              cu, n_seq, fixed_len, H, scale, ws.meta, ws.seq_chunk_off, ws.W,
                              ws.U, ws.Q, ws.Kd, ws.P, ws.D, ck, save);
  return cudaGetLastError();
}

}  // namespace

// ---------------------------------------------------------------------------
static size_t max_chunks_of(int64_t T_total, int n_seq) {
  // sum_s ceil(len_s / C) <= T_total / C + n_seq
  return (size_t)(T_total / C) + (size_t)n_seq + 1;
}

size_t chunk_ws_bytes(int64_t T_total, int n_seq, int H, int dk, int dv) {
  const size_t mc = max_chunks_of(T_total, n_seq);
  size_t b = align_up(sizeof(ChunkMeta), 256);
  b += align_up(sizeof(int) * (size_t)(n_seq + 1), 256);
  const size_t per = (size_t)mc * H;
  b += align_up(sizeof(float) * per * C * dk, 256) * 3;  // W, Q, Kd
  b += align_up(sizeof(float) * per * C * dv, 256);      // U
  b += align_up(sizeof(float) * per * C * C, 256);       // P
  b += align_up(sizeof(float) * per * dk, 256);          // D
  return b;
}

ChunkWs chunk_ws_carve(void *ws, int64_t T_total, int n_seq, int H, int dk, int dv) {
  ChunkWs w = {};
  const size_t mc = max_chunks_of(T_total, n_seq);
  char *p = (char *)ws;
  w.meta = (ChunkMeta *)p;
  p += align_up(sizeof(ChunkMeta), 256);
  w.seq_chunk_off = (int *)p;
  p += align_up(sizeof(int) * (size_t)(n_seq + 1), 256);
  const size_t per = (size_t)mc * H;
  w.W = (float *)p;  p += align_up(sizeof(float) * per * C * dk, 256);
  w.Q = (float *)p;  p += align_up(sizeof(float) * per * C * dk, 256);
  w.Kd = (float *)p; p += align_up(sizeof(float) * per * C * dk, 256);
  w.U = (float *)p;  p += align_up(sizeof(float) * per * C * dv, 256);
  w.P = (float *)p;  p += align_up(sizeof(float) * per * C * C, 256);
  w.D = (float *)p;
  w.max_chunks = (int)mc;
  return w;
}

cudaError_t launch_chunk_table(const int32_t *cu, int n_seq, int64_t T_total, const ChunkWs &ws,
                               cudaStream_t st) {
  // one thread per sequence up to 1024 (a warp at least): few sequences, few barrier members
  const int threads = n_seq >= 1024 ? 1024 : ((n_seq + 31) / 32) * 32 + (n_seq == 0 ? 32 : 0);
  const int nb = ws.nparts > 1 ? ws.nparts - 1 : 0;
  const int4 b = make_int4(ws.bound64[1], ws.bound64[2], 0, 0);
  kda_chunk_table<<<1, threads, 0, st>>>(cu, n_seq, T_total, ws.meta, ws.seq_chunk_off, nb, b,
                                         ws.seq_chunk_b, ws.seq_order);
  return cudaGetLastError();
}

#define KDA_DISPATCH_DKDV(dk, dv, ...)                                   \
  do {                                                                    \
    if (dk == 128 && dv == 128) { constexpr int DK = 128, DV = 128; __VA_ARGS__; } \
    else if (dk == 64 && dv == 64) { constexpr int DK = 64, DV = 64; __VA_ARGS__; } \
    else if (dk == 128 && dv == 64) { constexpr int DK = 128, DV = 64; __VA_ARGS__; } \
    else { constexpr int DK = 64, DV = 128; __VA_ARGS__; }                \
  } while (0)

cudaError_t launch_prep(const void *q, const void *k, const void *v, const void *la,
                        const void *beta, const int32_t *cu, int n_seq, int64_t T_total, int H,
                        int dk, int dv, unsigned flags, kda_dtype dt, const ChunkWs &ws,
                        bool need_q, cudaStream_t st, PrepSave save) {
  if (dt == KDA_DTYPE_BF16) {
    KDA_DISPATCH_DKDV(dk, dv, return launch_prep_t<DK, DV, __nv_bfloat16>(
                                  q, k, v, la, beta, cu, n_seq, T_total, H, flags, ws, need_q, st,
                                  save));
  } else {
    KDA_DISPATCH_DKDV(dk, dv, return launch_prep_t<DK, DV, float>(
                                  q, k, v, la, beta, cu, n_seq, T_total, H, flags, ws, need_q, st,
                                  save));
  }
}

cudaError_t launch_state_pass(int mode, unsigned flags, const void *gate, void *out, const float *S0,
                              float *S_final, float *X_out, float *Z_out, const int32_t *cu,
                              int n_seq, int64_t T_total, int H, int dk, int dv, float scale,
                              kda_dtype dt, const ChunkWs &ws, cudaStream_t st, CkptOut ck,
                              StateSave save) {
  if (dt == KDA_DTYPE_BF16) {
    KDA_DISPATCH_DKDV(dk, dv, return launch_state_t<DK, DV, __nv_bfloat16>(
                                  mode, flags, gate, out, S0, S_final, X_out, Z_out, cu, n_seq,
                                  T_total, H, scale, ws, st, ck, save));
  } else {
    KDA_DISPATCH_DKDV(dk, dv, return launch_state_t<DK, DV, float>(
                                  mode, flags, gate, out, S0, S_final, X_out, Z_out, cu, n_seq,
                                  T_total, H, scale, ws, st, ck, save));
  }
}

cudaError_t chunk_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_chunk_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_chunk_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

}  // namespace kda
