// One-token KDA decode against fp32 states resident in device memory.
//
// Per (sequence, head), with S' = Diag(a) S (K3 training overview,
// zuoshipin.com/article/18261, section 2 "KDA"; K3 explainer,
// devpress.csdn.net, section 2: predict from memory, then write the error):
//   u  = v - S'^T k                   (prediction error)
//   S  = S' + b k u^T                 (corrective write)
//   o  = g * scale * (S'^T q + b (k.q) u)   (= g * scale * S^T q, one pass)
// Each block owns one (sequence, head) state: it reads the dk x dv fp32 state
// once into registers with 16-byte loads, reduces the two dk-long dot products
// per column across warps through shared memory, and writes the state once.
// The kernel moves 2 * dk * dv * 4 bytes of state per (sequence, head) and is
// bound by HBM bandwidth; three blocks per SM (78 registers) keep more state
// loads in flight than two.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_common.cuh"

namespace kda {

__device__ unsigned g_decode_err;

namespace {

template <int DK, int DV, typename T>
__global__ void __launch_bounds__(256, 3) kda_decode_kernel(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
    const T *__restrict__ la, const T *__restrict__ beta, const T *__restrict__ gate,
    T *__restrict__ out, float *__restrict__ state, const int32_t *__restrict__ slot,
    int n_slots, int H, float scale, unsigned flags) {
  constexpr int TPR = DV / 4;          // threads per state row (float4 each)
  constexpr int RPP = 256 / TPR;       // rows covered per pass
  constexpr int RPT = DK / RPP;        // rows per thread
  static_assert(RPT * RPP == DK, "shape");
  __shared__ float sq[DK], sk[DK], sa[DK];
  __shared__ float4 red_k[RPP][TPR], red_q[RPP][TPR];
  __shared__ float s_kq;

  const int nh = blockIdx.x, n = nh / H, h = nh % H, tid = threadIdx.x;
  int row = n;
  if (slot) {
    row = slot[n];
    if (row < 0 || row >= n_slots) {
      if (tid == 0) atomicOr(&g_decode_err, kErrBadSeqlens);
      return;
    }
  }
  float4 *S = reinterpret_cast<float4 *>(state + ((size_t)row * H + h) * DK * DV);
  const int cg = tid % TPR, rg = tid / TPR;  // column group (4 cols), row group

  // issue the state loads first: they dominate the time
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = S[(size_t)(rg + i * RPP) * TPR + cg];

  const size_t tk = ((size_t)n * H + h) * DK, tv = ((size_t)n * H + h) * DV;
  for (int c = tid; c < DK; c += 256) {
    float l = prep_log_alpha(to_f32(la[tk + c]), flags);
    if ((flags & KDA_DEBUG_CHECK) && !(l >= kLogAlphaMin && l <= 0.f))
      atomicOr(&g_decode_err, kErrPrecondition);
    sq[c] = to_f32(q[tk + c]);
    sk[c] = to_f32(k[tk + c]);
    sa[c] = expf(l);
  }
  const float b = prep_beta(to_f32(beta[(size_t)n * H + h]), flags);
  if ((flags & KDA_DEBUG_CHECK) && tid == 0 && !(b >= 0.f && b <= 1.f))
    atomicOr(&g_decode_err, kErrPrecondition);
  __syncthreads();
  if (tid < 32) {
    float ssq = 0.f, ssk = 0.f, skq = 0.f;
    for (int c = tid; c < DK; c += 32) {
      ssq += sq[c] * sq[c];
      ssk += sk[c] * sk[c];
      skq += sq[c] * sk[c];
    }
    ssq = warp_sum(ssq);
    ssk = warp_sum(ssk);
    skq = warp_sum(skq);
    float rq = 1.f, rk = 1.f;
    if (flags & KDA_QK_L2NORM) {
      rq = rsqrtf(ssq + kL2Eps);
      rk = rsqrtf(ssk + kL2Eps);
    }
    for (int c = tid; c < DK; c += 32) {
      sq[c] *= rq;
      sk[c] *= rk;
    }
    if (tid == 0) s_kq = skq * rq * rk;
  }
  __syncthreads();

  // decay, then partial S'^T k and S'^T q over this thread's rows
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * RPP;
    const float a = sa[r], kr = sk[r], qr = sq[r];
    s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
    pk.x = fmaf(kr, s[i].x, pk.x); pk.y = fmaf(kr, s[i].y, pk.y);
    pk.z = fmaf(kr, s[i].z, pk.z); pk.w = fmaf(kr, s[i].w, pk.w);
    pq.x = fmaf(qr, s[i].x, pq.x); pq.y = fmaf(qr, s[i].y, pq.y);
    pq.z = fmaf(qr, s[i].z, pq.z); pq.w = fmaf(qr, s[i].w, pq.w);
  }
  red_k[rg][cg] = pk;
  red_q[rg][cg] = pq;
  __syncthreads();
  // column totals (every thread recomputes the totals of its 4 columns)
  float4 tk4 = make_float4(0.f, 0.f, 0.f, 0.f), tq4 = tk4;
#pragma unroll 4
  for (int g = 0; g < RPP; ++g) {
    float4 a = red_k[g][cg], c = red_q[g][cg];
    tk4.x += a.x; tk4.y += a.y; tk4.z += a.z; tk4.w += a.w;
    tq4.x += c.x; tq4.y += c.y; tq4.z += c.z; tq4.w += c.w;
  }
  const int c0 = cg * 4;
  float4 u;
  u.x = to_f32(v[tv + c0 + 0]) - tk4.x;
  u.y = to_f32(v[tv + c0 + 1]) - tk4.y;
  u.z = to_f32(v[tv + c0 + 2]) - tk4.z;
  u.w = to_f32(v[tv + c0 + 3]) - tk4.w;
  if (rg == 0) {
    const float bkq = b * s_kq;
    float o0 = scale * (tq4.x + bkq * u.x), o1 = scale * (tq4.y + bkq * u.y);
    float o2 = scale * (tq4.z + bkq * u.z), o3 = scale * (tq4.w + bkq * u.w);
    if (gate) {
      o0 *= prep_gate(to_f32(gate[tv + c0 + 0]), flags);
      o1 *= prep_gate(to_f32(gate[tv + c0 + 1]), flags);
      o2 *= prep_gate(to_f32(gate[tv + c0 + 2]), flags);
      o3 *= prep_gate(to_f32(gate[tv + c0 + 3]), flags);
    }
    out[tv + c0 + 0] = from_f32<T>(o0);
    out[tv + c0 + 1] = from_f32<T>(o1);
    out[tv + c0 + 2] = from_f32<T>(o2);
    out[tv + c0 + 3] = from_f32<T>(o3);
  }
  // corrective write and store. The state is not read again within the step, so it is stored
  // with the streaming (evict-first) hint: 3 % more bandwidth on the 512 MiB decode workload
  // (last-use loads alone gained 2.7 %; both together, or streaming loads, lost)
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * RPP;
    const float bk = b * sk[r];
    float4 x = s[i];
    x.x = fmaf(bk, u.x, x.x); x.y = fmaf(bk, u.y, x.y);
    x.z = fmaf(bk, u.z, x.z); x.w = fmaf(bk, u.w, x.w);
    __stcs(&S[(size_t)r * TPR + cg], x);
  }
}

template <int DK, int DV, typename T>
cudaError_t launch_t(const void *q, const void *k, const void *v, const void *la,
                     const void *beta, const void *gate, void *out, float *state,
                     const int32_t *slot, int n_slots, int N, int H, float scale,
                     unsigned flags, cudaStream_t st) {
  kda_decode_kernel<DK, DV, T><<<N * H, 256, 0, st>>>(
      (const T *)q, (const T *)k, (const T *)v, (const T *)la, (const T *)beta,
      (const T *)gate, (T *)out, state, slot, n_slots, H, scale, flags);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const void *la,
                          const void *beta, const void *gate, void *out, float *state,
                          const int32_t *slot, int n_slots, int N, int H, int dk, int dv,
                          float scale, unsigned flags, kda_dtype dt, cudaStream_t st) {
#define KDA_DEC(DK_, DV_)                                                                    \
  if (dk == DK_ && dv == DV_) {                                                              \
    if (dt == KDA_DTYPE_BF16)                                                                \
      return launch_t<DK_, DV_, __nv_bfloat16>(q, k, v, la, beta, gate, out, state, slot,   \
                                               n_slots, N, H, scale, flags, st);            \
    return launch_t<DK_, DV_, float>(q, k, v, la, beta, gate, out, state, slot, n_slots, N, \
                                     H, scale, flags, st);                                  \
  }
  KDA_DEC(128, 128)
  KDA_DEC(64, 64)
  KDA_DEC(128, 64)
  KDA_DEC(64, 128)
#undef KDA_DEC
  return cudaErrorInvalidValue;
}

cudaError_t decode_take_error(unsigned *bits) {
  unsigned v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbol(g_decode_err, &z, sizeof(unsigned));
  *bits = v;
  return e;
}

}  // namespace kda
