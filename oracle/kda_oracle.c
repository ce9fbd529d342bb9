/*
 * KDA oracle: plain, slow, token-by-token fp64 recurrence on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library path may link, load or call
 * this file. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (per sequence, per head, state S in R^{dk x dv}, rows = key
 * channels, columns = value channels):
 *
 *   q <- q / sqrt(sum q^2 + 1e-6),  k <- k / sqrt(sum k^2 + 1e-6)   (if l2norm)
 *   alpha = exp(log_alpha)                          (one factor per key channel)
 *   S'    = Diag(alpha) S                           (decay key-channel rows)
 *   S     = S' + beta * k (v^T - k^T S')            (delta-rule corrective write)
 *   o     = gate (.) (scale * S^T q)                (read the updated state)
 *
 * Sources:
 *  - K3 training overview (zuoshipin.com/article/18261), section 2 "KDA": a
 *    channel-wise forget gate, a delta-rule error-correcting write, a full-rank
 *    output gate, and a lower bound on the per-step retention.
 *  - K3 explainer (devpress.csdn.net/awstech/6a72dc33...), section 2 "KDA is
 *    not storing history but editing memory": the write first predicts from
 *    the current memory and then stores the prediction error; the update is a
 *    delta rule with a channel-wise retention factor.
 *  - The recurrence S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T with
 *    o_t = S_t^T q_t times a sigmoid output gate is the plain reading of those
 *    passages; S' + b k (v^T - k^T S') is the same expression multiplied out.
 *  - Context-parallel summaries: K3 training overview, section 3 "KDA context
 *    parallel": each segment emits (a) how it transforms the memory it is
 *    handed and (b) the state it produces from empty memory; an ordered prefix
 *    scan recovers the exact state entering every segment. Here (a) is the
 *    dk x dk matrix X with S_out = X S_in + Z and (b) is Z.
 *
 * Inputs are float arrays: bf16 and fp32 values convert to double exactly, so
 * the oracle sees the very numbers the device sees. All arithmetic is double.
 * Chains (sequence, head) are independent and run in parallel under OpenMP.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_REF_EPS 1e-6

/* One token of the recurrence on a state with `ncol` columns.
 * S: dk x ncol row-major; k, q: length dk (already normalised if asked);
 * alpha: length dk; vrow: length ncol; o (may be NULL): length ncol. */
static void ref_token(double *S, int dk, int ncol, const double *q,
                      const double *k, const double *alpha, const double *vrow,
                      double beta, const double *gate, double scale, double *o,
                      double *scratch /* length ncol */) {
  /* S' = Diag(alpha) S */
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < ncol; ++j) S[(size_t)i * ncol + j] *= alpha[i];
  /* prediction k^T S' and the error v - prediction */
  for (int j = 0; j < ncol; ++j) {
    double p = 0.0;
    for (int i = 0; i < dk; ++i) p += k[i] * S[(size_t)i * ncol + j];
    scratch[j] = vrow[j] - p;
  }
  /* corrective write */
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < ncol; ++j)
      S[(size_t)i * ncol + j] += beta * k[i] * scratch[j];
  /* read-out from the updated state */
  if (o) {
    for (int j = 0; j < ncol; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += q[i] * S[(size_t)i * ncol + j];
      o[j] = scale * acc * (gate ? gate[j] : 1.0);
    }
  }
}

static void load_vec(double *dst, const float *src, int n) {
  for (int i = 0; i < n; ++i) dst[i] = (double)src[i];
}

static void l2_normalise(double *x, int n) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss + KDA_REF_EPS);
  for (int i = 0; i < n; ++i) x[i] *= r;
}

static void set_threads(int n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
}

int kda_ref_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Prefill / full recurrence over packed sequences.
 *  q,k,log_alpha: [T_total, H, dk]; v, gate: [T_total, H, dv]; beta: [T_total, H]
 *  S0: [n_seq, H, dk, dv] or NULL (zero); cu_seqlens: [n_seq + 1]
 *  out: [T_total, H, dv] or NULL; S_final: [n_seq, H, dk, dv] or NULL
 *  t_stop: per sequence, the number of leading tokens to process (NULL = all);
 *  lets a caller run the recurrence over a prefix only.
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int kda_ref_forward(const float *q, const float *k, const float *v,
                    const float *log_alpha, const float *beta,
                    const float *gate, const double *S0,
                    const int64_t *cu_seqlens, int n_seq, int H, int dk,
                    int dv, double scale, int l2norm, double *out,
                    double *S_final, const int64_t *t_stop, int n_threads) {
  if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0 || dk > 512 || dv > 512 ||
      !cu_seqlens)
    return -1;
  set_threads(n_threads);
  int n_chain = n_seq * H;
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int c = 0; c < n_chain; ++c) {
    int s = c / H, h = c % H;
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * dv);
    double *buf = (double *)malloc(sizeof(double) * (size_t)(3 * dk + 2 * dv));
    if (!S || !buf) {
      free(S);
      free(buf);
      fail |= 1;
      continue;
    }
    double *qq = buf, *kk = qq + dk, *al = kk + dk, *scratch = al + dk,
           *ov = scratch + dv;
    if (S0)
      memcpy(S, S0 + ((size_t)s * H + h) * dk * dv, sizeof(double) * dk * dv);
    else
      memset(S, 0, sizeof(double) * (size_t)dk * dv);
    int64_t t0 = cu_seqlens[s], t1 = cu_seqlens[s + 1];
    if (t_stop && t0 + t_stop[s] < t1) t1 = t0 + t_stop[s];
    double vv[512], gg[512];
    for (int64_t t = t0; t < t1; ++t) {
      size_t rk = ((size_t)t * H + h) * dk, rv = ((size_t)t * H + h) * dv;
      load_vec(qq, q + rk, dk);
      load_vec(kk, k + rk, dk);
      if (l2norm) {
        l2_normalise(qq, dk);
        l2_normalise(kk, dk);
      }
      for (int i = 0; i < dk; ++i) al[i] = exp((double)log_alpha[rk + i]);
      load_vec(vv, v + rv, dv);
      if (gate) load_vec(gg, gate + rv, dv);
      ref_token(S, dk, dv, qq, kk, al, vv, (double)beta[(size_t)t * H + h],
                gate ? gg : NULL, scale, ov, scratch);
      if (out) memcpy(out + rv, ov, sizeof(double) * dv);
    }
    if (S_final)
      memcpy(S_final + ((size_t)s * H + h) * dk * dv, S,
             sizeof(double) * (size_t)dk * dv);
    free(S);
    free(buf);
  }
  return fail ? -1 : 0;
}

/*
 * One decode step for N independent sequences: the same token update as
 * kda_ref_forward, applied to state rows picked by `slot` (NULL = identity).
 *  q,k,log_alpha: [N, H, dk]; v, gate: [N, H, dv]; beta: [N, H]
 *  state: [n_slots, H, dk, dv], updated in place; out: [N, H, dv]
 */
int kda_ref_decode_step(const float *q, const float *k, const float *v,
                        const float *log_alpha, const float *beta,
                        const float *gate, double *state, const int64_t *slot,
                        int N, int H, int dk, int dv, double scale, int l2norm,
                        double *out, int n_threads) {
  if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || dk > 512 || dv > 512) return -1;
  set_threads(n_threads);
#pragma omp parallel for schedule(static)
  for (int c = 0; c < N * H; ++c) {
    int n = c / H, h = c % H;
    double qq[512], kk[512], al[512], vv[512], gg[512], scratch[512], ov[512];
    size_t rk = ((size_t)n * H + h) * dk, rv = ((size_t)n * H + h) * dv;
    load_vec(qq, q + rk, dk);
    load_vec(kk, k + rk, dk);
    if (l2norm) {
      l2_normalise(qq, dk);
      l2_normalise(kk, dk);
    }
    for (int i = 0; i < dk; ++i) al[i] = exp((double)log_alpha[rk + i]);
    load_vec(vv, v + rv, dv);
    if (gate) load_vec(gg, gate + rv, dv);
    int64_t row = slot ? slot[n] : n;
    double *S = state + ((size_t)row * H + h) * dk * dv;
    ref_token(S, dk, dv, qq, kk, al, vv, (double)beta[(size_t)n * H + h],
              gate ? gg : NULL, scale, ov, scratch);
    memcpy(out + rv, ov, sizeof(double) * dv);
  }
  return 0;
}

/*
 * Per-segment summaries. For every segment s and head h, run the recurrence
 * on the augmented state Y = [X | Z] (dk x (dk + dv)) from Y0 = [I | 0] with
 * augmented values [0 | v]. Afterwards X is the segment's transition and Z
 * the state it produces from zero memory, so S_out = X S_in + Z.
 *  cu_segs: [n_seg + 1] token offsets; X_out: [n_seg, H, dk, dk];
 *  Z_out: [n_seg, H, dk, dv]
 */
int kda_ref_segment_summary(const float *k, const float *v,
                            const float *log_alpha, const float *beta,
                            const int64_t *cu_segs, int n_seg, int H, int dk,
                            int dv, int l2norm, double *X_out, double *Z_out,
                            int n_threads) {
  if (n_seg < 0 || H <= 0 || dk <= 0 || dv <= 0 || dk > 512 || dv > 512)
    return -1;
  set_threads(n_threads);
  int ncol = dk + dv;
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int c = 0; c < n_seg * H; ++c) {
    int s = c / H, h = c % H;
    double *Y = (double *)calloc((size_t)dk * ncol, sizeof(double));
    if (!Y) {
      fail |= 1;
      continue;
    }
    for (int i = 0; i < dk; ++i) Y[(size_t)i * ncol + i] = 1.0;
    double kk[512], al[512], vaug[1024], scratch[1024];
    for (int64_t t = cu_segs[s]; t < cu_segs[s + 1]; ++t) {
      size_t rk = ((size_t)t * H + h) * dk, rv = ((size_t)t * H + h) * dv;
      load_vec(kk, k + rk, dk);
      if (l2norm) l2_normalise(kk, dk);
      for (int i = 0; i < dk; ++i) al[i] = exp((double)log_alpha[rk + i]);
      for (int j = 0; j < dk; ++j) vaug[j] = 0.0;
      load_vec(vaug + dk, v + rv, dv);
      ref_token(Y, dk, ncol, NULL, kk, al, vaug,
                (double)beta[(size_t)t * H + h], NULL, 1.0, NULL, scratch);
    }
    for (int i = 0; i < dk; ++i) {
      memcpy(X_out + (((size_t)s * H + h) * dk + i) * dk, Y + (size_t)i * ncol,
             sizeof(double) * dk);
      memcpy(Z_out + (((size_t)s * H + h) * dk + i) * dv,
             Y + (size_t)i * ncol + dk, sizeof(double) * dv);
    }
    free(Y);
  }
  return fail ? -1 : 0;
}

/*
 * Ordered (exclusive) prefix scan of the affine segment maps:
 *   E_0 = S_init (or 0),  E_s = X_{s-1} E_{s-1} + Z_{s-1},
 *   S_final = X_{n-1} E_{n-1} + Z_{n-1}.
 *  X: [n_seg, H, dk, dk]; Z, E_out: [n_seg, H, dk, dv]; S_init, S_final: [H, dk, dv]
 */
int kda_ref_scan_combine(const double *X, const double *Z, int n_seg, int H,
                         int dk, int dv, const double *S_init, double *E_out,
                         double *S_final) {
  if (n_seg < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  size_t st = (size_t)dk * dv;
  double *E = (double *)malloc(sizeof(double) * st);
  double *N = (double *)malloc(sizeof(double) * st);
  if (!E || !N) {
    free(E);
    free(N);
    return -1;
  }
  for (int h = 0; h < H; ++h) {
    if (S_init)
      memcpy(E, S_init + (size_t)h * st, sizeof(double) * st);
    else
      memset(E, 0, sizeof(double) * st);
    for (int s = 0; s < n_seg; ++s) {
      if (E_out)
        memcpy(E_out + ((size_t)s * H + h) * st, E, sizeof(double) * st);
      const double *Xs = X + ((size_t)s * H + h) * dk * dk;
      const double *Zs = Z + ((size_t)s * H + h) * st;
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) {
          double acc = Zs[(size_t)i * dv + j];
          for (int l = 0; l < dk; ++l)
            acc += Xs[(size_t)i * dk + l] * E[(size_t)l * dv + j];
          N[(size_t)i * dv + j] = acc;
        }
      memcpy(E, N, sizeof(double) * st);
    }
    if (S_final) memcpy(S_final + (size_t)h * st, E, sizeof(double) * st);
  }
  free(E);
  free(N);
  return 0;
}
