/*
 * kda.h - C ABI of libkda: Kimi Delta Attention (KDA) on NVIDIA GB300 (sm_103a).
 *
 * KDA keeps, per sequence and head, a state S in R^{dk x dv} (rows = key
 * channels, columns = value channels) and for every token t does
 *
 *     S_t = (I - b_t k_t k_t^T) Diag(a_t) S_{t-1} + b_t k_t v_t^T
 *     o_t = g_t (.) (scale * S_t^T q_t)
 *
 * with a_t = exp(log_alpha_t) in (0, 1]^{dk} a per-key-channel retention,
 * b_t in [0, 1] the write strength and g_t the (already sigmoided) output gate.
 * Sources: K3 training overview (zuoshipin.com/article/18261) section 2 "KDA"
 * (channel-wise forget gate, delta-rule corrective write, full-rank output
 * gate, lower bound on the per-step retention); K3 explainer
 * (devpress.csdn.net/awstech/6a72dc33...) section 2 (predict from memory,
 * write the error; delta rule with a channel-wise retention factor).
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller owns every buffer. The library allocates no device
 *    memory; scratch space is passed in as `workspace` (size from the matching
 *    *_workspace_size call, 256-byte aligned).
 *  - Pointers are device pointers to contiguous row-major arrays, 16-byte
 *    aligned. Token tensors are packed [T_total, H, d]; per-token scalars
 *    [T_total, H]; states [n, H, dk, dv] fp32 with dv fastest.
 *  - Work is enqueued on `stream` and is asynchronous. A call returns
 *    KDA_OK once its kernels are launched; argument errors are returned before
 *    anything is launched. Problems found on the device (a violated
 *    precondition under KDA_DEBUG_CHECK, malformed cu_seqlens, a bounded wait
 *    that ran out) set a per-device error word that kda_get_error() reads.
 *  - Supported shapes: dk, dv in {64, 128}; chunk = 64. Other values return
 *    KDA_ERR_UNSUPPORTED. T_total = 0 and empty sequences are valid; an empty
 *    sequence leaves final = initial.
 *  - Token tensors are fp32 or bf16 (`dtype`); the output has the input
 *    dtype; states are always fp32. bf16 results are rounded to nearest even.
 *  - Precondition (the retention lower bound): log_alpha >= -0.6953125
 *    (= log 0.5 less one bf16 ulp). Within a 64-token chunk the decay factors
 *    then stay below 2^64.2, well inside the fp32/bf16 range. The library does
 *    not clamp; KDA_DEBUG_CHECK reports KDA_ERR_PRECONDITION.
 *  - No atomics touch outputs: repeated calls give bitwise-equal results.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1,  /* NULL / misaligned pointer, negative size, bad combination */
  KDA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (dk, dv, chunk, dtype) */
  KDA_ERR_CUDA = 3,         /* a CUDA call or launch failed */
  KDA_ERR_TIMEOUT = 4,      /* a bounded on-device wait ran out (kda_get_error) */
  KDA_ERR_PRECONDITION = 5, /* input outside the documented domain (kda_get_error) */
  KDA_ERR_WORKSPACE = 6     /* workspace NULL or smaller than required */
} kda_status;

typedef enum { KDA_DTYPE_F32 = 0, KDA_DTYPE_BF16 = 1 } kda_dtype;

enum {
  KDA_QK_L2NORM = 1u,   /* normalise q and k rows: x / sqrt(sum x^2 + 1e-6) */
  KDA_DEBUG_CHECK = 2u, /* check log_alpha >= -0.6953125 and beta in [0,1] on device */
  /* Gate preparation fused into the kernels (K3 training overview section 2
   * "KDA": channel-wise forget gate with a lower bound on the per-step
   * retention, output gate; section 4 "FlashKDA": the forget gate is part of
   * the per-chunk update card). With this flag, `beta` and `gate` hold logits
   * and `log_alpha` holds the forget gate's pre-activation a; the kernels use
   *     beta = sigmoid(beta),  g = sigmoid(gate),
   *     log_alpha = max(-exp(a), log(1/2))      (so alpha >= 1/2)
   * as they load them, saving one element-wise pass over those inputs.
   * kda_chunk_bwd then returns gradients with respect to the logits and a. */
  KDA_GATE_LOGITS = 4u
};

/* Library version string, e.g. "libkda 0.1 sm_103a". */
const char *kda_version(void);

/*
 * Chunked prefill over packed sequences.
 * Source: K3 training overview section 4 "FlashKDA": per-chunk update cards
 * (forget gate, Q/K normalisation, decay, intra-chunk correction matrix) are
 * prepared in parallel; only the state hand-off and output read-out run in
 * order. The result equals the token recurrence above.
 *
 *  q, k, log_alpha : [T_total, H, dk]   dtype
 *  v, gate         : [T_total, H, dv]   dtype; gate NULL means g = 1
 *  beta            : [T_total, H]       dtype, values in [0, 1]
 *  out             : [T_total, H, dv]   dtype (written)
 *  initial_state   : [n_seq, H, dk, dv] fp32, or NULL for zero
 *  final_state     : [n_seq, H, dk, dv] fp32, or NULL (not written)
 *  cu_seqlens      : device int32 [n_seq + 1], cu[0] = 0, non-decreasing,
 *                    cu[n_seq] = T_total; NULL means n_seq sequences of
 *                    T_total / n_seq tokens each (must divide)
 *  chunk           : 64
 *  workspace       : >= kda_chunk_fwd_workspace_size(...) bytes
 * Malformed cu_seqlens found on the device set KDA_ERR_INVALID_ARG in the
 * error word and the call writes nothing.
 *
 * Scheduling (bf16, dk = dv = 128, at most 112 (sequence, head) pairs and
 * >= 16 chunks per sequence on average): the call splits every sequence after
 * floor(n_chunks * 47 / 64) chunks. The state pass of the
 * leading parts then runs on `stream` beside the card launch of the trailing
 * parts on a library-owned stream; events fork that stream off `stream` and
 * join it back before the call returns, so all work stays ordered on
 * `stream` (and the call can be captured in a CUDA graph). The library
 * stream is one per device for the process's lifetime; concurrent calls
 * from several host threads share it, so their trailing card launches run
 * one after another. Results are bitwise those of the unsplit schedule.
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *beta,
                         const void *gate, void *out,
                         const float *initial_state, float *final_state,
                         const int32_t *cu_seqlens, int n_seq, int64_t T_total,
                         int H, int dk, int dv, int chunk, float scale,
                         unsigned flags, kda_dtype dtype, void *workspace,
                         size_t workspace_bytes, kda_stream_t stream);

size_t kda_chunk_fwd_workspace_size(int64_t T_total, int n_seq, int H, int dk,
                                    int dv, int chunk, kda_dtype dtype);

/*
 * Kernel launches kda_chunk_fwd (and kda_chunk_fwd_checkpoints) make for this
 * problem; varlen != 0 when the call passes cu_seqlens. In order: the chunk
 * table (skipped on the tensor-core path, bf16 with dk = dv = 128, when
 * cu_seqlens is NULL: its kernels then index the fixed-length sequences
 * directly), then either chunk prep and state pass, or for a split prefill
 * the prep of the leading parts, the state pass of the leading parts, the
 * prep of the trailing parts and the state pass of the trailing parts.
 * So 2 to 5; 0 for an empty or invalid problem. Host only.
 */
int kda_chunk_fwd_launches(int64_t T_total, int n_seq, int H, int dk, int dv,
                           int chunk, kda_dtype dtype, int varlen);

/*
 * kda_chunk_fwd that also saves the state at fixed token boundaries, for a
 * prefix cache that resumes a sequence from its longest cached prefix.
 * Source: K3 explainer section 14 "Prefix Cache": a reused prefix must restore
 * the fixed-size KDA state at the same boundary as the attention KV pages, so
 * state checkpoints are kept at reusable boundaries.
 *
 * Arguments and results of kda_chunk_fwd (same workspace size), plus
 *  checkpoints         : [n_seq, checkpoints_per_seq, H, dk, dv] fp32. Slot
 *                        (s, i) receives the state of sequence s after its
 *                        first (i + 1) * checkpoint_every tokens (the state
 *                        the sequence's token (i + 1) * checkpoint_every
 *                        starts from), for every i < checkpoints_per_seq with
 *                        (i + 1) * checkpoint_every <= len_s. Other slots are
 *                        not written. A boundary at the end of a sequence
 *                        equals its final state.
 *  checkpoint_every    : > 0, a multiple of chunk (64)
 *  checkpoints_per_seq : >= 0; 0 writes no checkpoint (then checkpoints may
 *                        be NULL)
 * Checkpoints are the kernel's fp32 running state, bitwise equal to the
 * final_state a kda_chunk_fwd call over the prefix returns.
 */
kda_status kda_chunk_fwd_checkpoints(
    const void *q, const void *k, const void *v, const void *log_alpha,
    const void *beta, const void *gate, void *out, const float *initial_state,
    float *final_state, float *checkpoints, int64_t checkpoint_every,
    int checkpoints_per_seq, const int32_t *cu_seqlens, int n_seq,
    int64_t T_total, int H, int dk, int dv, int chunk, float scale,
    unsigned flags, kda_dtype dtype, void *workspace, size_t workspace_bytes,
    kda_stream_t stream);

/*
 * Chunked backward pass: gradients of
 *     L = sum_t <d_out_t, o_t> + sum_s <d_final_state_s, final_state_s>
 * for the forward that kda_chunk_fwd computes with the same arguments.
 * Source: K3 training overview section 4 "FlashKDA" presents the chunked
 * kernel as a training kernel; this is its reverse mode. The forward chunk
 * quantities are recomputed (nothing is kept from a forward call). All steps
 * run in fp32; the kernels are CUDA-core (SIMT) code.
 *
 *  q, k, v, log_alpha, beta, gate, initial_state, cu_seqlens, n_seq, T_total,
 *  H, dk, dv, chunk, scale, flags, dtype : as for kda_chunk_fwd
 *  d_out            : [T_total, H, dv] dtype, cotangent of out
 *  d_final_state    : [n_seq, H, dk, dv] fp32 cotangent of final_state, or NULL (0)
 *  d_q, d_k, d_log_alpha : [T_total, H, dk] dtype (written); gradients with
 *                     respect to the raw q and k (through the L2 normalisation
 *                     when KDA_QK_L2NORM is set) and to log_alpha
 *  d_v              : [T_total, H, dv] dtype (written)
 *  d_beta           : [T_total, H] dtype (written)
 *  d_gate           : [T_total, H, dv] dtype, or NULL (not written); must be
 *                     NULL when gate is NULL
 *  d_initial_state  : [n_seq, H, dk, dv] fp32, or NULL (not written)
 *  workspace        : >= kda_chunk_bwd_workspace_size(...) bytes
 * Gradients in bf16 are rounded to nearest even from fp32.
 */
kda_status kda_chunk_bwd(const void *q, const void *k, const void *v,
                         const void *log_alpha, const void *beta,
                         const void *gate, const float *initial_state,
                         const void *d_out, const float *d_final_state,
                         void *d_q, void *d_k, void *d_v, void *d_log_alpha,
                         void *d_beta, void *d_gate, float *d_initial_state,
                         const int32_t *cu_seqlens, int n_seq, int64_t T_total,
                         int H, int dk, int dv, int chunk, float scale,
                         unsigned flags, kda_dtype dtype, void *workspace,
                         size_t workspace_bytes, kda_stream_t stream);

size_t kda_chunk_bwd_workspace_size(int64_t T_total, int n_seq, int H, int dk,
                                    int dv, int chunk, kda_dtype dtype);

/*
 * One sequence split into n_seg segments, evaluated the context-parallel way
 * on one GPU: per-segment summaries (as kda_segment_summary), their ordered
 * scan (as kda_scan_combine, from initial_state), then every segment re-run
 * from its recovered entry state (as kda_chunk_fwd). The update cards are
 * computed once and serve both the summaries and the re-run.
 * Source: K3 training overview section 3 "KDA context parallel" (fixed-size
 * per-segment summaries merged by a prefix scan recover each segment's exact
 * entry state) and section 4 "FlashKDA" (update cards).
 *
 *  q, k, v, log_alpha, beta, gate, out : as kda_chunk_fwd over the T_total tokens
 *  initial_state        : [H, dk, dv] fp32 state before segment 0, or NULL (0)
 *  final_state          : [H, dk, dv] fp32 state after the last segment, or NULL
 *  segment_entry_states : [n_seg, H, dk, dv] fp32 (written: state entering
 *                         each segment), or NULL (kept in the workspace)
 *  cu_segs              : device int32 [n_seg + 1] segment bounds, cu_segs[0] = 0,
 *                         cu_segs[n_seg] = T_total; NULL = n_seg equal segments
 *  workspace            : >= kda_segmented_fwd_workspace_size(...) bytes
 * The output equals kda_chunk_fwd over the whole sequence up to rounding.
 */
kda_status kda_segmented_fwd(const void *q, const void *k, const void *v,
                             const void *log_alpha, const void *beta,
                             const void *gate, void *out,
                             const float *initial_state, float *final_state,
                             float *segment_entry_states,
                             const int32_t *cu_segs, int n_seg, int64_t T_total,
                             int H, int dk, int dv, int chunk, float scale,
                             unsigned flags, kda_dtype dtype, void *workspace,
                             size_t workspace_bytes, kda_stream_t stream);

size_t kda_segmented_fwd_workspace_size(int64_t T_total, int n_seg, int H,
                                        int dk, int dv, int chunk,
                                        kda_dtype dtype);

/*
 * kda_chunk_fwd without a workspace argument, for callers that cannot
 * allocate device memory where they run the mixer: host frameworks that
 * reserve the device heap up front and give a kernel only its inputs and
 * outputs, plugin interfaces with no workspace slot, and code that must not
 * call cudaMalloc/cudaFree because they can synchronise the device. The K3
 * pages have no counterpart to this entry point.
 *
 * Same arguments, results and status codes as kda_chunk_fwd, minus
 * workspace/workspace_bytes. Scratch comes from a fixed 64 MiB array in the
 * library's device memory (held on every device that loads the library until
 * it is unloaded); problems whose kda_chunk_fwd_workspace_size exceeds 64 MiB
 * are rejected with KDA_ERR_WORKSPACE before any launch. The call allocates
 * nothing. All calls on a device share that array: calls whose kernels may
 * overlap on the GPU (unordered streams) race and give wrong results. The
 * first call on a device looks up the array's address (cudaGetSymbolAddress);
 * make that first call before any stream capture.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const void *log_alpha, const void *beta,
                                 const void *gate, void *out,
                                 const float *initial_state, float *final_state,
                                 const int32_t *cu_seqlens, int n_seq,
                                 int64_t T_total, int H, int dk, int dv,
                                 int chunk, float scale, unsigned flags,
                                 kda_dtype dtype, kda_stream_t stream);

/*
 * kda_chunk_fwd on host-resident buffers: each sequence's inputs are copied
 * to the device, computed and its outputs copied back, the copies of one
 * sequence overlapped with the compute of its neighbours (three streams: the
 * caller's for the compute, two library-owned ones per device for the
 * copies). It serves callers whose activations live in host memory. The K3
 * pages have no counterpart to this entry point.
 *
 * Arguments and results of kda_chunk_fwd for fixed-length sequences (no
 * cu_seqlens: n_seq sequences of T_total / n_seq tokens), except:
 *  q, k, v, log_alpha, beta, gate, out, initial_state, final_state :
 *      page-locked host memory (cudaHostAlloc, cudaHostRegister), the same
 *      layouts. Other memory returns KDA_ERR_INVALID_ARG.
 *  tail_slices   : 1 to 16. The last sequence is computed in this many time
 *                  slices of equal length, each starting from the state the
 *                  slice before left, so that less compute and copy-out is left
 *                  after its last copy in. Its length must be a multiple of
 *                  64 * tail_slices.
 *  device_buffer : device memory of at least kda_chunk_fwd_host_buffer_size()
 *                  bytes, 256-byte aligned: the inputs' and outputs' device
 *                  copies and the compute's workspace.
 * Work is ordered after `stream`, and `stream` waits for the last copy back:
 * the host outputs are complete once the work queued on `stream` so far has
 * finished. Results are bitwise those of kda_chunk_fwd on the same values in
 * device memory.
 * Status: KDA_ERR_UNSUPPORTED for dk, dv, chunk or dtype; KDA_ERR_INVALID_ARG
 * for unequal lengths, a bad tail_slices, a missing or pageable buffer or a
 * misaligned device_buffer; KDA_ERR_WORKSPACE when device_buffer is NULL or
 * too small (all before any copy or launch); KDA_ERR_CUDA when a copy, event or
 * launch fails, after the copy streams are joined back into `stream`; and
 * kda_chunk_fwd's own codes for the compute.
 */
kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                              const void *log_alpha, const void *beta,
                              const void *gate, void *out,
                              const float *initial_state, float *final_state,
                              int n_seq, int64_t T_total, int H, int dk, int dv,
                              int chunk, float scale, unsigned flags,
                              kda_dtype dtype, int tail_slices,
                              void *device_buffer, size_t device_bytes,
                              kda_stream_t stream);

/* Bytes of device_buffer kda_chunk_fwd_host needs; 0 for an invalid problem. */
size_t kda_chunk_fwd_host_buffer_size(int64_t T_total, int n_seq, int H, int dk,
                                      int dv, int chunk, kda_dtype dtype,
                                      int tail_slices);

/*
 * One decode step for N sequences, one new token each, against fp32 states
 * resident in device memory (the recurrence above, applied once).
 * Source: K3 explainer section 2 (one corrective write per token) and the
 * prefix-cache section 14 (a fixed-size KDA state per sequence).
 *
 *  q, k, log_alpha : [N, H, dk] dtype;  v, gate : [N, H, dv] dtype (gate NULL = 1)
 *  beta            : [N, H] dtype
 *  out             : [N, H, dv] dtype (written)
 *  state           : [n_slots, H, dk, dv] fp32, updated in place
 *  state_slot      : device int32 [N] giving the state row of sequence n, or
 *                    NULL for row n. Slots must be distinct and < n_slots
 *                    (out-of-range slots set KDA_ERR_INVALID_ARG on device
 *                    and that sequence is skipped).
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const void *log_alpha, const void *beta,
                           const void *gate, void *out, float *state,
                           const int32_t *state_slot, int n_slots, int N, int H,
                           int dk, int dv, float scale, unsigned flags,
                           kda_dtype dtype, kda_stream_t stream);

/*
 * Context-parallel segment summaries. For each segment s (token range
 * [cu_segs[s], cu_segs[s+1])) and head: the transition X (dk x dk) and the
 * zero-init state Z (dk x dv) such that running the segment from any entry
 * state E gives X E + Z.
 * Source: K3 training overview section 3 "KDA context parallel": each device
 * emits two fixed-size pieces, how its segment rewrites existing memory and
 * the state it builds from empty memory.
 *
 *  k, log_alpha : [T_total, H, dk] dtype;  v : [T_total, H, dv];  beta : [T_total, H]
 *  cu_segs      : device int32 [n_seg + 1] (same rules as cu_seqlens)
 *  X_out        : [n_seg, H, dk, dk] fp32;  Z_out : [n_seg, H, dk, dv] fp32
 *  workspace    : >= kda_segment_summary_workspace_size(...) bytes
 */
kda_status kda_segment_summary(const void *k, const void *v,
                               const void *log_alpha, const void *beta,
                               const int32_t *cu_segs, int n_seg,
                               int64_t T_total, int H, int dk, int dv,
                               int chunk, unsigned flags, kda_dtype dtype,
                               float *X_out, float *Z_out, void *workspace,
                               size_t workspace_bytes, kda_stream_t stream);

size_t kda_segment_summary_workspace_size(int64_t T_total, int n_seg, int H,
                                          int dk, int dv, int chunk,
                                          kda_dtype dtype);

/*
 * Ordered prefix scan of the segment maps, per head:
 *   E_0 = S_init (or 0),  E_s = X_{s-1} E_{s-1} + Z_{s-1},
 *   S_final = X_{n-1} E_{n-1} + Z_{n-1}.
 * Source: K3 training overview section 3: the summaries are merged in order
 * by a prefix scan that recovers the exact state before every segment.
 *
 *  X : [n_seg, H, dk, dk] fp32;  Z : [n_seg, H, dk, dv] fp32
 *  S_init      : [H, dk, dv] fp32 or NULL (zero)
 *  S_entry_out : [n_seg, H, dk, dv] fp32 (E_s), or NULL
 *  S_final_out : [H, dk, dv] fp32, or NULL
 * All arithmetic is fp32.
 */
kda_status kda_scan_combine(const float *X, const float *Z, int n_seg, int H,
                            int dk, int dv, const float *S_init,
                            float *S_entry_out, float *S_final_out,
                            kda_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the device error word of the
 * current device. Returns KDA_OK, KDA_ERR_PRECONDITION, KDA_ERR_INVALID_ARG
 * (malformed cu_seqlens / slots), KDA_ERR_TIMEOUT or KDA_ERR_CUDA.
 */
kda_status kda_get_error(kda_stream_t stream);

/*
 * Tracing. After kda_trace_events(begin, end, n) with n > 0, every entry point
 * called from this host thread records begin[i] and end[i] (cudaEvent_t
 * handles, created and owned by the caller) on its stream around its i-th
 * kernel launch, i < n; launches past n are not traced. kda_segment_summary
 * launches, in order: 0 chunk table, 1 chunk prep, 2 state pass;
 * kda_chunk_fwd the launches that kda_chunk_fwd_launches lists, in its
 * order (the trailing cards' events of a split call on the library's card
 * stream). n = 0 turns tracing off. Records nothing else and allocates
 * nothing; the caller reads the elapsed times with cudaEventElapsedTime.
 */
kda_status kda_trace_events(void *const *begin, void *const *end, int n);

/* Human-readable message for the last non-OK status on this host thread. */
const char *kda_last_error_string(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
