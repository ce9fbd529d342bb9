/*
 * kda_selftest.h - diagnostic entry point of libkda.
 *
 * Runs one tcgen05 matrix product D = A * B (A: [M x K], B: [K x N], bf16,
 * row-major in device memory; D: [M x N] fp32) through the shared-memory tile
 * layouts the chunked kernels use: 128-byte-swizzled tiles read as K-major
 * (a_mn_major / b_mn_major = 0) or MN-major (= 1) operands. Comparing D with a
 * plain matrix product checks the descriptor encoding on the device at hand.
 * Supported: M = 128, N in 32..256 (multiple of 32), K in {64, 128}.
 * Synchronises `stream`. Returns KDA_OK, KDA_ERR_UNSUPPORTED,
 * KDA_ERR_INVALID_ARG, KDA_ERR_CUDA, or KDA_ERR_TIMEOUT if the MMA did not
 * complete within 2 s (bounded wait; the kernel then returns normally).
 * This is a check of the library itself; the K3 pages have no counterpart.
 */
#ifndef KDA_SELFTEST_H_
#define KDA_SELFTEST_H_

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

int kda_selftest_umma(const void *A, const void *B, float *D, int M, int N, int K,
                      int a_mn_major, int b_mn_major, kda_stream_t stream);

/*
 * Exercises the library's bounded device waits without a fault: one CTA of 128
 * threads waits on an mbarrier that nothing ever arrives on (no copy and no
 * tensor-core operation is issued against it) for at most `limit_us`
 * microseconds, votes on the outcome across its threads as the state pass does,
 * records KDA_ERR_TIMEOUT in the device error word and returns. Asynchronous on
 * `stream`: the next kda_get_error(stream) returns KDA_ERR_TIMEOUT (and clears
 * the word, so the call after it returns KDA_OK). limit_us in 1..1000000, else
 * KDA_ERR_INVALID_ARG; launch failures return KDA_ERR_CUDA. A check of the
 * library itself; the K3 pages have no counterpart.
 */
int kda_selftest_wait_timeout(unsigned limit_us, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_SELFTEST_H_ */
