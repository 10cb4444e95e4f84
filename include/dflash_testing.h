/*
 * dflash_testing.h -- test-only entry point of libdflash.
 *
 * Runs the tensor-core GEMM of the library on its own so that it can be
 * compared with a plain matrix product, and the FP8 encoder of the K/V cache
 * on given values; the draft pass never calls these entries.
 */
#ifndef DFLASH_TESTING_H
#define DFLASH_TESTING_H

#include "dflash.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Y[m, n] = sum_k A[m, k] * W[n, k] with bf16 inputs and fp32 accumulation.
 *   A       HOST array [n_src] of device pointers, each [M, K / n_src] bf16
 *           with row stride lda elements (the K-split operand of the fc step)
 *   W       device [N, K] bf16, row stride ldw
 *   op      0: out = Y as fp32 [M, N];
 *           2: act_out = silu(Y[:, :N/2]) * Y[:, N/2:] as bf16 [M, N/2];
 *           3: argmax keys of each row into ((uint64_t*)out)[M] (caller zeroes them)
 *   scratch device workspace of at least dflash_test_gemm_scratch(M, N) bytes
 * Returns a dflash_status.
 */
size_t dflash_test_gemm_scratch(int32_t M, int32_t N);
int dflash_test_gemm(int32_t M, int32_t N, int32_t K, int32_t n_src, const void *const *A,
                     int32_t lda, const void *W, int32_t ldw, int32_t op, void *out,
                     void *act_out, void *scratch, size_t scratch_bytes, dflash_stream_t stream);

/* As dflash_test_gemm; when trace is non-NULL each CTA of the (persistent)
 * GEMM writes %globaltimer stamps (ns) to trace[cta * dflash_test_trace_slots()
 * + slot]: 0 entry, 1 set-up done, 2 weight ring issued, 3 predecessor wait
 * returned, 4 first stage consumed by the MMA warp, 5 last MMA complete, 6
 * first accumulator received by the epilogue, 7 epilogue done; then per GEMM
 * phase i (a program has up to 4): 8+4i inputs ready at the producer, 9+4i
 * first segment's MMAs issued, 10+4i last MMA of the phase issued, 11+4i
 * epilogue done with the phase.  Slots a CTA never reaches stay untouched.
 * Caller provides dflash_test_trace_slots() * 160 entries (the grid never
 * exceeds 160 CTAs). */
int32_t dflash_test_trace_slots(void);
int dflash_test_gemm_traced(int32_t M, int32_t N, int32_t K, int32_t n_src, const void *const *A,
                            int32_t lda, const void *W, int32_t ldw, int32_t op, void *out,
                            void *act_out, void *scratch, size_t scratch_bytes,
                            unsigned long long *trace, dflash_stream_t stream);

/*
 * A chain of up to 4 dependent GEMMs run as one fused tensor-core launch (the
 * form the draft pass uses for a layer's O-proj / gate-up / down / next-QKV).
 * Phase i computes Y_i = A_i W_i^T with A_i device bf16 [M, K[i]] (row stride
 * K[i]) and W_i device bf16 [N[i], K[i]]; op[i] 0 stores Y_i as fp32 [M, N[i]]
 * into out[i], 1 as bf16 [M, N[i]], 2 stores silu(Y[:, :N/2]) * Y[:, N/2:] as
 * bf16 [M, N[i]/2].  A later phase may read an earlier phase's bf16 output
 * (A[i] == out[j], j < i).  N, K, A, W, op, out are HOST arrays of n_phases
 * entries; scratch: device, at least dflash_test_program_scratch() bytes.
 */
size_t dflash_test_program_scratch(int32_t n_phases, int32_t M, const int32_t *N,
                                   const int32_t *op);
int dflash_test_gemm_program(int32_t n_phases, int32_t M, const int32_t *N, const int32_t *K,
                             const void *const *A, const void *const *W, const int32_t *op,
                             void *const *out, void *scratch, size_t scratch_bytes,
                             dflash_stream_t stream);

/* As dflash_test_gemm_program, with the timestamps of dflash_test_gemm_traced. */
int dflash_test_gemm_program_traced(int32_t n_phases, int32_t M, const int32_t *N, const int32_t *K,
                                    const void *const *A, const void *const *W, const int32_t *op,
                                    void *const *out, void *scratch, size_t scratch_bytes,
                                    unsigned long long *trace, dflash_stream_t stream);

/* The FP8 encoder of the K/V cache epilogue on its own: codes[i] = the OCP
 * E4M3 code of x[i] / scale (IEEE float32 division, nearest code, ties to the
 * even code, saturation at +-448), the same device function the injection
 * epilogue calls.  x: device float32 [n]; codes: device uint8 [n]. */
int dflash_test_e4m3_encode(const float *x, int32_t n, float scale, uint8_t *codes,
                            dflash_stream_t stream);

/* Fused launches of dependent GEMMs in the draft pass on (1) or off (0, one
 * launch per GEMM) for this handle. */
int dflash_test_set_fusion(dflash_handle *h, int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_TESTING_H */
