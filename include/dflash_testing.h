/*
 * dflash_testing.h -- test-only entry point of libdflash.
 *
 * Runs the tensor-core GEMM of the library on its own so that it can be
 * compared with a plain matrix product, the FP8 encoder of the K/V cache on
 * given values, and the attention kernels on given inputs; the draft pass
 * never calls these entries.
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

/*
 * The QKV projection of a draft layer on its own (the tensor-core GEMM with
 * its EPI_QKV epilogue): Y = r[m] * (A W^T) with r[m] = 1 / sqrt(sum_t
 * ssq[t*M + m] / K + eps) when ssq is non-NULL (the deferred input RMSNorm:
 * A holds x * g, ssq the sums of squares of x's 128-column parts), else 1.
 * Column blocks of Y: n_heads query heads, then n_kv_heads key heads, then
 * n_kv_heads value heads, head_dim wide each.  Query and key heads get the
 * per-head RMSNorm (gain q_gain or k_gain, head_dim bf16 values, epsilon
 * eps), then rotate-half RoPE at position row_pos[m] with frequencies
 * rope_theta^(-2i/head_dim); value heads are stored as they are.
 *   A        device bf16 [M, K];  W device bf16 [N, K], N = (n_heads +
 *            2 n_kv_heads) * head_dim, a multiple of 128
 *   ssq      device float32 [K/128, M] or NULL
 *   row_pos  device int32 [M], every value in [0, max_position)
 *   q_out    device bf16 [M, n_heads * head_dim]; k_out, v_out device bf16
 *            [M, n_kv_heads * head_dim]
 *   scratch  device, at least dflash_test_qkv_scratch(M, N, max_position)
 *            bytes; its first 4 bytes are the device error word after the call
 * head_dim is 64 or 128; K a multiple of 128.  Returns DFLASH_EINVAL,
 * DFLASH_EUNSUPPORTED or DFLASH_ECAPACITY (scratch too small) on bad
 * arguments, DFLASH_ECUDA when a launch fails; nothing is launched then.
 */
size_t dflash_test_qkv_scratch(int32_t M, int32_t N, int32_t max_position);
int dflash_test_qkv(int32_t M, int32_t K, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                    int32_t max_position, float rope_theta, float eps, const void *A,
                    const void *W, const float *ssq, const void *q_gain, const void *k_gain,
                    const int32_t *row_pos, void *q_out, void *k_out, void *v_out, void *scratch,
                    size_t scratch_bytes, dflash_stream_t stream);

/* The FP8 encoder of the K/V cache epilogue on its own: codes[i] = the OCP
 * E4M3 code of x[i] / scale (IEEE float32 division, nearest code, ties to the
 * even code, saturation at +-448), the same device function the injection
 * epilogue calls.  x: device float32 [n]; codes: device uint8 [n]. */
int dflash_test_e4m3_encode(const float *x, int32_t n, float scale, uint8_t *codes,
                            dflash_stream_t stream);

/*
 * The bf16 attention step of the draft block on its own: for every request b
 * and query head h, out[b*S + j, h, :] = softmax over the visible keys of
 * q[b*S + j, h, :] . k / sqrt(128), weighted sum of the values.  The keys are
 * the request's committed context (kv_len[b] rows, paged: row r of request b
 * is row r % 64 of cache page page_table[b * pages_per_req + r / 64], or of
 * page page_table[b * pages_per_req + (r / 64) % pages_per_req] when
 * draft_window > 0) followed by the S block keys kb/vb[b*S .. b*S + S - 1].
 * A context key at position r is visible to block query j when
 * r >= kv_len[b] - draft_window (draft_window > 0) and, when window > 0,
 * kv_len[b] + j - r < window; block keys are always visible.
 *   kernel   0: the tcgen05 kernel (DFLASH_EUNSUPPORTED where it does not
 *            apply: more than 64 query rows per (request, KV head), batch
 *            above 1024); 1: the mma.sync kernels (cluster or split-KV)
 *   q, out   device bf16 [B*S, n_heads, 128]; kb, vb device bf16 [B*S, n_kv_heads, 128]
 *   k_cache, v_cache device bf16 [n_pages*64, n_kv_heads, 128]
 *   page_table, kv_len device int32 [B * pages_per_req], [B]
 *   scratch  device, at least dflash_test_attention_scratch(B, n_heads, n_kv_heads, S) bytes
 *   err      device uint32 error word (bits of dflash.h's device errors are OR-ed in)
 */
size_t dflash_test_attention_scratch(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t S);
int dflash_test_attention(int32_t kernel, int32_t B, int32_t S, int32_t n_heads, int32_t n_kv_heads,
                          int32_t pages_per_req, int32_t n_pages, int32_t window,
                          int32_t draft_window, const void *q, const void *kb, const void *vb,
                          const void *k_cache, const void *v_cache, const int32_t *page_table,
                          const int32_t *kv_len, void *out, void *scratch, size_t scratch_bytes,
                          uint32_t *err, dflash_stream_t stream);

/* Fused launches of dependent GEMMs in the draft pass on (1) or off (0, one
 * launch per GEMM) for this handle. */
int dflash_test_set_fusion(dflash_handle *h, int32_t on);

/* Attention kernel of the bf16 draft pass for this handle: 0 (default) the
 * tcgen05 kernel wherever it applies (head_dim 128, at most 64 query rows
 * per (request, KV head), more (request, KV head) pairs than half the SMs,
 * bf16 cache), else the mma.sync kernels; 1 the mma.sync kernels only. */
int dflash_test_set_attention(dflash_handle *h, int32_t kernel);

/* Tiling of the QKV GEMM (128-wide heads, more than 128 rows) for every
 * later launch of this process: 1 (default) tiles of two consecutive heads
 * by 128 tokens, whose epilogue reads whole head rows from the tensor-memory
 * accumulator; 0 tiles of 128 features by 256 tokens with the staged
 * epilogue.  Returns DFLASH_EINVAL for other values. */
int dflash_test_set_head_pairs(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_TESTING_H */
