/*
 * dflash.h -- C ABI of the GB300 (sm_103a) DFlash draft-pass library.
 *
 * The DFlash draft pass (block-diffusion speculative decoding) has three
 * steps, each one entry point below:
 *
 *   dflash_inject_context  target features -> fc -> hidden_norm -> every draft
 *                          layer's K/V (k-norm, RoPE) -> paged draft KV cache.
 *   dflash_draft_block     one non-causal forward of [anchor, MASK x (S-1)]
 *                          and a greedy lm_head argmax for block rows 1..S-1.
 *   dflash_accept_commit   greedy prefix acceptance, commit of the accepted
 *                          drafts plus the bonus token, and the crop index.
 *
 * Sources: "Inside SGLang: DFlash and DFlash 2 Implementation" (Steps 1-7),
 * the CSDN DFlash article (sections "target model prefill", "draft model
 * predict", "target model verify", "fused_kv_materialize") and SGLang PR
 * #23000 "Spec V2 DFlash Support".
 *
 * Conventions shared by every entry point
 *  - Every pointer named "device" is CUDA device memory owned by the caller;
 *    "host" pointers are read during the call only.  The library allocates no
 *    device memory: it uses only the workspace bound with
 *    dflash_bind_workspace.  Weights must outlive the handle.
 *  - Calls are asynchronous and stream-ordered on the given stream; none of
 *    them synchronizes with the host except dflash_get_error.
 *  - Host-checkable errors (null pointers, sizes beyond the configured
 *    maxima, unsupported shapes) return a negative dflash_status at once and
 *    launch nothing; dflash_last_error() then describes the failure.
 *  - Data-dependent errors found on the device (a context past the page
 *    table's capacity, a page id outside the pool, a token id outside the
 *    vocabulary, a position past max_position, an output row overflow) set
 *    a bit of a sticky device error word; the offending row is skipped
 *    (nothing is written for it).  dflash_get_error reads and clears it.
 *  - Matrices are row-major.  Weight matrices use the [out, in] layout of a
 *    linear layer (y = x W^T), i.e. the reduction dimension is contiguous.
 *  - Storage type of weights, features, K/V pages and the optional hidden
 *    output is the configured dtype (fp32 or bf16); ids are int32.  With
 *    kv_fp8 set, the K/V pages hold one-byte FP8 E4M3 codes instead.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *dflash_stream_t;

typedef enum {
  DFLASH_OK = 0,
  DFLASH_EINVAL = -1,        /* null pointer, negative or inconsistent size */
  DFLASH_EUNSUPPORTED = -2,  /* shape outside what the kernels implement */
  DFLASH_ECAPACITY = -3,     /* batch/rows beyond the configured maxima, workspace too small */
  DFLASH_ECUDA = -4,         /* a CUDA runtime/driver call failed */
  DFLASH_EDEVICE = -5,       /* dflash_get_error: the device error word was non-zero */
  DFLASH_ESTATE = -6         /* no workspace bound yet */
} dflash_status;

typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

/* Bits of the sticky device error word. */
#define DFLASH_DERR_KV_CAPACITY 0x1u  /* kv_len + rows beyond pages_per_req * page_size */
#define DFLASH_DERR_PAGE_RANGE 0x2u   /* page table entry outside [0, n_pages) */
#define DFLASH_DERR_TOKEN_RANGE 0x4u  /* anchor or draft/posterior id outside [0, vocab) */
#define DFLASH_DERR_POSITION 0x8u     /* a block/context position >= max_position */
#define DFLASH_DERR_OUTPUT_ROW 0x10u  /* output_ids write past out_stride */
#define DFLASH_DERR_TIMEOUT 0x20u     /* a bounded wait inside a kernel gave up */
#define DFLASH_DERR_ROW_RANGE 0x40u   /* inject: negative n_rows, or rows outside [0, total_rows) */

/*
 * Draft model shape.  The draft shares the target's embedding and lm_head,
 * so its hidden size equals the embedding width ("Inside SGLang", Step 4;
 * CSDN article, "Draft 模型结构").
 *   n_sel          number of selected target layers (target_layer_ids);
 *                  the fc input width is n_sel * target_hidden.
 *   block_size     S, including the anchor.
 *   page_size      rows per KV page; must be 64.
 *   sliding_window host array [n_layers]; 0 = full attention, W > 0 keeps a
 *                  context key at position pk for a query at pq iff pq-pk < W
 *                  (Kimi-K2.6 draft card: sliding_window 2048 on layers 0-4).
 *   max_batch      largest batch any call will pass.
 *   max_rows       rows processed per internal chunk of dflash_inject_context
 *                  (larger calls are chunked); also bounds workspace size.
 *   max_position   positions (context + block) must stay below this; sizes
 *                  the RoPE table.
 *   kv_fp8         0: the K/V pages hold the configured dtype.  1: they hold
 *                  one-byte OCP FP8 E4M3 codes (CSDN article, Kimi-K2.6 draft
 *                  card: "KV cache per token (FP8)" of 6 x 2 x 8 x 128 bytes =
 *                  12 KiB, i.e. one byte per element and no per-token scale):
 *                  element x of layer l's K (V) is stored as the E4M3 code
 *                  nearest to x / k_scale[l] (x / v_scale[l]) -- IEEE float32
 *                  division, ties to the even code, magnitudes beyond 448
 *                  saturate to 448 -- and attention reads code value * scale.
 *                  The scales are given per call in dflash_kv.  bf16
 *                  configurations with head_dim 128 and block_size <= 16 only.
 * Supported: head_dim in {64, 128}; hidden, target_hidden, intermediate and
 * n_heads*head_dim multiples of 128; n_heads a multiple of n_kv_heads;
 * block_size in [2, 32]; (n_heads/n_kv_heads)*block_size <= 128.
 */
typedef struct {
  dflash_dtype dtype;
  int32_t target_hidden;
  int32_t n_sel;
  int32_t hidden;
  int32_t n_layers;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate;
  int32_t vocab;
  int32_t mask_token_id;
  int32_t block_size;
  int32_t page_size;
  const int32_t *sliding_window;
  float rms_eps;
  float rope_theta;
  int32_t max_batch;
  int32_t max_rows;
  int32_t max_position;
  int32_t kv_fp8;
} dflash_config;

/*
 * Weights (device pointers).  Per-layer members are HOST arrays of n_layers
 * device pointers; the arrays are copied by dflash_create.
 *   fc_w       [hidden, n_sel*target_hidden]  (column block j = layer id j of
 *              target_layer_ids, in list order: CSDN article,
 *              extract_context_feature)
 *   qkv_w[l]   [(n_heads + 2*n_kv_heads)*head_dim, hidden]: q rows, then k
 *              rows, then v rows (SGLang's fused qkv_proj)
 *   o_w[l]     [hidden, n_heads*head_dim]
 *   gate_up_w[l] [2*intermediate, hidden]: gate rows, then up rows
 *   down_w[l]  [hidden, intermediate]
 *   *_norm_g   RMSNorm gains: hidden_norm/final_norm/in_norm/post_norm
 *              [hidden]; q_norm/k_norm [head_dim] shared by all heads
 *   embed, lm_head  the target's [vocab, hidden] embedding and output head
 */
typedef struct {
  const void *fc_w;
  const void *hidden_norm_g;
  const void *final_norm_g;
  const void *embed;
  const void *lm_head;
  const void *const *qkv_w;
  const void *const *o_w;
  const void *const *gate_up_w;
  const void *const *down_w;
  const void *const *in_norm_g;
  const void *const *post_norm_g;
  const void *const *q_norm_g;
  const void *const *k_norm_g;
} dflash_weights;

/*
 * Paged draft KV cache (caller-owned, device).  Draft context K/V come only
 * from projected target features, never from draft hidden states ("Inside
 * SGLang", Step 4: two K/V sources).
 *   k_pages/v_pages  HOST arrays [n_layers] of device pointers, each to
 *                    [n_pages, page_size, n_kv_heads, head_dim] elements of
 *                    the configured dtype (one byte each with kv_fp8).
 *   page_table       device int32 [batch, pages_per_req]: page of logical
 *                    position p of request b is page_table[b][p / page_size]
 *                    (logical positions and physical slots are distinct,
 *                    "Inside SGLang", Step 3); with a draft window, the page
 *                    of p is page_table[b][(p / page_size) % pages_per_req].
 *   kv_len           device int32 [batch]: committed context rows.  Context
 *                    row i of request b has position i.
 *   draft_window     0: every committed row is kept.  W > 0: draft KV
 *                    windowing ("Inside SGLang", worker/memory section: "a
 *                    private compact mapping over the shared global index
 *                    space"; CSDN article, --speculative-dflash-draft-window-size):
 *                    the cache keeps only the most recent W committed rows of
 *                    each request, at their original positions, in a ring of
 *                    pages_per_req pages (at least ceil(W / page_size) + 1);
 *                    every block query sees exactly those rows and the block
 *                    (a sliding layer still applies its own window on top);
 *                    dflash_inject_context skips rows that fall out of the
 *                    window within the same call.
 *   k_scale/v_scale  HOST float arrays [n_layers] (read during the call),
 *                    kv_fp8 only (else ignored, may be NULL): the per-layer
 *                    scales of the FP8 codes (positive, finite).
 */
typedef struct {
  void *const *k_pages;
  void *const *v_pages;
  const int32_t *page_table;
  int32_t pages_per_req;
  int32_t n_pages;
  int32_t *kv_len;
  int32_t draft_window;
  const float *k_scale;
  const float *v_scale;
} dflash_kv;

typedef struct dflash_handle dflash_handle;

/* Validate the config, copy it and the weight pointer arrays, prepare TMA
 * descriptors.  No device memory is allocated.  *out is NULL on failure. */
int dflash_create(const dflash_config *cfg, const dflash_weights *w, dflash_handle **out);

/* Release host-side state.  Does not touch caller buffers.  NULL is a no-op. */
void dflash_destroy(dflash_handle *h);

/* Bytes of device workspace the handle needs (depends on max_batch,
 * max_rows, max_position and the shape). */
int dflash_workspace_size(const dflash_handle *h, size_t *bytes);

/* Bind caller-allocated device workspace (256-byte aligned, >= the size
 * above).  Initialises it on `stream` (RoPE table, counters, error word).
 * The workspace must not be shared by calls that may overlap on the GPU. */
int dflash_bind_workspace(dflash_handle *h, void *dev_ptr, size_t bytes, dflash_stream_t stream);

/*
 * Step 1: context injection ("Inside SGLang", Steps 1 and 7; CSDN article,
 * "fused_kv_materialize").  For request b, feature rows
 * row_offset[b] .. row_offset[b]+n_rows[b]-1 are projected
 * (concat -> fc -> hidden_norm) and written to every layer's cache at
 * positions kv_len[b] .. kv_len[b]+n_rows[b]-1 (k-normed and rotated K,
 * plain V); then kv_len[b] += n_rows[b].  Rows of the feature buffers that
 * belong to no request (e.g. rejected rows of a dense [B, S] verify block)
 * are never written: this is the prefix-valid commit of Step 7.  In bf16
 * with fused launches (the default), when total_rows is above 128 and at
 * most min(max_rows, max_batch * block_size), they are not projected either:
 * the rows of the requests are first gathered into the workspace (16-byte
 * aligned feature pointers).  Results do not depend on which way a call
 * goes beyond float rounding.
 *   batch        <= max_batch
 *   total_rows   rows in each feature buffer (an upper bound of every row
 *                index used); processed in chunks of max_rows
 *   target_feats HOST array [n_sel] of device pointers, each
 *                [total_rows, target_hidden] (selected layer j first = j-th
 *                entry of target_layer_ids)
 *   row_offset, n_rows  device int32 [batch]; n_rows may be 0
 */
int dflash_inject_context(dflash_handle *h, const dflash_kv *kv, int32_t batch, int32_t total_rows,
                          const void *const *target_feats, const int32_t *row_offset,
                          const int32_t *n_rows, dflash_stream_t stream);

/*
 * Step 2: draft block ("Inside SGLang", Steps 3-4; CSDN article, "draft
 * model predict").  Block ids [anchor[b], mask x (S-1)] at positions
 * kv_len[b] + j; draft layers with non-causal attention over the committed
 * context and all S block rows; final norm; lm_head argmax for rows 1..S-1.
 *   anchor     device int32 [batch]
 *   draft_ids  device int32 [batch, S]: column 0 = anchor, 1..S-1 = argmax
 *              (lowest id among equal maxima)
 *   hidden_out optional device [batch, S, hidden] final-normed hidden states
 *              (configured dtype); NULL to skip
 * The KV cache and kv_len are read only: block K/V never enter the cache.
 */
int dflash_draft_block(dflash_handle *h, const dflash_kv *kv, int32_t batch, const int32_t *anchor,
                       int32_t *draft_ids, void *hidden_out, dflash_stream_t stream);

/*
 * Step 3: greedy verification ("Inside SGLang", Step 6; CSDN article,
 * "target model verify" and SGLang item 8).
 *   accept_len[b] = number of leading i < S-1 with draft[b][i+1] == posterior[b][i]
 *   bonus[b]      = posterior[b][accept_len[b]]
 *   commit_len[b] = accept_len[b] + 1
 *   out_tokens[b] = draft[b][1..accept_len], bonus, then 0 padding   [batch, S]
 *   seq_len[b]    in: start (position of the anchor); out: start+accept+1,
 *                 the crop index of the draft/target caches
 *   output_ids    optional (NULL to skip) device [batch, out_stride]:
 *                 [start .. start+accept] <- draft[b][0..accept],
 *                 [start+accept+1] <- bonus; rows overflowing out_stride set
 *                 DFLASH_DERR_OUTPUT_ROW and are not written.
 * The commit of the verified feature rows into the draft cache is the
 * following dflash_inject_context call with n_rows = commit_len.
 */
int dflash_accept_commit(dflash_handle *h, int32_t batch, const int32_t *draft_ids,
                         const int32_t *posterior, int32_t *seq_len, int32_t *accept_len,
                         int32_t *commit_len, int32_t *bonus, int32_t *out_tokens,
                         int32_t *output_ids, int32_t out_stride, dflash_stream_t stream);

/*
 * Step 3, sampled variant: lossless rejection-sampling verification with the
 * argmax drafter ("Inside SGLang", "Sampling: preserve the proposal
 * distribution the walk actually used": a proposed token y is accepted with
 * probability min(1, p(y)/q(y)); at the first rejection the correction is
 * drawn from the normalised residual [p - q]+; after full acceptance the
 * target supplies a bonus token.  The plain drafter proposes argmax tokens,
 * so q is the point mass at y.)  Random numbers are inputs:
 *   probs      device float32 [batch, S, vocab]: the target's distribution at
 *              block position i (over the token after draft[b][i])
 *   accept_u   device float32 [batch, S-1], uniform on [0, 1):
 *              draft[b][i+1] is accepted iff accept_u[b][i] < probs[b][i][draft[b][i+1]]
 *   exp_noise  device float32 [batch, vocab], Exp(1) variates (> 0): the bonus
 *              (correction or full-acceptance bonus) is the argmax over v of
 *              w(v) / exp_noise[b][v], w the target row at the stop position
 *              with the rejected token's entry set to 0, lowest id on ties
 *              (the "exponential race", an exact draw from w / sum(w))
 * Decisions are taken in float32 (IEEE division and comparison).  All other
 * arguments and outputs as in dflash_accept_commit; a proposed id outside
 * [0, vocab) sets DFLASH_DERR_TOKEN_RANGE and that request is not committed.
 * Caller owns every buffer; the call allocates nothing.
 */
int dflash_accept_commit_sampled(dflash_handle *h, int32_t batch, const int32_t *draft_ids,
                                 const float *probs, const float *accept_u, const float *exp_noise,
                                 int32_t *seq_len, int32_t *accept_len, int32_t *commit_len,
                                 int32_t *bonus, int32_t *out_tokens, int32_t *output_ids,
                                 int32_t out_stride, dflash_stream_t stream);

/*
 * Step 3, sampled variant for a drafter with a real proposal distribution
 * (the DFlash 2 selector's q_rows; "Inside SGLang", "Sampling: preserve the
 * proposal distribution the walk actually used").  q is zero outside each
 * position's K candidates:
 *   cand_ids   device int32 [batch, S-1, K]: candidates of block position i+1
 *   q_rows     device float32 [batch, S-1, K]: their proposal probabilities
 * draft[b][i+1] = y is accepted iff q(y) > 0 and
 * accept_u[b][i] < probs[b][i][y] / q(y) (float32 IEEE division), q(y) the
 * probability of the first candidate equal to y (0 if none: rejected).  At
 * the first rejection the correction is the exponential race over
 * [p - q]+ (p minus q on the candidates, clipped at 0, float32); after full
 * acceptance over the target's last row.  K in [1, 8].  Every other argument
 * and output as in dflash_accept_commit_sampled.
 */
int dflash_accept_commit_sampled_q(dflash_handle *h, int32_t batch, const int32_t *draft_ids,
                                   const float *probs, int32_t K, const int32_t *cand_ids,
                                   const float *q_rows, const float *accept_u,
                                   const float *exp_noise, int32_t *seq_len, int32_t *accept_len,
                                   int32_t *commit_len, int32_t *bonus, int32_t *out_tokens,
                                   int32_t *output_ids, int32_t out_stride, dflash_stream_t stream);

/*
 * DFlash 2 candidate selector ("Inside SGLang", "DFlash 2: replace selection,
 * retain the serving loop").  After the same backbone pass as
 * dflash_draft_block, every draft position j = 1..S-1 keeps the K best
 * lm_head tokens as candidates (their logits are the unary scores U), and a
 * left-to-right walk from the anchor chooses one candidate per position.
 * From predecessor p (the anchor, then the candidate chosen before) candidate
 * c of position j scores
 *     score(p, c) = U(c) + sum_i A[p][i] * (W_h h_j)[i] * B[c][i]
 * with h_j the final-normed hidden state of position j.  Greedy walk: the
 * highest score, earliest candidate on ties.  Sampled walk: the exponential
 * race over q = softmax(score(p, .)) with caller-given Exp(1) noise (largest
 * q_k / noise_k, earliest on ties).  The walk does not search for the best
 * full path.  Logits are never stored: the lm_head launch keeps each
 * 128-token tile's K best per row, a small kernel merges them and walks.
 *
 * dflash_selector:
 *   K        candidates per position, 1..8 (<= vocab)
 *   rank     width of the compatibility term, 1..256
 *   W_h      device [rank, hidden], A and B device [vocab, rank], all in the
 *            configured dtype; W_h 16-byte aligned.  Caller-owned; must
 *            outlive their use.
 * dflash_selector_workspace_size: device bytes the selector needs for this
 * handle's max_batch and block size (per-tile candidate keys of every row,
 * per-row bounds, W_h h_j).  dflash_set_selector binds the weights and that
 * workspace (256-byte aligned, caller-owned, not shared with overlapping
 * calls); NULL sel removes the selector.  block_size must be <= 33.
 *
 * dflash_draft_block_selector: as dflash_draft_block (same anchor, kv and
 * draft_ids layout; column 0 = anchor), with
 *   exp_noise  device float32 [batch, S-1, K] Exp(1) variates (> 0) for the
 *              sampled walk, or NULL for the greedy walk
 *   cand_ids   optional device int32 [batch, S-1, K]: the candidates of every
 *              position in logit order (lower id first among equal logits)
 *   q_rows     optional device float32 [batch, S-1, K]: softmax of the chosen
 *              predecessor's scores: the walk's proposal distribution, the
 *              input of dflash_accept_commit_sampled_q
 * Returns DFLASH_ESTATE when no selector is set.
 */
typedef struct {
  int32_t K;
  int32_t rank;
  const void *W_h;
  const void *A;
  const void *B;
} dflash_selector;

int dflash_selector_workspace_size(const dflash_handle *h, int32_t K, int32_t rank, size_t *bytes);
int dflash_set_selector(dflash_handle *h, const dflash_selector *sel, void *workspace, size_t bytes);
int dflash_draft_block_selector(dflash_handle *h, const dflash_kv *kv, int32_t batch,
                                const int32_t *anchor, const float *exp_noise, int32_t *draft_ids,
                                int32_t *cand_ids, float *q_rows, dflash_stream_t stream);

/* Synchronise `stream`, read the sticky device error word into *word (may be
 * NULL) and clear it.  Returns DFLASH_OK if it was zero, DFLASH_EDEVICE if
 * not. */
int dflash_get_error(dflash_handle *h, dflash_stream_t stream, uint32_t *word);

/*
 * Optional per-kernel timing (off by default).  While enabled, every launch
 * of the three entry points is bracketed by a pair of CUDA events recorded on
 * the launching stream (at most max_records launches; later ones are not
 * recorded).  dflash_profile_collect waits for the recorded events, sums the
 * durations per kernel name into out[0..*n) and forgets the records.
 * Creating the events is a host-side runtime call; no device memory is
 * allocated.
 */
typedef struct {
  char name[32];
  int32_t launches;
  float total_ms;
} dflash_profile_entry;

int dflash_profile_enable(dflash_handle *h, int32_t max_records);
int dflash_profile_disable(dflash_handle *h);
int dflash_profile_collect(dflash_handle *h, dflash_profile_entry *out, int32_t cap, int32_t *n);

/*
 * Token selection that allocates nothing (no counterpart on the pages: it
 * exists for callers that cannot give this library device memory, e.g. a
 * plugin inside a serving engine whose caching allocator owns all device
 * memory, or code that may not call cudaMalloc at all).
 *   ids[r] = argmax_v <hidden[r], lm_head[v]>   (lowest id among equal maxima)
 *   rows    1 .. 32
 *   hidden  device [rows, hidden] in the configured dtype (bf16 only), rows
 *           contiguous, 16-byte aligned (e.g. rows 1..S-1 of
 *           dflash_draft_block's hidden_out); the hidden size must be a
 *           multiple of 64
 *   ids     device int32 [rows]; all -1 when the call's status is non-zero
 *   status  optional device uint32 (NULL: not reported): written when the
 *           call's last kernel runs with the call's device error bits, 0 on
 *           success, DFLASH_DERR_TIMEOUT if a bounded wait inside the GEMM
 *           gave up.  Read it after synchronising the stream.
 * Needs a handle (host memory) but no bound workspace.  Its scratch (argmax
 * keys, GEMM partial tiles and tickets, a status word; about 5.3 MB) is one
 * static device array of the library, held by every GPU that loads it until
 * the process exits.  The first call on a device sets that device up (looks
 * up the array's address and sets kernel attributes): make that first call
 * before any stream capture.  Every call clears the status word, the keys and
 * the tickets on `stream` before its GEMM.  All calls share the one array, so
 * calls that may overlap on the GPU (other streams, other threads) race;
 * serialise them.  No cudaMalloc/cudaFree is made.
 * Returns DFLASH_ECAPACITY for rows > 32 or vocab > 262144, DFLASH_EINVAL
 * for a misaligned hidden, DFLASH_EUNSUPPORTED for fp32 handles or a hidden
 * size that is not a multiple of 64.
 */
int dflash_select_tokens_noalloc(dflash_handle *h, int32_t rows, const void *hidden, int32_t *ids,
                                 uint32_t *status, dflash_stream_t stream);

/* Static description of a status code. */
const char *dflash_status_string(int status);

/* Message of the last failed host-side check in this thread ("" if none). */
const char *dflash_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
