// Internal launch interface between the C-ABI runtime (dflash_api.cu) and the
// kernels.  Host-side declarations only; no torch types anywhere.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dflash {

enum StoreType { ST_F32 = 0, ST_BF16 = 1 };

// What the GEMM epilogue does with the fp32 tile Y[m, n] = sum_k A[m,k] W[n,k].
enum EpiOp {
  EPI_STORE_F32 = 0,  // out_f32[m*ld + n] = y
  EPI_RESID = 1,      // out_f32[m*ld + n] += y                (residual stream)
  EPI_SWIGLU = 2,     // out_act[m*ld + n] = silu(y_gate) * y_up (paired tiles)
  EPI_ARGMAX = 3,     // argmax_keys[m] = max(key(y, n))
  EPI_QKV = 4,        // per-head RMSNorm (q, k) + RoPE -> q/k/v block buffers
  EPI_KV_CACHE = 5,   // k-norm + RoPE (k), plain v -> paged cache rows (slot)
  EPI_STORE_ACT = 6,  // out_act[m*ld + n] = y
  EPI_RESID_NORM = 7, // x = out_f32 += y; out_act = x * norm_gain; ssq_out += x^2 per row
  EPI_STORE_NORM = 8, // out_act = y * norm_gain; ssq_out = y^2 per row
  EPI_TOPK = 9,       // topk_keys[n0/128][m][0..K) = the tile's K best keys of row m
};

// Deferred RMSNorm.  A producer of a tensor that feeds a normalised GEMM
// (EPI_RESID_NORM / EPI_STORE_NORM, or the block embedding) writes
//   out_act[m, n] = x[m, n] * g[n]                      (the GEMM's A operand)
//   ssq[n / 128][m] = sum over its 128 features of x^2   (one slot per tile)
// and the consuming GEMM multiplies row m of its result by
//   rstd[m] = 1 / sqrt(sum_t ssq[t][m] / H + eps)
// before its own epilogue: RMSNorm(x) W^T = rstd * ((x * g) W^T) because the
// projection is linear.  Slots are summed in a fixed order (deterministic).

struct EpiParams {
  int op;
  int N;                         // valid output features of this segment
  int ld;                        // row stride of the output (elements)
  float *out_f32;
  void *out_act;
  unsigned long long *argmax_keys;
  // per-head epilogues
  void *q_out, *k_out, *v_out;   // EPI_QKV: [M, n_heads*D], [M, kvh*D], [M, kvh*D]
  void *k_cache, *v_cache;       // EPI_KV_CACHE: [n_pages*page, kvh, D]
  const void *q_gain, *k_gain;   // [D]
  const int *row_pos;            // [M] RoPE position of each row
  const int *row_slot;           // [M] cache row of each row, -1 = skip
  const float2 *rope;            // [max_position, D/2] (cos, sin)
  int n_heads, n_kv_heads, head_dim;
  float eps;
  // deferred RMSNorm of the A operand (NULL: the operand is already final)
  const float *ssq_in;           // [ssq_parts][ssq_ld]
  int ssq_parts, ssq_ld;
  float norm_eps;                // eps of that RMSNorm
  float inv_h;                   // 1 / (normalised width)
  // EPI_RESID_NORM / EPI_STORE_NORM outputs
  const void *norm_gain;         // [N] gain of the next RMSNorm
  float *ssq_out;                // [N / 128][ssq_ld]
  // EPI_TOPK: per 128-feature tile and row, the tile's topk best argmax keys
  // (descending; 0 = none) at topk_keys[((n0 / 128) * topk_ld + m) * topk + i],
  // or zeros when even the tile's best key is below the row's running bound:
  // topk_bound[s * topk_ld + m], s < topk, holds the best key of the tiles
  // t % topk == s so far (zeroed before the launch); the smallest slot is a
  // lower bound on the row's topk-th best key
  unsigned long long *topk_keys;
  unsigned long long *topk_bound;
  int topk, topk_ld;
  // EPI_KV_CACHE into an FP8 E4M3 cache: code of x / scale, one byte per element
  int kv_fp8;
  float k_scale, v_scale;
};

constexpr int kMaxSrc = 8;   // sources of the K-split A operand (selected layers)
constexpr int kMaxSeg = 8;   // weight segments of a grouped launch

struct GemmA {
  const void *ptr[kMaxSrc];  // each [M, k_per_src], row stride ld
  int64_t ld;
  int k_per_src;
  int n_src;
};

struct GemmSeg {
  const void *W;   // [N, K] row-major (row stride ldw)
  int64_t ldw;
  int N;           // rows of W used by this segment (for EPI_SWIGLU: 2 * I)
  EpiParams epi;
};

struct GemmProblem {
  GemmA A;
  int M, K;
  int nseg;
  GemmSeg seg[kMaxSeg];
  // optional device row count (<= M), read by the launch after its
  // predecessor finished: tiles past it are not scheduled (M bounds the
  // schedule and the scratch)
  const int *M_dev;
};

struct AttnParams {
  const void *q;       // [B*S, n_heads*D]
  const void *kb, *vb; // [B*S, kvh*D] block keys / values
  const void *k_cache, *v_cache;  // [n_pages*page, kvh, D]
  const int *page_table;
  const int *kv_len;
  void *out;           // [B*S, n_heads*D]
  int B, S, n_heads, n_kv_heads, head_dim, page_size, pages_per_req, n_pages;
  int window;          // 0 = full
  float scale;
  unsigned int *err;
  int draft_window;    // 0 = off; W > 0: the page table is a ring, keys below kv_len - W hidden
  int fp8;             // context pages hold E4M3 codes: value = code * k_scale / v_scale
  float k_scale, v_scale;
};

struct AttnScratch {
  int *item_start;   // [max_batch * kvh + 1]
  int *pps;          // [2]: pages per split; the tensor-core kernel's work-queue position
  int *order;        // [max_items][8] the tensor-core kernel's work queue (two int4 per item)
  float *part_o;     // [max_items][R][128]
  float *part_ml;    // [max_items][R][2]
  int *tickets;      // [max_batch * kvh], zero between launches
};

// DFlash 2 candidate selector: merge of the per-tile top-K keys and the walk.
constexpr int kSelMaxK = 8;       // candidates per position
constexpr int kSelMaxRank = 256;  // rank of the compatibility term
struct SelectorParams {
  const unsigned long long *topk_keys;  // [n_vt][topk_ld][K] (EPI_TOPK)
  unsigned long long *cand_keys;        // [topk_ld][K] the merged candidates of every row
  int n_vt, topk_ld;                    // 128-row vocabulary tiles; row stride
  const float *wh;                      // [B*S, rank] W_h (x * g), before the row's rstd
  const float *ssq;                     // [H / 128][ssq_ld] sums of squares of the final norm
                                        // (NULL: the lm_head operand was already normalised)
  int ssq_ld, H;
  float eps;
  const void *A, *Bf;                   // [V, rank] predecessor / successor factors (model dtype)
  int store;                            // ST_F32 / ST_BF16: dtype of A and Bf
  const int *anchor;                    // [B]
  const float *exp_noise;               // [B, S-1, K] Exp(1) or NULL (greedy walk)
  int *draft_ids;                       // [B, S]
  int *cand_ids;                        // [B, S-1, K] or NULL
  float *q_rows;                        // [B, S-1, K] or NULL
  int B, S, K, rank, vocab;
  unsigned int *err;
};
// Two launches: the per-row merge of the tiles' lists, then the walk.
cudaError_t launch_selector_walk(const SelectorParams &p, cudaStream_t s);
cudaError_t prepare_selector();

constexpr int kTcMaxCtas = 160;   // persistent tensor-core GEMM grid cap (>= SM count)
constexpr int kMaxPhases = 5;     // phases of one fused tensor-core launch (GEMMs and GEMM-free ones)
constexpr int kMaxGemmPhases = 4; // dependent GEMMs a caller may chain in one launch

// ---- launchers (return cudaGetLastError()) ----
cudaError_t launch_gemm_tc(const GemmProblem &P, float *partials, int *counters, int max_tiles,
                           unsigned int *err, cudaStream_t s, unsigned long long *trace = nullptr);
// Work a GEMM program can do besides its GEMMs (bf16 only).
// ProgramEmbed: the block embedding, as a phase without GEMM work before the
// first GEMM (rows M = B*S; writes x, x*g, the per-128-feature sums of
// squares, the RoPE positions and clears the argmax keys -- what
// launch_embed does).  ProgramFinalize: draft_ids from the argmax keys, done
// by the last CTA to leave the launch.
struct ProgramEmbed {
  const void *table;            // [vocab, H]
  const int *anchor, *kv_len;   // [B]
  int M, S, H, vocab, mask_id, max_position;
  float *x;                     // [M, H]
  const void *gain;             // [H] first layer's input norm
  void *xg;                     // [M, H]
  float *ssq;                   // [H/128][ssq_ld]
  int ssq_ld;
  int *row_pos;                 // [M]
  unsigned long long *keys;     // [M]
};
struct ProgramFinalize {
  const unsigned long long *keys;
  const int *anchor;            // [B]
  int M, S;
  int *draft_ids;               // [M]
};

// ProgramInject: the injection row map of feature rows row0 .. row0+rows-1
// (into row_slot / row_pos), computed during the first phase for the K/V
// phase that follows; with advance set, the last CTA out also advances kv_len
// by n_rows (what launch_inject_prep / launch_inject_finalize do).
struct ProgramInject {
  int B, row0, rows;
  const int *row_offset, *n_rows;
  int *kv_len;
  const int *page_table;
  int pages_per_req, n_pages, page_size, max_position;
  int *row_slot, *row_pos;
  int advance, total_rows;
  int draft_window;             // 0: off; W > 0: ring page table (inject_rows.cuh)
};

// ProgramNorm: a GEMM-free phase placed just before a program's last GEMM.
// Every row m of the fp32 residual x is normalised with the sums of squares
// the previous phase wrote (ssq[t * ssq_ld + m], one per 128-feature part):
// out[m, :] = x[m, :] * rsqrt(sum_t ssq / H + eps) * gain, rounded to the
// store type, into out (the last GEMM's operand) and, when non-NULL, out2.
struct ProgramNorm {
  const float *x;               // [M, H]
  const float *ssq;             // [H/128][ssq_ld]
  int ssq_ld;
  const void *gain;             // [H]
  void *out, *out2;             // [M, H] bf16
  int M, H;
  float eps;
};

// Up to kMaxGemmPhases dependent GEMMs of equal row count in one cooperative
// launch, separated by grid barriers (grid_bar: two zeroed words); an
// optional embedding phase first, an optional normalisation phase before the
// last GEMM (each takes one of the kMaxPhases) and an optional argmax
// finalisation at the end.
cudaError_t launch_gemm_program(const GemmProblem *probs, int n, float *partials, int *counters,
                                int max_tiles, unsigned int *grid_bar, unsigned int *err,
                                cudaStream_t s, unsigned long long *trace = nullptr,
                                const ProgramEmbed *embed = nullptr,
                                const ProgramFinalize *fin = nullptr,
                                const ProgramInject *inject = nullptr,
                                const ProgramNorm *norm = nullptr);
size_t gemm_tc_partials_bytes();
int gemm_tc_trace_slots();   // timestamps per CTA written by a traced launch
int gemm_tc_tiles(int n_tiles, int M, bool pair);
int gemm_tc_num_sms();   // SMs of the current device (cached)
void gemm_tc_set_head_pairs(bool on);   // QKV head-pair tiles (default on)
cudaError_t prepare_gemm_tc();
cudaError_t launch_attention_mma(const AttnParams &p, const AttnScratch &w, cudaStream_t s);
size_t attention_mma_scratch_items(int max_batch, int kvh);
cudaError_t prepare_attention_mma();
// Whether launch_attention_mma takes its cluster path (few (request, head) pairs).
bool attention_mma_uses_cluster(const AttnParams &p);
// tcgen05 attention: bf16 cache, head_dim 128, 64-row pages, at most 64 query
// rows per (request, KV head), batch <= 1024.
bool attention_tc_eligible(const AttnParams &p);
cudaError_t launch_attention_tc(const AttnParams &p, const AttnScratch &w, cudaStream_t s);
cudaError_t prepare_attention_tc();
cudaError_t launch_gemm_simt(int store, const GemmProblem &P, cudaStream_t s);
cudaError_t launch_attention_simt(int store, const AttnParams &p, cudaStream_t s);

cudaError_t launch_embed(int store, const void *embed, const int *anchor, const int *kv_len,
                         int B, int S, int H, int vocab, int mask_id, int max_position,
                         float *x, const void *norm_gain, void *xg, float *ssq, int ssq_ld,
                         int *row_pos, unsigned long long *keys, unsigned int *err,
                         cudaStream_t s);
cudaError_t launch_rmsnorm(int in_f32, int store, const void *x, const void *gain, int M, int H,
                           float eps, void *out, void *out2, cudaStream_t s);
cudaError_t launch_argmax_finalize(const unsigned long long *keys, const int *anchor, int B, int S,
                                   int *draft_ids, cudaStream_t s);
cudaError_t launch_inject_prep(int B, int row0, int rows, const int *row_offset, const int *n_rows,
                               const int *kv_len, const int *page_table, int pages_per_req,
                               int n_pages, int page_size, int max_position, int draft_window,
                               int *row_slot, int *row_pos, unsigned int *err, cudaStream_t s);
// Prefix-valid compaction of the injection's feature rows: the rows of every
// request (row_offset[b] .. + n_rows[b] - 1 of the n_sel buffers [total_rows,
// th]) go, in request order, to rows coff[b] .. coff[b] + crows[b] - 1 of x
// [rows, n_sel * th] (bf16); crows[b] = n_rows[b], or 0 (flagged) when those
// rows are not inside the buffers; *count = the rows kept.
struct FeatPtrs {
  const void *p[kMaxSrc];
};
cudaError_t launch_inject_compact(int B, int total_rows, const FeatPtrs &src, int n_sel, int th,
                                  const int *row_offset, const int *n_rows, void *x, int *coff,
                                  int *crows, int *count, unsigned int *err, cudaStream_t s);
cudaError_t launch_inject_finalize(int B, int total_rows, const int *row_offset,
                                   const int *n_rows, int *kv_len, int capacity,
                                   unsigned int *err, cudaStream_t s);
// One-time kernel attribute setup (dynamic shared memory limits).
cudaError_t prepare_kernels();
cudaError_t launch_rope_table(float2 *table, int max_position, int head_dim, float theta,
                              cudaStream_t s);
cudaError_t launch_accept(int B, int S, int vocab, const int *draft, const int *post,
                          int *seq_len, int *accept_len, int *commit_len, int *bonus,
                          int *out_tokens, int *output_ids, int out_stride, unsigned int *err,
                          cudaStream_t s);

// Lossless sampled verification (accept.cu); keys, tickets: [B] zeroed
// scratch that the launch leaves zeroed; sms: SM count (grid sizing).
cudaError_t launch_accept_sampled(int B, int S, int vocab, const int *draft, const float *probs,
                                  const float *u, const float *noise, unsigned long long *keys,
                                  int *tickets, int *seq_len, int *accept_len, int *commit_len,
                                  int *bonus, int *out_tokens, int *output_ids, int out_stride,
                                  unsigned int *err, cudaStream_t s, int sms,
                                  const int *cand = nullptr, const float *qr = nullptr,
                                  int K = 0);

// Host-side helpers implemented next to the handle (dflash_api.cu).
int handle_lm_head(const dflash_handle *h, const void **lm_head, int *hidden, int *vocab,
                   int *dtype);
void set_last_error(const char *msg);

}  // namespace dflash
