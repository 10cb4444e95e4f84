// Test-only entry points: the tensor-core GEMM on its own, the FP8 encoder of
// the K/V cache epilogue, the bf16 attention kernels on their own
// (include/dflash_testing.h).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "../../include/dflash_testing.h"
#include "common.cuh"
#include "kernels.h"

using namespace dflash;

extern "C" size_t dflash_test_gemm_scratch(int32_t M, int32_t N) {
  const int tiles = gemm_tc_tiles((N + 127) / 128, M > 0 ? M : 1, false);
  return gemm_tc_partials_bytes() + 4 * (size_t)tiles + 256;
}

extern "C" int dflash_test_gemm(int32_t M, int32_t N, int32_t K, int32_t n_src,
                                const void *const *A, int32_t lda, const void *W, int32_t ldw,
                                int32_t op, void *out, void *act_out, void *scratch,
                                size_t scratch_bytes, dflash_stream_t stream) {
  return dflash_test_gemm_traced(M, N, K, n_src, A, lda, W, ldw, op, out, act_out, scratch,
                                 scratch_bytes, nullptr, stream);
}

extern "C" int dflash_test_gemm_traced(int32_t M, int32_t N, int32_t K, int32_t n_src,
                                       const void *const *A, int32_t lda, const void *W,
                                       int32_t ldw, int32_t op, void *out, void *act_out,
                                       void *scratch, size_t scratch_bytes,
                                       unsigned long long *trace, dflash_stream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0 || n_src <= 0 || n_src > kMaxSrc || !A || !W || !scratch)
    return DFLASH_EINVAL;
  if (K % n_src || (K / n_src) % 64) return DFLASH_EUNSUPPORTED;
  if (scratch_bytes < dflash_test_gemm_scratch(M, N)) return DFLASH_ECAPACITY;
  if (op != EPI_STORE_F32 && op != EPI_SWIGLU && op != EPI_ARGMAX) return DFLASH_EINVAL;
  if (op == EPI_SWIGLU && (N % 2 || !act_out)) return DFLASH_EINVAL;
  if (op != EPI_SWIGLU && !out) return DFLASH_EINVAL;
  cudaStream_t s = (cudaStream_t)stream;
  GemmProblem P;
  std::memset(&P, 0, sizeof(P));
  for (int j = 0; j < n_src; ++j) P.A.ptr[j] = A[j];
  P.A.ld = lda;
  P.A.k_per_src = K / n_src;
  P.A.n_src = n_src;
  P.M = M;
  P.K = K;
  GemmSeg &g = P.seg[P.nseg++];
  g.W = W;
  g.ldw = ldw;
  g.N = N;
  std::memset(&g.epi, 0, sizeof(g.epi));
  g.epi.op = op;
  g.epi.N = N;
  g.epi.ld = op == EPI_SWIGLU ? N / 2 : N;
  g.epi.out_f32 = (float *)out;
  g.epi.out_act = act_out;
  g.epi.argmax_keys = (unsigned long long *)out;
  char *base = (char *)scratch;
  unsigned int *err = (unsigned int *)base;
  float *partials = (float *)(base + 256);
  int *counters = (int *)(base + 256 + gemm_tc_partials_bytes());
  const int tiles = gemm_tc_tiles((N + 127) / 128, M, false);
  if (cudaMemsetAsync(base, 0, 256, s) != cudaSuccess) return DFLASH_ECUDA;
  if (cudaMemsetAsync(counters, 0, 4 * (size_t)tiles, s) != cudaSuccess) return DFLASH_ECUDA;
  if (prepare_gemm_tc() != cudaSuccess) return DFLASH_ECUDA;
  if (launch_gemm_tc(P, partials, counters, tiles, err, s, trace) != cudaSuccess) return DFLASH_ECUDA;
  return DFLASH_OK;
}

// ---------------------------------------------------------------- programs
namespace {
int program_tiles(int n, int32_t M, const int32_t *N, const int32_t *op) {
  int t = 0;
  bool pair = false;
  for (int i = 0; i < n; ++i) pair |= op[i] == 2;
  for (int i = 0; i < n; ++i) {
    const int feats = op[i] == 2 ? N[i] / 2 : N[i];
    t += gemm_tc_tiles((feats + 127) / 128, M, pair);
  }
  return t;
}
}  // namespace

extern "C" size_t dflash_test_program_scratch(int32_t n_phases, int32_t M, const int32_t *N,
                                              const int32_t *op) {
  if (n_phases <= 0 || n_phases > kMaxGemmPhases || M <= 0 || !N || !op) return 0;
  return 256 + gemm_tc_partials_bytes() + 4 * (size_t)program_tiles(n_phases, M, N, op) + 256;
}

extern "C" int dflash_test_gemm_program(int32_t n_phases, int32_t M, const int32_t *N,
                                        const int32_t *K, const void *const *A,
                                        const void *const *W, const int32_t *op,
                                        void *const *out, void *scratch, size_t scratch_bytes,
                                        dflash_stream_t stream) {
  return dflash_test_gemm_program_traced(n_phases, M, N, K, A, W, op, out, scratch, scratch_bytes,
                                         nullptr, stream);
}

extern "C" int32_t dflash_test_trace_slots(void) { return gemm_tc_trace_slots(); }

extern "C" int dflash_test_gemm_program_traced(int32_t n_phases, int32_t M, const int32_t *N,
                                               const int32_t *K, const void *const *A,
                                               const void *const *W, const int32_t *op,
                                               void *const *out, void *scratch,
                                               size_t scratch_bytes, unsigned long long *trace,
                                               dflash_stream_t stream) {
  if (n_phases <= 0 || n_phases > kMaxGemmPhases || M <= 0 || !N || !K || !A || !W || !op || !out ||
      !scratch)
    return DFLASH_EINVAL;
  for (int i = 0; i < n_phases; ++i) {
    if (N[i] <= 0 || K[i] <= 0 || !A[i] || !W[i] || !out[i]) return DFLASH_EINVAL;
    if (op[i] != 0 && op[i] != 1 && op[i] != 2) return DFLASH_EINVAL;
    if (op[i] == 2 && N[i] % 2) return DFLASH_EINVAL;
    if (K[i] % 64) return DFLASH_EUNSUPPORTED;
  }
  if (scratch_bytes < dflash_test_program_scratch(n_phases, M, N, op)) return DFLASH_ECAPACITY;
  cudaStream_t s = (cudaStream_t)stream;
  GemmProblem P[kMaxGemmPhases];
  for (int i = 0; i < n_phases; ++i) {
    std::memset(&P[i], 0, sizeof(P[i]));
    P[i].A.ptr[0] = A[i];
    P[i].A.ld = K[i];
    P[i].A.k_per_src = K[i];
    P[i].A.n_src = 1;
    P[i].M = M;
    P[i].K = K[i];
    GemmSeg &g = P[i].seg[P[i].nseg++];
    g.W = W[i];
    g.ldw = K[i];
    g.N = N[i];
    std::memset(&g.epi, 0, sizeof(g.epi));
    g.epi.op = op[i] == 0 ? EPI_STORE_F32 : op[i] == 1 ? EPI_STORE_ACT : EPI_SWIGLU;
    g.epi.N = N[i];
    g.epi.ld = op[i] == 2 ? N[i] / 2 : N[i];
    g.epi.out_f32 = (float *)out[i];
    g.epi.out_act = out[i];
  }
  const int tiles = program_tiles(n_phases, M, N, op);
  char *base = (char *)scratch;
  unsigned int *err = (unsigned int *)base;
  float *partials = (float *)(base + 256);
  int *counters = (int *)(base + 256 + gemm_tc_partials_bytes());
  unsigned int *grid_bar = (unsigned int *)((char *)counters + 4 * (size_t)tiles);
  if (cudaMemsetAsync(base, 0, 256, s) != cudaSuccess) return DFLASH_ECUDA;
  if (cudaMemsetAsync(counters, 0, 4 * (size_t)tiles + 256, s) != cudaSuccess) return DFLASH_ECUDA;
  if (prepare_gemm_tc() != cudaSuccess) return DFLASH_ECUDA;
  if (launch_gemm_program(P, n_phases, partials, counters, tiles, grid_bar, err, s, trace) !=
      cudaSuccess)
    return DFLASH_ECUDA;
  return DFLASH_OK;
}

namespace {
// The K/V cache epilogue's encoder (e4m3x2 in common.cuh) on n given values.
__global__ void e4m3_encode_kernel(const float *__restrict__ x, int n, float scale,
                                   uint8_t *__restrict__ codes) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const uint32_t c = e4m3x2(x[i], i + 1 < n ? x[i + 1] : 0.f, scale);
  codes[i] = (uint8_t)(c & 0xFF);
  if (i + 1 < n) codes[i + 1] = (uint8_t)(c >> 8);
}
}  // namespace

// ------------------------------------------------------------------ QKV GEMM
namespace {
size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }
size_t qkv_tiles(int32_t M, int32_t N) { return (size_t)gemm_tc_tiles((N + 127) / 128, M, false); }
}  // namespace

extern "C" size_t dflash_test_qkv_scratch(int32_t M, int32_t N, int32_t max_position) {
  if (M <= 0 || N <= 0 || max_position <= 0) return 0;
  return 256 + gemm_tc_partials_bytes() + align256(4 * qkv_tiles(M, N)) +
         (size_t)max_position * 64 * sizeof(float2);
}

extern "C" int dflash_test_qkv(int32_t M, int32_t K, int32_t n_heads, int32_t n_kv_heads,
                               int32_t head_dim, int32_t max_position, float rope_theta, float eps,
                               const void *A, const void *W, const float *ssq, const void *q_gain,
                               const void *k_gain, const int32_t *row_pos, void *q_out,
                               void *k_out, void *v_out, void *scratch, size_t scratch_bytes,
                               dflash_stream_t stream) {
  if (M <= 0 || K <= 0 || n_heads <= 0 || n_kv_heads <= 0 || max_position <= 0 || !A || !W ||
      !q_gain || !k_gain || !row_pos || !q_out || !k_out || !v_out || !scratch)
    return DFLASH_EINVAL;
  if (head_dim != 128 && head_dim != 64) return DFLASH_EUNSUPPORTED;
  if (K % 128 || !(rope_theta > 0.f) || !(eps >= 0.f)) return DFLASH_EINVAL;
  const int N = (n_heads + 2 * n_kv_heads) * head_dim;
  if (N % 128) return DFLASH_EUNSUPPORTED;
  if (scratch_bytes < dflash_test_qkv_scratch(M, N, max_position)) return DFLASH_ECAPACITY;
  cudaStream_t s = (cudaStream_t)stream;
  GemmProblem P;
  std::memset(&P, 0, sizeof(P));
  P.A.ptr[0] = A;
  P.A.ld = K;
  P.A.k_per_src = K;
  P.A.n_src = 1;
  P.M = M;
  P.K = K;
  GemmSeg &g = P.seg[P.nseg++];
  g.W = W;
  g.ldw = K;
  g.N = N;
  char *base = (char *)scratch;
  unsigned int *err = (unsigned int *)base;
  float *partials = (float *)(base + 256);
  int *counters = (int *)(base + 256 + gemm_tc_partials_bytes());
  float2 *rope = (float2 *)(base + 256 + gemm_tc_partials_bytes() + align256(4 * qkv_tiles(M, N)));
  EpiParams &e = g.epi;
  std::memset(&e, 0, sizeof(e));
  e.op = EPI_QKV;
  e.N = N;
  e.n_heads = n_heads;
  e.n_kv_heads = n_kv_heads;
  e.head_dim = head_dim;
  e.eps = eps;
  e.q_out = q_out;
  e.k_out = k_out;
  e.v_out = v_out;
  e.q_gain = q_gain;
  e.k_gain = k_gain;
  e.row_pos = row_pos;
  e.rope = rope;
  if (ssq) {
    e.ssq_in = ssq;
    e.ssq_parts = K / 128;
    e.ssq_ld = M;
    e.norm_eps = eps;
    e.inv_h = 1.0f / (float)K;
  }
  if (cudaMemsetAsync(base, 0, 256, s) != cudaSuccess) return DFLASH_ECUDA;
  if (cudaMemsetAsync(counters, 0, 4 * qkv_tiles(M, N), s) != cudaSuccess) return DFLASH_ECUDA;
  if (prepare_gemm_tc() != cudaSuccess) return DFLASH_ECUDA;
  if (launch_rope_table(rope, max_position, head_dim, rope_theta, s) != cudaSuccess)
    return DFLASH_ECUDA;
  if (launch_gemm_tc(P, partials, counters, (int)qkv_tiles(M, N), err, s) != cudaSuccess)
    return DFLASH_ECUDA;
  return DFLASH_OK;
}

extern "C" int dflash_test_e4m3_encode(const float *x, int32_t n, float scale, uint8_t *codes,
                                       dflash_stream_t stream) {
  if (n < 0 || (n > 0 && (!x || !codes)) || !(scale > 0.f)) return DFLASH_EINVAL;
  if (n == 0) return DFLASH_OK;
  const int pairs = (n + 1) / 2;
  e4m3_encode_kernel<<<(pairs + 255) / 256, 256, 0, (cudaStream_t)stream>>>(x, n, scale, codes);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ECUDA;
}

// ------------------------------------------------------------ attention
namespace {
struct AttnScratchLayout {
  size_t item_start, pps, order, part_o, part_ml, tickets, total;
};
AttnScratchLayout attn_scratch_layout(int B, int n_heads, int kvh, int S) {
  AttnScratchLayout L;
  const size_t items = attention_mma_scratch_items(B, kvh);
  const size_t R = (size_t)(n_heads / kvh) * S;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = (o + std::max<size_t>(bytes, 1) + 255) & ~(size_t)255;
    return at;
  };
  L.item_start = take(4 * ((size_t)B * kvh + 1));
  L.pps = take(8);
  L.order = take(32 * items);
  L.part_o = take(4 * items * R * 128);
  L.part_ml = take(8 * items * R);
  L.tickets = take(4 * (size_t)B * kvh);
  L.total = o;
  return L;
}
}  // namespace

extern "C" size_t dflash_test_attention_scratch(int32_t B, int32_t n_heads, int32_t n_kv_heads,
                                                int32_t S) {
  if (B <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 || S <= 0) return 0;
  return attn_scratch_layout(B, n_heads, n_kv_heads, S).total;
}

extern "C" int dflash_test_attention(int32_t kernel, int32_t B, int32_t S, int32_t n_heads,
                                     int32_t n_kv_heads, int32_t pages_per_req, int32_t n_pages,
                                     int32_t window, int32_t draft_window, const void *q,
                                     const void *kb, const void *vb, const void *k_cache,
                                     const void *v_cache, const int32_t *page_table,
                                     const int32_t *kv_len, void *out, void *scratch,
                                     size_t scratch_bytes, uint32_t *err, dflash_stream_t stream) {
  if (B <= 0 || S <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 || !q || !kb || !vb ||
      !k_cache || !v_cache || !page_table || !kv_len || !out || !scratch || !err)
    return DFLASH_EINVAL;
  if (kernel != 0 && kernel != 1) return DFLASH_EINVAL;
  const AttnScratchLayout L = attn_scratch_layout(B, n_heads, n_kv_heads, S);
  if (scratch_bytes < L.total) return DFLASH_ECAPACITY;
  AttnParams a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.kb = kb;
  a.vb = vb;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.page_table = page_table;
  a.kv_len = kv_len;
  a.out = out;
  a.B = B;
  a.S = S;
  a.n_heads = n_heads;
  a.n_kv_heads = n_kv_heads;
  a.head_dim = 128;
  a.page_size = 64;
  a.pages_per_req = pages_per_req;
  a.n_pages = n_pages;
  a.window = window;
  a.scale = 1.0f / sqrtf(128.0f);
  a.err = (unsigned int *)err;
  a.draft_window = draft_window;
  uint8_t *base = (uint8_t *)scratch;
  AttnScratch w;
  w.item_start = (int *)(base + L.item_start);
  w.pps = (int *)(base + L.pps);
  w.order = (int *)(base + L.order);
  w.part_o = (float *)(base + L.part_o);
  w.part_ml = (float *)(base + L.part_ml);
  w.tickets = (int *)(base + L.tickets);
  cudaStream_t s = (cudaStream_t)stream;
  if (prepare_kernels() != cudaSuccess) return DFLASH_ECUDA;
  if (cudaMemsetAsync(w.tickets, 0, 4 * (size_t)B * n_kv_heads, s) != cudaSuccess) return DFLASH_ECUDA;
  cudaError_t e;
  if (kernel == 0) {
    if (!attention_tc_eligible(a)) return DFLASH_EUNSUPPORTED;
    e = launch_attention_tc(a, w, s);
  } else {
    e = launch_attention_mma(a, w, s);
  }
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ECUDA;
}
