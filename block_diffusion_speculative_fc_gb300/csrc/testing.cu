// Test-only entry points: the tensor-core GEMM on its own, the FP8 encoder of
// the K/V cache epilogue (include/dflash_testing.h).
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

extern "C" int dflash_test_e4m3_encode(const float *x, int32_t n, float scale, uint8_t *codes,
                                       dflash_stream_t stream) {
  if (n < 0 || (n > 0 && (!x || !codes)) || !(scale > 0.f)) return DFLASH_EINVAL;
  if (n == 0) return DFLASH_OK;
  const int pairs = (n + 1) / 2;
  e4m3_encode_kernel<<<(pairs + 255) / 256, 256, 0, (cudaStream_t)stream>>>(x, n, scale, codes);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ECUDA;
}
