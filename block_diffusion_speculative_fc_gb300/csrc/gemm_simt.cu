// CUDA-core GEMM with the shared epilogues: the fp32 path of the library.
//
// tcgen05 has no exact-fp32 MMA kind, so fp32 configurations contract on the
// CUDA cores: Y[m, n] = sum_k A[m, k] * W[n, k] with fp32 FMA.  One CTA makes a
// tile of 128 output features x 32 token rows (x2 for a SwiGLU gate/up pair).
// The A operand may be split along K over several source tensors (the
// selected target layers), so the concatenation of the CSDN DFlash article's
// extract_context_feature is never materialised.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dflash {

namespace {
constexpr int BN = 128, BM = 32, BK = 32, THREADS = 256;
constexpr int WLD = BK + 1, TLD = BN + 1;

__device__ __forceinline__ int seg_tiles(const GemmSeg &s, bool pair) {
  const int n = pair ? s.N / 2 : s.N;
  return (n + BN - 1) / BN;
}
}  // namespace

template <typename T, bool PAIR>
__global__ void __launch_bounds__(THREADS) gemm_simt_kernel(const __grid_constant__ GemmProblem P) {
  pdl_wait();
  __shared__ float smem[(PAIR ? 2 : 1) * BN * WLD + BM * WLD];
  float *Ws = smem;                              // [PAIR?2:1][BN][WLD]
  float *As = smem + (PAIR ? 2 : 1) * BN * WLD;  // [BM][WLD]

  // which weight segment / feature tile
  int t = blockIdx.x, si = 0;
  while (si < P.nseg - 1 && t >= seg_tiles(P.seg[si], PAIR)) t -= seg_tiles(P.seg[si++], PAIR);
  const GemmSeg &seg = P.seg[si];
  const int n0 = t * BN;
  const int m0 = blockIdx.y * BM;
  const int nrows = PAIR ? seg.N / 2 : seg.N;
  const T *W = (const T *)seg.W;

  const int tid = threadIdx.x;
  const int tf = tid & 31, tm = tid >> 5;
  float acc[PAIR ? 2 : 1][4][4];
#pragma unroll
  for (int p = 0; p < (PAIR ? 2 : 1); ++p)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[p][i][j] = 0.f;

  for (int k0 = 0; k0 < P.K; k0 += BK) {
#pragma unroll
    for (int p = 0; p < (PAIR ? 2 : 1); ++p) {
      const int wrow0 = n0 + (p ? seg.N / 2 : 0);
      for (int idx = tid; idx < BN * BK; idx += THREADS) {
        const int r = idx / BK, k = idx % BK;
        float v = 0.f;
        if (n0 + r < nrows && k0 + k < P.K) v = to_f32(W[(int64_t)(wrow0 + r) * seg.ldw + k0 + k]);
        Ws[p * BN * WLD + r * WLD + k] = v;
      }
    }
    {
      const int src = k0 / P.A.k_per_src;
      const int kk0 = k0 - src * P.A.k_per_src;
      const T *A = (const T *)P.A.ptr[src];
      for (int idx = tid; idx < BM * BK; idx += THREADS) {
        const int r = idx / BK, k = idx % BK;
        float v = 0.f;
        if (m0 + r < P.M && kk0 + k < P.A.k_per_src) v = to_f32(A[(int64_t)(m0 + r) * P.A.ld + kk0 + k]);
        As[r * WLD + k] = v;
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < BK; ++k) {
      float a[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) a[j] = As[(tm * 4 + j) * WLD + k];
#pragma unroll
      for (int p = 0; p < (PAIR ? 2 : 1); ++p)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float w = Ws[p * BN * WLD + (tf + 32 * i) * WLD + k];
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[p][i][j] = fmaf(a[j], w, acc[p][i][j]);
        }
    }
    __syncthreads();
  }

  // stage the fp32 tile(s) [BM][TLD] in shared memory for the epilogue
  float *t0 = smem, *t1 = smem + BM * TLD;
#pragma unroll
  for (int p = 0; p < (PAIR ? 2 : 1); ++p)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) (p ? t1 : t0)[(tm * 4 + j) * TLD + tf + 32 * i] = acc[p][i][j];
  __syncthreads();
  const int rows = min(BM, P.M - m0);
  __shared__ int s_int[kEpiScratchInts];
  run_epilogue<T>(seg.epi, t0, PAIR ? t1 : nullptr, TLD, m0, rows, n0, tid, THREADS, s_int,
                  [] { __syncthreads(); });
}

cudaError_t launch_gemm_simt(int store, const GemmProblem &P, cudaStream_t s) {
  if (P.M <= 0 || P.nseg <= 0) return cudaSuccess;
  const bool pair = P.seg[0].epi.op == EPI_SWIGLU;
  int tiles = 0;
  for (int i = 0; i < P.nseg; ++i) {
    const int n = pair ? P.seg[i].N / 2 : P.seg[i].N;
    tiles += (n + BN - 1) / BN;
  }
  dim3 grid(tiles, (P.M + BM - 1) / BM);
  if (store != ST_F32) return cudaErrorInvalidValue;   // bf16 runs on the tensor cores
  if (pair) return launch_pdl(gemm_simt_kernel<float, true>, grid, dim3(THREADS), 0, s, P);
  return launch_pdl(gemm_simt_kernel<float, false>, grid, dim3(THREADS), 0, s, P);
}

}  // namespace dflash
