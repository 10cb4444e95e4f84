// CUDA-core block attention: the fp32 path of the library (tcgen05 and
// mma.sync have no exact-fp32 kind; bf16 configurations use attention_mma.cu).
//
// Non-causal attention of the S block queries of every query head over
// [committed context keys ; all S block keys] ("Inside SGLang", Step 4: two
// K/V sources inside draft attention; CSDN DFlash article, is_causal=False).
// One CTA per (request, KV head) holds the G*S query rows of that KV head's
// query-head group and streams keys in tiles of 32 with an online softmax.
// Sliding layers keep a context key at position pk for the query at position
// pq only when pq - pk < window (Kimi-K2.6 draft card, sliding_window 2048).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace dflash {

namespace {
constexpr int KT = 32, THREADS = 256;
}

size_t attention_simt_smem(int R, int D) {
  return sizeof(float) * ((size_t)R * (D + 1) + (size_t)R * D + KT * (D + 1) + KT * D +
                          (size_t)R * (KT + 1) + 3 * (size_t)R);
}

template <typename T>
__global__ void __launch_bounds__(THREADS) attn_simt_kernel(const __grid_constant__ AttnParams p) {
  pdl_wait();
  const int b = blockIdx.x / p.n_kv_heads, g = blockIdx.x % p.n_kv_heads;
  const int G = p.n_heads / p.n_kv_heads, S = p.S, R = G * S, D = p.head_dim;
  const int kvd = p.n_kv_heads * D;
  extern __shared__ float sm[];
  float *Qs = sm;                       // [R][D+1]
  float *Os = Qs + R * (D + 1);         // [R][D]
  float *Ks = Os + R * D;               // [KT][D+1]
  float *Vs = Ks + KT * (D + 1);        // [KT][D]
  float *Ps = Vs + KT * D;              // [R][KT+1]
  float *mrow = Ps + R * (KT + 1), *lrow = mrow + R, *srow = lrow + R;
  const int tid = threadIdx.x;

  const T *q = (const T *)p.q;
  for (int idx = tid; idx < R * D; idx += THREADS) {
    const int r = idx / D, d = idx % D;
    const int h = g * G + r / S, j = r % S;
    Qs[r * (D + 1) + d] = to_f32(q[((int64_t)(b * S + j) * p.n_heads + h) * D + d]) * p.scale;
    Os[r * D + d] = 0.f;
  }
  for (int r = tid; r < R; r += THREADS) {
    mrow[r] = -INFINITY;
    lrow[r] = 0.f;
  }
  const int cap = p.pages_per_req * p.page_size;
  const bool ring = p.draft_window > 0;   // draft KV windowing: ring page table, no capacity
  int kv = p.kv_len[b];
  if ((!ring && kv > cap) || kv < 0) {
    if (tid == 0) raise_error(p.err, DFLASH_DERR_KV_CAPACITY);
    kv = kv < 0 ? 0 : cap;
  }
  // first key query j=0 can see: the draft window's newest W rows, the layer window
  const int lw = ring ? max(0, kv - p.draft_window) : 0;
  const int lo = p.window > 0 ? max(lw, kv - p.window + 1) : lw;
  const int nctx = kv - lo, total = nctx + S;
  const T *kc = (const T *)p.k_cache, *vc = (const T *)p.v_cache;
  const T *kb = (const T *)p.kb, *vb = (const T *)p.vb;
  __syncthreads();

  for (int kt0 = 0; kt0 < total; kt0 += KT) {
    for (int idx = tid; idx < KT * D; idx += THREADS) {
      const int k = idx / D, d = idx % D, kk = kt0 + k;
      float kv_k = 0.f, kv_v = 0.f;
      if (kk < nctx) {
        const int pos = lo + kk;
        const int lp = pos / p.page_size;
        const int page = p.page_table[(int64_t)b * p.pages_per_req + (ring ? lp % p.pages_per_req : lp)];
        if (page >= 0 && page < p.n_pages) {
          const int64_t row = (int64_t)page * p.page_size + pos % p.page_size;
          kv_k = to_f32(kc[row * kvd + g * D + d]);
          kv_v = to_f32(vc[row * kvd + g * D + d]);
        } else if (d == 0) {
          raise_error(p.err, DFLASH_DERR_PAGE_RANGE);
        }
      } else if (kk < total) {
        const int64_t row = (int64_t)b * S + (kk - nctx);
        kv_k = to_f32(kb[row * kvd + g * D + d]);
        kv_v = to_f32(vb[row * kvd + g * D + d]);
      }
      Ks[k * (D + 1) + d] = kv_k;
      Vs[k * D + d] = kv_v;
    }
    __syncthreads();
    for (int idx = tid; idx < R * KT; idx += THREADS) {
      const int r = idx / KT, k = idx % KT, kk = kt0 + k;
      bool valid = kk < total;
      if (valid && kk < nctx && p.window > 0) valid = (kv + r % S) - (lo + kk) < p.window;
      float s = -INFINITY;
      if (valid) {
        s = 0.f;
        for (int d = 0; d < D; ++d) s = fmaf(Qs[r * (D + 1) + d], Ks[k * (D + 1) + d], s);
      }
      Ps[r * (KT + 1) + k] = s;
    }
    __syncthreads();
    for (int r = tid; r < R; r += THREADS) {
      float mx = mrow[r];
      for (int k = 0; k < KT; ++k) mx = fmaxf(mx, Ps[r * (KT + 1) + k]);
      const float sc = mx == -INFINITY ? 1.f : expf(mrow[r] - mx);
      float sum = 0.f;
      for (int k = 0; k < KT; ++k) {
        const float s = Ps[r * (KT + 1) + k];
        const float e = s == -INFINITY ? 0.f : expf(s - mx);
        Ps[r * (KT + 1) + k] = e;
        sum += e;
      }
      lrow[r] = lrow[r] * sc + sum;
      mrow[r] = mx;
      srow[r] = sc;
    }
    __syncthreads();
    for (int idx = tid; idx < R * D; idx += THREADS) {
      const int r = idx / D, d = idx % D;
      float o = Os[r * D + d] * srow[r];
      for (int k = 0; k < KT; ++k) o = fmaf(Ps[r * (KT + 1) + k], Vs[k * D + d], o);
      Os[r * D + d] = o;
    }
    __syncthreads();
  }
  T *out = (T *)p.out;
  for (int idx = tid; idx < R * D; idx += THREADS) {
    const int r = idx / D, d = idx % D;
    const int h = g * G + r / S, j = r % S;
    out[((int64_t)(b * S + j) * p.n_heads + h) * D + d] = from_f32<T>(Os[r * D + d] / lrow[r]);
  }
}

cudaError_t launch_attention_simt(int store, const AttnParams &p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  const int R = (p.n_heads / p.n_kv_heads) * p.S;
  const size_t smem = attention_simt_smem(R, p.head_dim);
  if (store != ST_F32) return cudaErrorInvalidValue;   // bf16 runs on the tensor cores
  return launch_pdl(attn_simt_kernel<float>, dim3(p.B * p.n_kv_heads), dim3(THREADS), smem, s, p);
}

cudaError_t prepare_attention_simt() {
  const int smem = (int)attention_simt_smem(128, 128);
  return cudaFuncSetAttribute(attn_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem);
}

cudaError_t prepare_kernels() {
  cudaError_t e = prepare_attention_simt();
  if (e == cudaSuccess) e = prepare_gemm_tc();
  if (e == cudaSuccess) e = prepare_attention_mma();
  if (e == cudaSuccess) e = prepare_attention_tc();
  if (e == cudaSuccess) e = prepare_selector();
  return e;
}

}  // namespace dflash
