// GEMM epilogues shared by every GEMM kernel of the library.
//
// A GEMM hands over an fp32 tile Y[r][c] (r = token row m0 + r, c = output
// feature n0 + c, 128 features wide) staged in shared memory; the epilogue
// turns it into the step's output:
//   EPI_QKV       per-head RMSNorm of q and k, RoPE of q and k, plain v
//                 ("Inside SGLang", Step 4: DFlashAttention computes block
//                 Q/K/V, normalizes Q/K, applies RoPE).
//   EPI_KV_CACHE  k-norm and RoPE of k, plain v, written to the paged cache
//                 row of each context row (CSDN DFlash article,
//                 "fused_kv_materialize": K RMSNorm + K RoPE + V relayout
//                 for all layers, heads and tokens).
//   EPI_SWIGLU    silu(gate) * up of a paired gate/up tile.
//   EPI_ARGMAX    greedy token choice without materialising logits.
//   EPI_RESID / EPI_STORE_*  residual add / plain stores.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace dflash {

// Rotate-half RoPE on one head held by a warp (component i pairs with
// i + D/2), optionally preceded by a per-head RMSNorm with gain g[D].
template <typename T>
__device__ __forceinline__ void head_epilogue(const float *src, int D, bool norm, bool rope,
                                              const T *gain, float eps, const float2 *rope_row,
                                              T *dst, int lane) {
  const int half = D >> 1;
  float rstd = 1.f;
  if (norm) {
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) ss += src[i] * src[i];
    ss = warp_sum(ss);
    rstd = rsqrtf(ss / (float)D + eps);
  }
  for (int i = lane; i < half; i += 32) {
    float lo = src[i], hi = src[i + half];
    if (norm) {
      lo *= rstd * to_f32(gain[i]);
      hi *= rstd * to_f32(gain[i + half]);
    }
    if (rope) {
      const float2 cs = rope_row[i];
      const float a = lo * cs.x - hi * cs.y;
      const float b = hi * cs.x + lo * cs.y;
      lo = a;
      hi = b;
    }
    dst[i] = from_f32<T>(lo);
    dst[i + half] = from_f32<T>(hi);
  }
}

// t0: fp32 tile [rows][ldt] (features n0 .. n0+127); t1: the "up" tile of a
// SwiGLU pair.  All `nthreads` threads of the caller take part; the caller
// synchronises before (tile complete) and after (tile reuse).
template <typename T>
__device__ void run_epilogue(const EpiParams &e, const float *t0, const float *t1, int ldt, int m0,
                             int rows, int n0, int tid, int nthreads) {
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  switch (e.op) {
    case EPI_STORE_F32:
    case EPI_RESID:
    case EPI_STORE_ACT:
    case EPI_SWIGLU: {
      const int nvalid = e.op == EPI_SWIGLU ? e.N / 2 : e.N;
      for (int idx = tid; idx < rows * 128; idx += nthreads) {
        const int r = idx >> 7, c = idx & 127, n = n0 + c;
        if (n >= nvalid) continue;
        const int64_t o = (int64_t)(m0 + r) * e.ld + n;
        const float y = t0[r * ldt + c];
        if (e.op == EPI_STORE_F32)
          e.out_f32[o] = y;
        else if (e.op == EPI_RESID)
          e.out_f32[o] += y;
        else if (e.op == EPI_STORE_ACT)
          ((T *)e.out_act)[o] = from_f32<T>(y);
        else
          ((T *)e.out_act)[o] = from_f32<T>(silu(y) * t1[r * ldt + c]);
      }
      break;
    }
    case EPI_ARGMAX: {
      for (int r = warp; r < rows; r += nwarps) {
        unsigned long long best = 0ull;
        for (int c = lane; c < 128; c += 32) {
          const int n = n0 + c;
          if (n < e.N) {
            const unsigned long long k = argmax_key(t0[r * ldt + c], n);
            best = k > best ? k : best;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
          best = other > best ? other : best;
        }
        if (lane == 0 && best) atomicMax(e.argmax_keys + m0 + r, best);
      }
      break;
    }
    case EPI_QKV:
    case EPI_KV_CACHE: {
      const int D = e.head_dim;
      const int hpt = 128 / D;  // heads per 128-feature tile
      const int kvd = e.n_kv_heads * D;
      for (int item = warp; item < rows * hpt; item += nwarps) {
        const int r = item / hpt, hh = item % hpt;
        const int f0 = n0 + hh * D;
        if (f0 >= e.N) continue;
        const int m = m0 + r;
        const int hg = f0 / D;
        const float *src = t0 + r * ldt + hh * D;
        const float2 *rope_row = e.rope + (int64_t)e.row_pos[m] * (D >> 1);
        if (e.op == EPI_QKV) {
          if (hg < e.n_heads) {
            T *dst = (T *)e.q_out + (int64_t)m * e.n_heads * D + hg * D;
            head_epilogue<T>(src, D, true, true, (const T *)e.q_gain, e.eps, rope_row, dst, lane);
          } else if (hg < e.n_heads + e.n_kv_heads) {
            T *dst = (T *)e.k_out + (int64_t)m * kvd + (hg - e.n_heads) * D;
            head_epilogue<T>(src, D, true, true, (const T *)e.k_gain, e.eps, rope_row, dst, lane);
          } else {
            T *dst = (T *)e.v_out + (int64_t)m * kvd + (hg - e.n_heads - e.n_kv_heads) * D;
            head_epilogue<T>(src, D, false, false, (const T *)nullptr, e.eps, rope_row, dst, lane);
          }
        } else {
          const int slot = e.row_slot[m];
          if (slot < 0) continue;
          if (hg < e.n_kv_heads) {
            T *dst = (T *)e.k_cache + (int64_t)slot * kvd + hg * D;
            head_epilogue<T>(src, D, true, true, (const T *)e.k_gain, e.eps, rope_row, dst, lane);
          } else {
            T *dst = (T *)e.v_cache + (int64_t)slot * kvd + (hg - e.n_kv_heads) * D;
            head_epilogue<T>(src, D, false, false, (const T *)nullptr, e.eps, rope_row, dst, lane);
          }
        }
      }
      break;
    }
    default:
      break;
  }
}

}  // namespace dflash
