// DFlash 2 candidate selector: the walk over the candidate lattice
// ("Inside SGLang: DFlash and DFlash 2 Implementation", "DFlash 2: replace
// selection, retain the serving loop").
//
// The lm_head launch before this kernel (EPI_TOPK) left, for every
// 128-token vocabulary tile and draft row, that tile's K best (logit, id) keys
// -- or nothing when the tile could not reach the row's top K -- and W_h (x*g)
// for every row.  One CTA per request then
//   1. merges the tiles' lists into the row's K candidates (logit order, lower
//      id first on ties: the key order),
//   2. scales the logits and W_h h by the row's final-RMSNorm factor, and
//   3. walks the positions left to right: from predecessor p (the anchor,
//      then the candidate chosen before) every candidate c of the position
//      scores U(c) + <A[p] * W_h h, B[c]>; the walk takes the highest score
//      (earliest candidate on ties) or, given Exp(1) noise, samples from the
//      softmax of the scores by the exponential race (largest q_k / e_k,
//      earliest on ties).  q_rows is that softmax: the proposal distribution
//      a lossless sampled verification needs.
// The walk is sequential by definition but tiny (K dot products of length
// rank per position); the merge reads one key per skipped tile.
#include "common.cuh"
#include "kernels.h"

namespace dflash {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelMaxRows = 32;   // S - 1 positions per request

// value of an argmax key (inverse of the order-preserving float map)
__device__ __forceinline__ float key_value(unsigned long long k) {
  unsigned int u = (unsigned int)(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
  return __uint_as_float(u);
}

template <typename T>
__global__ void __launch_bounds__(kSelThreads) selector_walk_kernel(const __grid_constant__ SelectorParams p) {
  pdl_wait();
  __shared__ unsigned long long s_key[kSelMaxRows][kSelMaxK];
  __shared__ float s_wh[kSelMaxRows][kSelMaxRank];
  __shared__ float s_rstd[kSelMaxRows];
  const int b = blockIdx.x, S = p.S, K = p.K, R = p.rank;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int n = S - 1;

  // row scales of the final RMSNorm from its per-128-feature sums of squares
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int m = b * S + 1 + j;
    float ss = 0.f;
    for (int part = 0; part < p.H / 128; ++part) ss += p.ssq[(size_t)part * p.ssq_ld + m];
    s_rstd[j] = rsqrtf(ss / (float)p.H + p.eps);
  }
  // 1. candidates: each lane keeps its best K keys over a stride of tiles
  //    (a tile's list is descending and ends at its first zero), then K rounds
  //    of a warp max
  for (int j = warp; j < n; j += nw) {
    const int m = b * S + 1 + j;
    unsigned long long top[kSelMaxK];
#pragma unroll
    for (int q = 0; q < kSelMaxK; ++q) top[q] = 0ull;
    unsigned long long least = 0ull;   // top[K-1]
    for (int t = lane; t < p.n_vt; t += 32) {
      const unsigned long long *src = p.topk_keys + ((size_t)t * p.topk_ld + m) * K;
      for (int i = 0; i < K; ++i) {
        unsigned long long x = __ldcg(src + i);
        if (x <= least) break;   // descending: nothing after it can enter either
#pragma unroll
        for (int q = 0; q < kSelMaxK; ++q) {
          if (q < K && x > top[q]) {
            const unsigned long long y = top[q];
            top[q] = x;
            x = y;
          }
        }
#pragma unroll
        for (int q = 0; q < kSelMaxK; ++q)
          if (q == K - 1) least = top[q];
      }
    }
    int head = 0;
    for (int i = 0; i < K; ++i) {
      unsigned long long mine = 0ull;
#pragma unroll
      for (int q = 0; q < kSelMaxK; ++q)
        if (q == head) mine = top[q];
      unsigned long long best = mine;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if (best != 0ull && mine == best) ++head;
      if (lane == 0) s_key[j][i] = best;
    }
  }
  // 2. W_h h of every position: W_h (x * g) times the row's scale
  for (int idx = threadIdx.x; idx < n * R; idx += blockDim.x) {
    const int j = idx / R, i = idx - j * R;
    s_wh[j][i] = p.wh[(size_t)(b * S + 1 + j) * R + i] * s_rstd[j];
  }
  __syncthreads();
  if (warp != 0) return;
  // 3. the walk (one warp: lanes split the rank of every dot product)
  const T *A = (const T *)p.A, *Bf = (const T *)p.Bf;
  int pred = p.anchor[b];
  if (lane == 0) p.draft_ids[(size_t)b * S] = pred;
  for (int j = 0; j < n; ++j) {
    float sc[kSelMaxK];
    int id[kSelMaxK];
    const bool pred_ok = pred >= 0 && pred < p.vocab;
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k) {
      sc[k] = -INFINITY;
      id[k] = -1;
      if (k < K) {
        const unsigned long long key = s_key[j][k];
        const int c = key ? argmax_key_index(key) : -1;
        float dot = 0.f;
        if (c >= 0 && pred_ok)
          for (int i = lane; i < R; i += 32)
            dot += to_f32(A[(size_t)pred * R + i]) * s_wh[j][i] * to_f32(Bf[(size_t)c * R + i]);
        dot = warp_sum(dot);
        if (c >= 0) {
          id[k] = c;
          sc[k] = key_value(key) * s_rstd[j] + dot;
        }
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k) mx = fmaxf(mx, sc[k]);
    float q[kSelMaxK], sum = 0.f;
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k) {
      q[k] = id[k] >= 0 ? expf(sc[k] - mx) : 0.f;
      sum += q[k];
    }
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k) q[k] = q[k] / sum;
    int pick = 0;
    if (!p.exp_noise) {
#pragma unroll
      for (int k = 1; k < kSelMaxK; ++k)
        if (sc[k] > sc[pick]) pick = k;
    } else {
      const float *e = p.exp_noise + ((size_t)b * n + j) * K;
      float best = -1.f;
#pragma unroll
      for (int k = 0; k < kSelMaxK; ++k) {
        if (k < K && id[k] >= 0) {
          const float w = q[k] / e[k];
          if (w > best) {
            best = w;
            pick = k;
          }
        }
      }
    }
    int y = -1;
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k)
      if (k == pick) y = id[k];
    if (y < 0) {   // no candidate at all (vocabulary smaller than K cannot happen: checked)
      if (lane == 0) raise_error(p.err, DFLASH_DERR_TOKEN_RANGE);
      y = 0;
    }
    if (lane == 0) p.draft_ids[(size_t)b * S + 1 + j] = y;
    const size_t o = ((size_t)b * n + j) * K;
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k) {
      if (k < K && lane == k) {
        if (p.cand_ids) p.cand_ids[o + k] = id[k];
        if (p.q_rows) p.q_rows[o + k] = q[k];
      }
    }
    pred = y;
  }
}

}  // namespace

cudaError_t launch_selector_walk(const SelectorParams &p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  if (p.K < 1 || p.K > kSelMaxK || p.rank < 1 || p.rank > kSelMaxRank || p.S < 2 ||
      p.S - 1 > kSelMaxRows || p.H % 128)
    return cudaErrorInvalidValue;
  if (p.store == ST_BF16)
    return launch_pdl(selector_walk_kernel<bf16>, dim3(p.B), dim3(kSelThreads), 0, s, p);
  return launch_pdl(selector_walk_kernel<float>, dim3(p.B), dim3(kSelThreads), 0, s, p);
}

}  // namespace dflash
