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
// Two launches: the merge (one CTA per draft row; a skipped tile costs one
// key read, issued eight at a time) and the walk (one CTA per request, all
// factor rows staged in shared memory first, then a sequential but tiny walk:
// K dot products of length rank per position).
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

// Insert key x into a descending list top[0..K) (static indexing only).
__device__ __forceinline__ void topk_insert(unsigned long long (&top)[kSelMaxK], int K,
                                            unsigned long long x) {
#pragma unroll
  for (int q = 0; q < kSelMaxK; ++q) {
    if (q < K && x > top[q]) {
      const unsigned long long y = top[q];
      top[q] = x;
      x = y;
    }
  }
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, v, o);
    v = other > v ? other : v;
  }
  return v;
}

// 1. Candidates of one draft row (block (j, b)): every thread keeps the best K
//    keys of its stride of vocabulary tiles -- the first key of eight tiles is
//    read at once, and a tile's list is read on only when its first key can
//    still enter -- then each warp, and finally warp 0, takes K rounds of a
//    warp max.  The row's K candidate keys go to cand[m][0..K).
constexpr int kMergeBatch = 8;
__global__ void __launch_bounds__(kSelThreads) selector_merge_kernel(const __grid_constant__ SelectorParams p) {
  pdl_wait();
  __shared__ unsigned long long s_w[kSelThreads / 32][kSelMaxK];
  const int j = blockIdx.x, b = blockIdx.y, K = p.K;
  const int m = b * p.S + 1 + j;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long top[kSelMaxK];
#pragma unroll
  for (int q = 0; q < kSelMaxK; ++q) top[q] = 0ull;
  unsigned long long least = 0ull;
  for (int t0 = tid; t0 < p.n_vt; t0 += kSelThreads * kMergeBatch) {
    unsigned long long first[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int t = t0 + u * kSelThreads;
      first[u] = t < p.n_vt ? __ldcg(p.topk_keys + ((size_t)t * p.topk_ld + m) * K) : 0ull;
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      if (first[u] <= least) continue;   // the tile was skipped, or cannot enter
      const unsigned long long *src =
          p.topk_keys + ((size_t)(t0 + u * kSelThreads) * p.topk_ld + m) * K;
      unsigned long long xs[kSelMaxK];   // the rest of the tile's list, loaded together
#pragma unroll
      for (int i = 1; i < kSelMaxK; ++i) xs[i] = i < K ? __ldcg(src + i) : 0ull;
      xs[0] = first[u];
#pragma unroll
      for (int i = 0; i < kSelMaxK; ++i) {
        if (i < K && xs[i] > least) {   // descending list: zeros and small keys never enter
          topk_insert(top, K, xs[i]);
#pragma unroll
          for (int q = 0; q < kSelMaxK; ++q)
            if (q == K - 1) least = top[q];
        }
      }
    }
  }
  // each warp's best K
  int head = 0;
  for (int i = 0; i < K; ++i) {
    unsigned long long mine = 0ull;
#pragma unroll
    for (int q = 0; q < kSelMaxK; ++q)
      if (q == head) mine = top[q];
    const unsigned long long best = warp_max_u64(mine);
    if (best != 0ull && mine == best) ++head;
    if (lane == 0) s_w[warp][i] = best;
  }
  __syncthreads();
  if (warp != 0) return;
  // warp 0 over the warps' lists: lane l holds entries l and l + 32 of the
  // flattened [warps][K] array
  const int nkeys = (kSelThreads / 32) * K;
  unsigned long long a0 = lane < nkeys ? s_w[lane / K][lane % K] : 0ull;
  unsigned long long a1 = lane + 32 < nkeys ? s_w[(lane + 32) / K][(lane + 32) % K] : 0ull;
  if (a0 < a1) {
    const unsigned long long t = a0;
    a0 = a1;
    a1 = t;
  }
  int h2 = 0;
  for (int i = 0; i < K; ++i) {
    const unsigned long long mine = h2 == 0 ? a0 : h2 == 1 ? a1 : 0ull;
    const unsigned long long best = warp_max_u64(mine);
    if (best != 0ull && mine == best) ++h2;
    if (lane == i) p.cand_keys[(size_t)m * K + i] = best;
  }
}

// 2. The walk of one request (block b).  Every factor row the walk can read
//    -- B of every candidate, A of the anchor and of every candidate that can
//    be a predecessor -- and W_h h of every position come into shared memory
//    first with independent, coalesced loads; the walk itself (warp 0, lanes
//    over the rank) then reads shared memory only.  `cached` false: the rows
//    are read from global memory instead (large rank x K x S).
template <typename T>
__global__ void __launch_bounds__(kSelThreads) selector_walk_kernel(const __grid_constant__ SelectorParams p,
                                                                     int cached) {
  pdl_wait();
  extern __shared__ __align__(16) uint8_t sm[];
  const int b = blockIdx.x, S = p.S, K = p.K, R = p.rank, n = S - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long *s_key = (unsigned long long *)sm;           // [n][K]
  float *s_rstd = (float *)(s_key + kSelMaxRows * kSelMaxK);      // [n]
  float *s_wh = s_rstd + kSelMaxRows;                             // [n][R]
  T *s_B = (T *)(s_wh + (size_t)n * R);                           // [n*K][R]
  T *s_A = s_B + (size_t)n * K * R;                               // [1 + (n-1)*K][R]
  const int nA = 1 + (n - 1) * K;
  for (int i = tid; i < n * K; i += blockDim.x)
    s_key[i] = __ldcg(p.cand_keys + (size_t)(b * S + 1) * K + i);
  for (int j = tid; j < n; j += blockDim.x) s_rstd[j] = 0.f;
  __syncthreads();
  // row scales of the final RMSNorm when the lm_head read unnormalised rows
  // (every (row, 128-feature part) sum at once); 1 when its operand is
  // already the normalised hidden state (ssq NULL)
  if (p.ssq) {
    const int parts = p.H / 128;
    for (int idx = tid; idx < n * parts; idx += blockDim.x) {
      const int j = idx / parts, part = idx - j * parts;
      atomicAdd(&s_rstd[j], p.ssq[(size_t)part * p.ssq_ld + b * S + 1 + j]);
    }
    __syncthreads();
  }
  for (int j = tid; j < n; j += blockDim.x)
    s_rstd[j] = p.ssq ? rsqrtf(s_rstd[j] / (float)p.H + p.eps) : 1.f;
  __syncthreads();
  const T *A = (const T *)p.A, *Bf = (const T *)p.Bf;
  int anchor = p.anchor[b];
  const bool anchor_ok = anchor >= 0 && anchor < p.vocab;
  for (int idx = tid; idx < n * R; idx += blockDim.x) {
    const int j = idx / R, i = idx - j * R;
    s_wh[idx] = p.wh[(size_t)(b * S + 1 + j) * R + i] * s_rstd[j];
  }
  const bool vec = (R * sizeof(T)) % 16 == 0 && ((uintptr_t)A & 15) == 0 && ((uintptr_t)Bf & 15) == 0;
  if (cached && vec) {
    // 16-byte copies, four in flight per thread; s_A follows s_B, so one
    // index runs over both: rows [0, n*K) are B rows of the candidates, then
    // the anchor's A row and the A rows of positions 0..n-2's candidates
    const int per_row = R * (int)sizeof(T) / 16, nB = n * K;
    const int tot = (nB + nA) * per_row;
    uint4 *dst = reinterpret_cast<uint4 *>(s_B);
    for (int x0 = tid; x0 < tot; x0 += 4 * blockDim.x) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int x = x0 + u * blockDim.x;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (x < tot) {
          const int row = x / per_row, c = x - row * per_row;
          int tok = -1;
          const T *src = Bf;
          if (row < nB) {
            tok = s_key[row] ? argmax_key_index(s_key[row]) : -1;
          } else {
            src = A;
            const int r2 = row - nB;
            if (r2 == 0)
              tok = anchor_ok ? anchor : -1;
            else
              tok = s_key[r2 - 1] ? argmax_key_index(s_key[r2 - 1]) : -1;
          }
          if (tok >= 0) v[u] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)tok * R) + c);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int x = x0 + u * blockDim.x;
        if (x < tot) dst[x] = v[u];
      }
    }
  } else if (cached) {
    for (int idx = tid; idx < n * K * R; idx += blockDim.x) {
      const int row = idx / R, i = idx - row * R;
      const unsigned long long key = s_key[row];
      s_B[idx] = key ? Bf[(size_t)argmax_key_index(key) * R + i] : T(0.f);
    }
    for (int idx = tid; idx < nA * R; idx += blockDim.x) {
      const int row = idx / R, i = idx - row * R;
      int tok = -1;
      if (row == 0) {
        tok = anchor_ok ? anchor : -1;
      } else {
        const unsigned long long key = s_key[row - 1];
        tok = key ? argmax_key_index(key) : -1;
      }
      s_A[idx] = tok >= 0 ? A[(size_t)tok * R + i] : T(0.f);
    }
  }
  __syncthreads();
  if (warp != 0) return;
  int pred = anchor, pred_row = 0;   // row of s_A holding A[pred]
  if (lane == 0) p.draft_ids[(size_t)b * S] = anchor;
  for (int j = 0; j < n; ++j) {
    float sc[kSelMaxK];
    int id[kSelMaxK];
    const bool pred_ok = pred >= 0 && pred < p.vocab;
#pragma unroll
    for (int k = 0; k < kSelMaxK; ++k) {
      sc[k] = -INFINITY;
      id[k] = -1;
      if (k < K) {
        const unsigned long long key = s_key[j * K + k];
        const int c = key ? argmax_key_index(key) : -1;
        float dot = 0.f;
        if (c >= 0 && pred_ok) {
          if (cached) {
            const T *a = s_A + (size_t)pred_row * R, *bb = s_B + (size_t)(j * K + k) * R;
            for (int i = lane; i < R; i += 32) dot += to_f32(a[i]) * s_wh[j * R + i] * to_f32(bb[i]);
          } else {
            for (int i = lane; i < R; i += 32)
              dot += to_f32(A[(size_t)pred * R + i]) * s_wh[j * R + i] * to_f32(Bf[(size_t)c * R + i]);
          }
        }
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
    if (y < 0) {   // no candidate at all: K <= vocab is checked, so never
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
    pred_row = 1 + j * K + pick;
  }
}

constexpr size_t kSelWalkCacheBytes = 200 * 1024;   // staged factor rows at most

size_t walk_smem(const SelectorParams &p, size_t elem, bool cached) {
  const size_t n = p.S - 1;
  size_t b = kSelMaxRows * kSelMaxK * 8 + kSelMaxRows * 4 + n * p.rank * 4;
  if (cached) b += (n * p.K + 1 + (n - 1) * p.K) * p.rank * elem;
  return b;
}

}  // namespace

// Shared-memory opt-in of the walk kernels on the current device (kernel
// attributes are per device; run once per handle with the others).
cudaError_t prepare_selector() {
  cudaError_t e = cudaFuncSetAttribute(selector_walk_kernel<bf16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSelWalkCacheBytes + 4096);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(selector_walk_kernel<float>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSelWalkCacheBytes + 4096);
}

cudaError_t launch_selector_walk(const SelectorParams &p, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  if (p.K < 1 || p.K > kSelMaxK || p.rank < 1 || p.rank > kSelMaxRank || p.S < 2 ||
      p.S - 1 > kSelMaxRows || p.H % 128 || !p.cand_keys)
    return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(selector_merge_kernel, dim3(p.S - 1, p.B), dim3(kSelThreads), 0, s, p);
  if (e != cudaSuccess) return e;
  const size_t elem = p.store == ST_BF16 ? 2 : 4;
  constexpr size_t kCacheLimit = kSelWalkCacheBytes;
  const bool cached = walk_smem(p, elem, true) <= kCacheLimit;
  const size_t smem = walk_smem(p, elem, cached);
  if (p.store == ST_BF16)
    return launch_pdl(selector_walk_kernel<bf16>, dim3(p.B), dim3(kSelThreads), smem, s, p,
                      cached ? 1 : 0);
  return launch_pdl(selector_walk_kernel<float>, dim3(p.B), dim3(kSelThreads), smem, s, p,
                    cached ? 1 : 0);
}

}  // namespace dflash
