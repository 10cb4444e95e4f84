// Greedy verification acceptance and commit: one warp per request.
//
// "Inside SGLang: DFlash and DFlash 2 Implementation", Step 6: the greedy
// kernel compares candidates[:, 1:] with the target's preceding rows, stops at
// the first mismatch, takes the target token there as bonus and builds the
// padded output row.  CSDN DFlash article, "target model verify":
// acceptance_length = sum(cumprod(block[1:] == posterior[:-1])), output_ids
// writes and start += acceptance_length + 1.
//
// A prefix product of matches is the position of the first zero bit of the
// lane-wise match ballot, so one __ballot_sync and one __ffs replace the
// cumulative product.
#include "common.cuh"
#include "kernels.h"

namespace dflash {

// Commit of one request by one warp, lane = block position: out_tokens,
// output_ids, accept/commit/bonus and the crop index (seq_len).  d / d_next:
// this lane's draft id and the next lane's.
__device__ __forceinline__ void commit_row(int b, int S, int lane, int acc, int bonus_id, int d,
                                           int d_next, int *seq_len, int *accept_len,
                                           int *commit_len, int *bonus, int *out_tokens,
                                           int *output_ids, int out_stride, unsigned int *err) {
  const bool live = lane < S;
  const int start = seq_len[b];
  const bool write_ids = output_ids != nullptr;
  if (write_ids && (start < 0 || (int64_t)start + acc + 1 >= out_stride)) {
    if (lane == 0) raise_error(err, DFLASH_DERR_OUTPUT_ROW);
    return;
  }
  if (live) out_tokens[(int64_t)b * S + lane] = lane < acc ? d_next : (lane == acc ? bonus_id : 0);
  if (write_ids) {
    int *row = output_ids + (int64_t)b * out_stride + start;
    if (lane <= acc) row[lane] = d;
    if (lane == acc) row[acc + 1] = bonus_id;
  }
  if (lane == 0) {
    accept_len[b] = acc;
    commit_len[b] = acc + 1;
    bonus[b] = bonus_id;
    seq_len[b] = start + acc + 1;
  }
}

__global__ void __launch_bounds__(128) accept_kernel(
    int B, int S, int vocab, const int *__restrict__ draft, const int *__restrict__ post,
    int *seq_len, int *accept_len, int *commit_len, int *bonus, int *out_tokens,
    int *output_ids, int out_stride, unsigned int *err) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (b >= B) return;
  const bool live = lane < S;
  const int d = live ? draft[(int64_t)b * S + lane] : -1;
  const int p = live ? post[(int64_t)b * S + lane] : -1;
  const int d_next = __shfl_down_sync(0xffffffffu, d, 1);
  const unsigned int match = __ballot_sync(0xffffffffu, lane < S - 1 && d_next == p);
  const int acc = __ffs(~match) - 1;               // leading run of matches, <= S-1
  const int bonus_id = __shfl_sync(0xffffffffu, p, acc);
  // ids this row commits: draft[0..acc] and the bonus
  const bool bad_id = (lane <= acc && (d < 0 || d >= vocab)) || (lane == acc && (p < 0 || p >= vocab));
  if (__any_sync(0xffffffffu, bad_id)) {
    if (lane == 0) raise_error(err, DFLASH_DERR_TOKEN_RANGE);
    return;
  }
  commit_row(b, S, lane, acc, bonus_id, d, d_next, seq_len, accept_len, commit_len, bonus,
             out_tokens, output_ids, out_stride, err);
}

cudaError_t launch_accept(int B, int S, int vocab, const int *draft, const int *post, int *seq_len,
                          int *accept_len, int *commit_len, int *bonus, int *out_tokens,
                          int *output_ids, int out_stride, unsigned int *err, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  const int warps = 4;
  return launch_pdl(accept_kernel, dim3((B + warps - 1) / warps), dim3(warps * 32), 0, s, B, S,
                    vocab, draft, post, seq_len, accept_len, commit_len, bonus, out_tokens,
                    output_ids, out_stride, err);
}

// ---------------------------------------------------------------------------
// Lossless sampled verification with the greedy drafter ("Inside SGLang",
// "Sampling: preserve the proposal distribution the walk actually used"):
// draft[i+1] is accepted with probability min(1, p(y)/q(y)) = p(y), as q is
// the point mass of an argmax drafter, i.e. iff u[i] < p_i(y); at the first
// rejection the correction comes from the residual [p - q]+ = p with y's
// entry zeroed; after full acceptance the bonus comes from the target row of
// the last position.  The draw is an exponential race, argmax_v w(v) / e_v
// with e_v ~ Exp(1) given by the caller (lowest id on ties).
// ---------------------------------------------------------------------------
// Stop position of request b (accepted count) and the excluded id (-1 for
// none); false if the stop position's proposed id lies outside the
// vocabulary.  One warp, lane i decides block position i: every load is in
// flight at once and a ballot finds the first rejection (S <= 32).
// With a real proposal (cand/qr: the K candidates of every position and their
// probabilities) y is accepted iff q(y) > 0 and u < p(y) / q(y), q(y) the
// probability of the first candidate equal to y (0 if none).
__device__ __forceinline__ bool sampled_stop(int b, int S, int vocab, const int *draft,
                                             const float *probs, const float *u, int lane,
                                             int &acc, int &excl, const int *cand = nullptr,
                                             const float *qr = nullptr, int K = 0) {
  const bool live = lane < S - 1;
  const int y = live ? draft[(int64_t)b * S + lane + 1] : 0;
  const bool bad = live && (y < 0 || y >= vocab);
  const float py = (live && !bad) ? probs[((int64_t)b * S + lane) * vocab + y] : 0.f;
  const float uu = live ? u[(int64_t)b * (S - 1) + lane] : 1.f;
  bool take = live && !bad && uu < py;
  if (cand) {
    float qy = 0.f;
    if (live && !bad) {
      const int64_t o = ((int64_t)b * (S - 1) + lane) * K;
      for (int k = K - 1; k >= 0; --k)   // the first match wins
        if (cand[o + k] == y) qy = qr[o + k];
    }
    take = live && !bad && qy > 0.f && uu < py / qy;
  }
  const unsigned int taken = __ballot_sync(0xffffffffu, take);
  acc = __ffs(~taken) - 1;   // first position not accepted, <= S-1
  const int ystop = __shfl_sync(0xffffffffu, y, acc);
  const bool bad_stop = __shfl_sync(0xffffffffu, bad ? 1 : 0, acc) != 0;
  excl = acc < S - 1 ? ystop : -1;
  return !(acc < S - 1 && bad_stop);
}

// grid (blocks per request, B): each CTA races a slice of the vocabulary of
// request b's stop row and folds its winner into keys[b]; the last CTA of the
// request (ticket) commits it and clears keys[b] and the ticket.
// QMODE: the proposal is a real distribution over K candidates per position
// (cand/qr); the residual at a rejection is [p - q]+ on those candidates.
constexpr int kMaxQ = 8;
template <bool QMODE>
__global__ void __launch_bounds__(256) sampled_race_kernel(
    int S, int vocab, const int *__restrict__ draft, const float *__restrict__ probs,
    const float *__restrict__ u, const float *__restrict__ noise, unsigned long long *keys,
    int *tickets, int *seq_len, int *accept_len, int *commit_len, int *bonus, int *out_tokens,
    int *output_ids, int out_stride, unsigned int *err, const int *__restrict__ cand,
    const float *__restrict__ qr, int K) {
  pdl_wait();
  __shared__ int s_acc, s_excl, s_ok, s_last;
  __shared__ unsigned long long s_best[8];
  __shared__ int s_cid[kMaxQ];
  __shared__ float s_q[kMaxQ];
  const int b = blockIdx.y;
  if (threadIdx.x < 32) {
    int acc, excl;
    const bool ok = QMODE ? sampled_stop(b, S, vocab, draft, probs, u, threadIdx.x, acc, excl,
                                         cand, qr, K)
                          : sampled_stop(b, S, vocab, draft, probs, u, threadIdx.x, acc, excl);
    if (QMODE && threadIdx.x < kMaxQ) {
      // the stop position's candidates; none after full acceptance
      const bool have = acc < S - 1 && (int)threadIdx.x < K;
      const int64_t o = ((int64_t)b * (S - 1) + (have ? acc : 0)) * K + threadIdx.x;
      s_cid[threadIdx.x] = have ? cand[o] : -1;
      s_q[threadIdx.x] = have ? qr[o] : 0.f;
    }
    if (threadIdx.x == 0) {
      s_ok = ok;
      s_acc = acc;
      s_excl = QMODE ? -1 : excl;
    }
  }
  __syncthreads();
  const float *row = probs + ((int64_t)b * S + s_acc) * vocab;
  const float *e = noise + (int64_t)b * vocab;
  unsigned long long best = 0ull;
  const int excl = s_excl;
  const int stride = gridDim.x * blockDim.x;
  // [p - q]+ on the candidates (QMODE); p elsewhere
  auto resid = [&](int v, float w) {
    if (QMODE) {
#pragma unroll
      for (int k = 0; k < kMaxQ; ++k)
        if (v == s_cid[k]) w = fmaxf(w - s_q[k], 0.f);
    }
    return w;
  };
  if ((vocab & 3) == 0 && ((uintptr_t)row & 15) == 0 && ((uintptr_t)e & 15) == 0) {
    // four entries per load (16-byte loads of the row and the noise)
#pragma unroll 2
    for (int v = 4 * (blockIdx.x * blockDim.x + threadIdx.x); v < vocab; v += 4 * stride) {
      const float4 w4 = *reinterpret_cast<const float4 *>(row + v);
      const float4 e4 = *reinterpret_cast<const float4 *>(e + v);
      const float w[4] = {w4.x, w4.y, w4.z, w4.w}, en[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned long long k =
            argmax_key((v + j == excl ? 0.f : resid(v + j, w[j])) / en[j], v + j);
        best = k > best ? k : best;
      }
    }
  } else {
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < vocab; v += stride) {
      const float w = v == excl ? 0.f : resid(v, row[v]);
      const unsigned long long k = argmax_key(w / e[v], v);
      best = k > best ? k : best;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
    best = other > best ? other : best;
  }
  if ((threadIdx.x & 31) == 0) s_best[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) best = s_best[i] > best ? s_best[i] : best;
    if (s_ok && best) atomicMax(keys + b, best);
    // the last CTA of the request commits it
    __threadfence();
    s_last = atomicAdd(tickets + b, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x >= 32) return;
  __threadfence();
  const int lane = threadIdx.x;
  const bool live = lane < S;
  const int d = live ? draft[(int64_t)b * S + lane] : -1;
  const int d_next = __shfl_down_sync(0xffffffffu, d, 1);
  const int acc = s_acc;
  const unsigned long long k = __ldcg(keys + b);
  const bool bad = !s_ok || k == 0ull || __any_sync(0xffffffffu, lane <= acc && (d < 0 || d >= vocab));
  if (lane == 0) {
    keys[b] = 0ull;     // ready for the next call
    tickets[b] = 0;
  }
  if (bad) {
    if (lane == 0) raise_error(err, DFLASH_DERR_TOKEN_RANGE);
    return;
  }
  commit_row(b, S, lane, acc, argmax_key_index(k), d, d_next, seq_len, accept_len, commit_len,
             bonus, out_tokens, output_ids, out_stride, err);
}

cudaError_t launch_accept_sampled(int B, int S, int vocab, const int *draft, const float *probs,
                                  const float *u, const float *noise, unsigned long long *keys,
                                  int *tickets, int *seq_len, int *accept_len, int *commit_len,
                                  int *bonus, int *out_tokens, int *output_ids, int out_stride,
                                  unsigned int *err, cudaStream_t s, int sms, const int *cand,
                                  const float *qr, int K) {
  if (B <= 0) return cudaSuccess;
  if (S > 32 || (cand && (K < 1 || K > kMaxQ || !qr))) return cudaErrorInvalidValue;
  // about two waves of 256-thread CTAs over all requests' rows, each thread
  // taking at least four entries per pass
  int per = (2 * sms * 4 + B - 1) / B;
  per = per < 1 ? 1 : per;
  const int need = (vocab + 1023) / 1024;
  per = per > need ? need : per;
  if (cand)
    return launch_pdl(sampled_race_kernel<true>, dim3(per, B), dim3(256), 0, s, S, vocab, draft,
                      probs, u, noise, keys, tickets, seq_len, accept_len, commit_len, bonus,
                      out_tokens, output_ids, out_stride, err, cand, qr, K);
  return launch_pdl(sampled_race_kernel<false>, dim3(per, B), dim3(256), 0, s, S, vocab, draft,
                    probs, u, noise, keys, tickets, seq_len, accept_len, commit_len, bonus,
                    out_tokens, output_ids, out_stride, err, (const int *)nullptr,
                    (const float *)nullptr, 0);
}

}  // namespace dflash
