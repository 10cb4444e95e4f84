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

cudaError_t launch_accept(int B, int S, int vocab, const int *draft, const int *post, int *seq_len,
                          int *accept_len, int *commit_len, int *bonus, int *out_tokens,
                          int *output_ids, int out_stride, unsigned int *err, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  const int warps = 4;
  return launch_pdl(accept_kernel, dim3((B + warps - 1) / warps), dim3(warps * 32), 0, s, B, S,
                    vocab, draft, post, seq_len, accept_len, commit_len, bonus, out_tokens,
                    output_ids, out_stride, err);
}

}  // namespace dflash
