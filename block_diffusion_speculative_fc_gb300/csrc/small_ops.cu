// Row-wise kernels around the GEMMs: block embedding, RMSNorm, argmax
// finalisation, injection row mapping and the RoPE table.
#include <algorithm>

#include "common.cuh"
#include "inject_rows.cuh"
#include "kernels.h"

namespace dflash {

// ---------------------------------------------------------------------------
// Block embedding ("Inside SGLang", Step 3: input id = anchor at j = 0, else
// mask_token_id; logical position = prefix length + j).  Writes the fp32
// residual stream, the RoPE position of every block row and clears the
// argmax keys of the lm_head pass.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void embed_kernel(const T *__restrict__ embed, const int *__restrict__ anchor,
                             const int *__restrict__ kv_len, int S, int H, int vocab, int mask_id,
                             int max_position, float *__restrict__ x, const T *__restrict__ gain,
                             T *__restrict__ xg, float *__restrict__ ssq, int ssq_ld,
                             int *__restrict__ row_pos, unsigned long long *__restrict__ keys,
                             unsigned int *err) {
  // one CTA of 256 threads per block row; also the deferred RMSNorm of the
  // first layer's input (x * g and per-128-feature sums of squares)
  pdl_wait();
  __shared__ float s_ws[64][4];
  const int m = blockIdx.x;
  const int b = m / S, j = m % S;
  int id = j == 0 ? anchor[b] : mask_id;
  const bool bad_id = id < 0 || id >= vocab;
  const int pos = kv_len[b] + j;
  const bool bad_pos = pos < 0 || pos >= max_position;
  if (threadIdx.x == 0) {
    if (bad_id) raise_error(err, DFLASH_DERR_TOKEN_RANGE);
    if (bad_pos) raise_error(err, DFLASH_DERR_POSITION);
    row_pos[m] = bad_pos ? 0 : pos;
    keys[m] = 0ull;
  }
  const T *src = embed + (int64_t)(bad_id ? 0 : id) * H;
  const int warp = threadIdx.x >> 5;
  // every load of the row is issued before any use (H <= 64 * 128 = 32 x 256)
  constexpr int MAXV = 32;
  float v[MAXV], gv[MAXV];
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int c = k * blockDim.x + threadIdx.x;
    v[k] = (c < H && !bad_id) ? to_f32(src[c]) : 0.f;
    gv[k] = c < H ? to_f32(gain[c]) : 0.f;
  }
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int c = k * blockDim.x + threadIdx.x;   // H is a multiple of 128: a warp stays in one part
    if (k * (int)blockDim.x >= H) break;
    if (c < H) {
      x[(int64_t)m * H + c] = v[k];
      xg[(int64_t)m * H + c] = from_f32<T>(v[k] * gv[k]);
    }
    const float t = warp_sum(v[k] * v[k]);
    if ((threadIdx.x & 31) == 0 && c < H) s_ws[c >> 7][warp & 3] = t;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < (H >> 7); q += blockDim.x)
    ssq[(int64_t)q * ssq_ld + m] = ((s_ws[q][0] + s_ws[q][1]) + s_ws[q][2]) + s_ws[q][3];
}

cudaError_t launch_embed(int store, const void *embed, const int *anchor, const int *kv_len, int B,
                         int S, int H, int vocab, int mask_id, int max_position, float *x,
                         const void *norm_gain, void *xg, float *ssq, int ssq_ld, int *row_pos,
                         unsigned long long *keys, unsigned int *err, cudaStream_t s) {
  const int M = B * S;
  if (M <= 0) return cudaSuccess;
  if (H % 128 || H > 64 * 128) return cudaErrorInvalidValue;
  if (store == ST_F32)
    return launch_pdl(embed_kernel<float>, dim3(M), dim3(256), 0, s, (const float *)embed, anchor,
                      kv_len, S, H, vocab, mask_id, max_position, x, (const float *)norm_gain,
                      (float *)xg, ssq, ssq_ld, row_pos, keys, err);
  return launch_pdl(embed_kernel<bf16>, dim3(M), dim3(256), 0, s, (const bf16 *)embed, anchor,
                    kv_len, S, H, vocab, mask_id, max_position, x, (const bf16 *)norm_gain,
                    (bf16 *)xg, ssq, ssq_ld, row_pos, keys, err);
}

// ---------------------------------------------------------------------------
// RMSNorm y = x / sqrt(mean(x^2) + eps) * g, one CTA per row, fp32 math.
// out2 (optional) receives a second copy (the hidden_out of the draft pass).
// ---------------------------------------------------------------------------
template <typename Tin, typename Tout>
__global__ void rmsnorm_kernel(const Tin *__restrict__ x, const Tout *__restrict__ g, int H,
                               float eps, Tout *__restrict__ out, Tout *__restrict__ out2) {
  // one CTA per row; each thread keeps up to 32 values in registers so the
  // row is read once with all loads in flight
  constexpr int MAXV = 32;
  pdl_wait();
  const int m = blockIdx.x;
  const Tin *row = x + (int64_t)m * H;
  float v[MAXV];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    v[k] = c < H ? to_f32(row[c]) : 0.f;
    ss += v[k] * v[k];
  }
  __shared__ float red[32];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    t = warp_sum(t);
    if (threadIdx.x == 0) red[0] = t;
  }
  __syncthreads();
  const float r = rsqrtf(red[0] / (float)H + eps);
  Tout *o = out + (int64_t)m * H;
  Tout *o2 = out2 ? out2 + (int64_t)m * H : nullptr;
#pragma unroll
  for (int k = 0; k < MAXV; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    if (c >= H) continue;
    const Tout y = from_f32<Tout>(v[k] * r * to_f32(g[c]));
    o[c] = y;
    if (o2) o2[c] = y;
  }
  __syncthreads();
  pdl_trigger();
}

cudaError_t launch_rmsnorm(int in_f32, int store, const void *x, const void *gain, int M, int H,
                           float eps, void *out, void *out2, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  const int thr = H <= 8192 ? 256 : 1024;   // rows up to 32 values per thread
  if (H > 32 * thr) return cudaErrorInvalidValue;
  if (!in_f32) return cudaErrorInvalidValue;
  if (store == ST_F32)
    return launch_pdl(rmsnorm_kernel<float, float>, dim3(M), dim3(thr), 0, s, (const float *)x,
                      (const float *)gain, H, eps, (float *)out, (float *)out2);
  return launch_pdl(rmsnorm_kernel<float, bf16>, dim3(M), dim3(thr), 0, s, (const float *)x,
                    (const bf16 *)gain, H, eps, (bf16 *)out, (bf16 *)out2);
}

// ---------------------------------------------------------------------------
// draft_ids[b, 0] = anchor, draft_ids[b, j] = argmax of block row j (j >= 1).
// ---------------------------------------------------------------------------
__global__ void argmax_finalize_kernel(const unsigned long long *__restrict__ keys,
                                       const int *__restrict__ anchor, int M, int S,
                                       int *__restrict__ draft_ids) {
  pdl_wait();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  const int j = m % S;
  draft_ids[m] = j == 0 ? anchor[m / S] : argmax_key_index(keys[m]);
}

cudaError_t launch_argmax_finalize(const unsigned long long *keys, const int *anchor, int B, int S,
                                   int *draft_ids, cudaStream_t s) {
  const int M = B * S;
  if (M <= 0) return cudaSuccess;
  return launch_pdl(argmax_finalize_kernel, dim3((M + 127) / 128), dim3(128), 0, s, keys, anchor, M,
                    S, draft_ids);
}

// ---------------------------------------------------------------------------
// Injection row map of the feature rows row0 .. row0+rows-1 of one chunk
// (inject_rows.cuh states the map); request data staged in shared memory.
// ---------------------------------------------------------------------------
__global__ void inject_prep_kernel(int B, int row0, int rows, const int *__restrict__ row_offset,
                                   const int *__restrict__ n_rows, const int *__restrict__ kv_len,
                                   const int *__restrict__ page_table, int pages_per_req,
                                   int n_pages, int page_size, int max_position, int draft_window,
                                   int *__restrict__ row_slot, int *__restrict__ row_pos,
                                   unsigned int *err) {
  pdl_wait();
  extern __shared__ int sm[];
  int *s_off = sm, *s_n = sm + B, *s_len = sm + 2 * B;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    s_off[b] = row_offset[b];
    s_n[b] = n_rows[b];
    s_len[b] = kv_len[b];
  }
  __syncthreads();
  const int local = blockIdx.x * blockDim.x + threadIdx.x;
  if (local >= rows) return;
  InjectArgs a;
  a.B = B;
  a.page_table = page_table;
  a.pages_per_req = pages_per_req;
  a.n_pages = n_pages;
  a.page_size = page_size;
  a.max_position = max_position;
  a.draft_window = draft_window;
  int slot, pos;
  inject_map_row(a, row0 + local, [&](int b) { return s_len[b]; }, [&](int b) { return s_off[b]; },
                 [&](int b) { return s_n[b]; }, slot, pos, err);
  row_slot[local] = slot;
  row_pos[local] = pos;
}

cudaError_t launch_inject_prep(int B, int row0, int rows, const int *row_offset, const int *n_rows,
                               const int *kv_len, const int *page_table, int pages_per_req,
                               int n_pages, int page_size, int max_position, int draft_window,
                               int *row_slot, int *row_pos, unsigned int *err, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int thr = 256;
  return launch_pdl(inject_prep_kernel, dim3((rows + thr - 1) / thr), dim3(thr),
                    3 * B * sizeof(int), s, B, row0, rows, row_offset, n_rows, kv_len, page_table,
                    pages_per_req, n_pages, page_size, max_position, draft_window, row_slot,
                    row_pos, err);
}

// kv_len[b] += n_rows[b] (inject_rows.cuh).
__global__ void inject_finalize_kernel(int B, int total_rows, const int *__restrict__ row_offset,
                                       const int *__restrict__ n_rows, int *kv_len, int capacity,
                                       unsigned int *err) {
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  InjectArgs a;
  a.B = B;
  a.row_offset = row_offset;
  a.n_rows = n_rows;
  a.kv_len = kv_len;
  inject_advance(a, b, total_rows, capacity, err);
}

cudaError_t launch_inject_finalize(int B, int total_rows, const int *row_offset, const int *n_rows,
                                   int *kv_len, int capacity, unsigned int *err, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(inject_finalize_kernel, dim3((B + 127) / 128), dim3(128), 0, s, B, total_rows,
                    row_offset, n_rows, kv_len, capacity, err);
}

// Prefix-valid compaction ("Inside SGLang", Step 7: of a verify block only
// the accepted rows reach the draft cache).  Every block scans the (few)
// requests itself in shared memory; then compact row r of request b (the
// last request whose compact offset is <= r) is copied from feature row
// row_offset[b] + r - coff[b] of each of the n_sel buffers, 16 bytes per
// thread and step.  A request with negative n_rows, or rows outside
// [0, total_rows), keeps none (flagged, as the length update would).
// Requests may share feature rows; the compact rows never exceed
// total_rows (the operand's size): rows past it are dropped from the last
// requests and flagged.
__global__ void inject_compact_kernel(int B, int total_rows, FeatPtrs src, int n_sel, int th,
                                      const int *__restrict__ row_offset,
                                      const int *__restrict__ n_rows, bf16 *__restrict__ x,
                                      int *__restrict__ coff, int *__restrict__ crows,
                                      int *__restrict__ count, unsigned int *err) {
  pdl_wait();
  extern __shared__ int sm[];
  int *s_off = sm, *s_n = sm + B, *s_c = sm + 2 * B;   // s_c: B + 1 entries
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int n = n_rows[b], off = row_offset[b];
    const bool inside = off >= 0 && (int64_t)off + n <= (int64_t)total_rows;
    const bool keep = n > 0 && inside;
    if (blockIdx.x == 0 && (n < 0 || (n > 0 && !inside))) raise_error(err, DFLASH_DERR_ROW_RANGE);
    s_off[b] = off;
    s_n[b] = keep ? n : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    bool trimmed = false;
    for (int b = 0; b < B; ++b) {
      s_c[b] = acc;
      const int keep = min(s_n[b], total_rows - acc);
      trimmed |= keep < s_n[b];
      s_n[b] = keep;
      acc += keep;
    }
    s_c[B] = acc;
    if (trimmed && blockIdx.x == 0) raise_error(err, DFLASH_DERR_ROW_RANGE);
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      coff[b] = s_c[b];
      crows[b] = s_n[b];
    }
    if (threadIdx.x == 0) *count = s_c[B];
  }
  const int total = s_c[B];
  const int vecs = th >> 3;   // 16-byte vectors per source row
  for (int r = blockIdx.x; r < total; r += gridDim.x) {
    int lo = 0, hi = B - 1;   // last b with s_c[b] <= r (it has s_n[b] > 0)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_c[mid] <= r) lo = mid;
      else hi = mid - 1;
    }
    const int64_t row = (int64_t)s_off[lo] + (r - s_c[lo]);
    uint4 *dst = reinterpret_cast<uint4 *>(x + (int64_t)r * n_sel * th);
    // the row's n_sel * vecs vectors, U per thread in flight at a time (all
    // loads of a batch issued before its stores)
    constexpr int U = 8;
    const int total = n_sel * vecs, step = blockDim.x * U;
    for (int v0 = threadIdx.x; v0 < total; v0 += step) {
      uint4 t[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * blockDim.x;
        if (v < total) {
          const int j = v / vecs;
          t[u] = __ldg(reinterpret_cast<const uint4 *>((const bf16 *)src.p[j] + row * th) + (v - j * vecs));
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * blockDim.x;
        if (v < total) dst[v] = t[u];
      }
    }
  }
}

cudaError_t launch_inject_compact(int B, int total_rows, const FeatPtrs &src, int n_sel, int th,
                                  const int *row_offset, const int *n_rows, void *x, int *coff,
                                  int *crows, int *count, unsigned int *err, cudaStream_t s) {
  if (B <= 0 || n_sel <= 0 || n_sel > kMaxSrc || th % 8) return cudaErrorInvalidValue;
  const int grid = std::max(1, std::min(std::max(total_rows, 1), 2 * gemm_tc_num_sms()));
  const size_t smem = sizeof(int) * (3 * (size_t)B + 1);
  return launch_pdl(inject_compact_kernel, dim3(grid), dim3(256), smem, s, B, total_rows, src, n_sel,
                    th, row_offset, n_rows, (bf16 *)x, coff, crows, count, err);
}

// ---------------------------------------------------------------------------
// RoPE table (cos, sin) of angle p * theta^(-2i/D), i < D/2, for every
// position p < max_position.  Angles are formed and reduced in double
// precision so that large positions keep full fp32 accuracy.
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float2 *table, int max_position, int half, double theta) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)max_position * half) return;
  const int p = (int)(idx / half), i = (int)(idx % half);
  const double freq = pow(theta, -2.0 * (double)i / (double)(2 * half));
  double sn, cs;
  sincos((double)p * freq, &sn, &cs);
  table[idx] = make_float2((float)cs, (float)sn);
}

cudaError_t launch_rope_table(float2 *table, int max_position, int head_dim, float theta,
                              cudaStream_t s) {
  const int half = head_dim / 2;
  const int64_t n = (int64_t)max_position * half;
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(table, max_position, half,
                                                                (double)theta);
  return cudaGetLastError();
}

}  // namespace dflash
