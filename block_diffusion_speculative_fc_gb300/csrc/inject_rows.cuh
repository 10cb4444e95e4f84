// Injection bookkeeping shared by the standalone kernels (small_ops.cu) and
// the fused injection launch (gemm_tc.cu).
//   Row map ("Inside SGLang", Step 7: prefix-valid writes): feature row r
//   belongs to the request b with row_offset[b] <= r < row_offset[b] +
//   n_rows[b]; its position is kv_len[b] + (r - row_offset[b]) and its cache
//   row is page_table[b][pos / page] * page + pos % page.  Rows owned by no
//   request, or failing a capacity / page-range / position check, get slot -1.
//   With a draft window W ("Inside SGLang", worker/memory section: the draft's
//   private compact mapping), the page table is a ring: the cache row of pos
//   is page_table[b][(pos / page) % pages_per_req] * page + pos % page, there
//   is no capacity limit, and a row older than the newest W rows the request
//   will have after this call (pos < kv_len[b] + n_rows[b] - W) is skipped
//   (slot -1, no error): the ring slot it would take belongs to a newer row.
//   Length update: kv_len[b] += n_rows[b], not past what was written.
#pragma once
#include "common.cuh"

namespace dflash {

struct InjectArgs {
  int B;
  const int *row_offset, *n_rows;   // [B]
  int *kv_len;                      // [B]
  const int *page_table;            // [B, pages_per_req]
  int pages_per_req, n_pages, page_size, max_position;
  int draft_window;                 // 0: off; W > 0: ring of pages_per_req pages
};

// Cache slot and position of feature row r (len(b) read through `len_of`).
template <class LenOf, class OffOf, class NOf>
__device__ __forceinline__ void inject_map_row(const InjectArgs &a, int r, LenOf len_of, OffOf off_of,
                                               NOf n_of, int &slot, int &pos, unsigned int *err) {
  slot = -1;
  pos = 0;
  for (int b = 0; b < a.B; ++b) {
    const int i = r - off_of(b);
    if (i < 0 || i >= n_of(b)) continue;
    pos = len_of(b) + i;
    const bool ring = a.draft_window > 0;
    const int64_t cap = (int64_t)a.pages_per_req * a.page_size;
    if ((!ring && pos >= cap) || pos < 0) {
      raise_error(err, DFLASH_DERR_KV_CAPACITY);
    } else if (pos >= a.max_position) {
      raise_error(err, DFLASH_DERR_POSITION);
    } else if (ring && (int64_t)pos < (int64_t)len_of(b) + n_of(b) - a.draft_window) {
      // out of the window before the call ends: nothing to write
    } else {
      const int lp = pos / a.page_size;
      const int page = a.page_table[(int64_t)b * a.pages_per_req + (ring ? lp % a.pages_per_req : lp)];
      if (page < 0 || page >= a.n_pages)
        raise_error(err, DFLASH_DERR_PAGE_RANGE);
      else
        slot = page * a.page_size + pos % a.page_size;
    }
    break;
  }
  if (slot < 0) pos = 0;
}

// kv_len[b] += n_rows[b]; a request whose rows do not lie inside the feature
// buffers is flagged and keeps its length.
__device__ __forceinline__ void inject_advance(const InjectArgs &a, int b, int total_rows,
                                               int64_t capacity, unsigned int *err) {
  const int n = a.n_rows[b], off = a.row_offset[b];
  if (n <= 0) {
    if (n < 0) raise_error(err, DFLASH_DERR_ROW_RANGE);
    return;
  }
  if (off < 0 || (int64_t)off + n > total_rows) {
    raise_error(err, DFLASH_DERR_ROW_RANGE);
    return;
  }
  const int64_t v = (int64_t)a.kv_len[b] + n;
  a.kv_len[b] = (int)(v > capacity ? capacity : v);
}

}  // namespace dflash
