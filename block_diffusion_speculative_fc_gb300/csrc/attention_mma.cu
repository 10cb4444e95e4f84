// bf16 block attention on the tensor cores, paged KV staged by TMA.
//
// Non-causal attention of the S block queries over [committed context ; the S
// block keys] ("Inside SGLang: DFlash and DFlash 2 Implementation", Step 4:
// two K/V sources inside draft attention; CSDN DFlash article, "draft model
// predict", is_causal=False), with the optional sliding window of the
// Kimi-K2.6 draft card (a context key at pk is visible to a query at pq iff
// pq - pk < W).
//
// Work split (flash-decoding): every (request b, KV head g) owns the R = G*S
// query rows of its query-head group.  Its context pages are cut into splits of
// `pps` pages; the last split also takes the S block keys.  A prep kernel
// sizes the splits from the device-side kv_len so that the whole batch makes
// about one work item per resident CTA, and a persistent kernel walks the item list.
// Per item: one 64-key tile at a time (one KV page of one head: two TMA boxes
// of 64 rows x 64 dims for K and two for V, 128-byte swizzle, 2-stage ring),
// S = Q K^T and O += P V with mma.sync m16n8k16 (bf16 in, fp32 accumulate),
// online softmax in registers with quad shuffles.  A split that is not alone
// writes (O, m, l) to scratch; the last split of a (b, g) to finish (atomic
// ticket) merges the splits in split order and writes the output.
// FP8 cache (CSDN article, Kimi-K2.6 draft card: one byte per K/V element):
// a context tile is one 8 KB box of E4M3 codes per tensor; all threads widen
// it into a 16-bit staging tile before the MMAs: every E4M3 value is exact
// in f16 (the hardware conversion, two codes per instruction), so the MMAs
// run in f16 (Q rounded to f16 once per item) and k_scale / v_scale fold
// into the softmax scale and into P.  The S block keys stay bf16 (16-row
// boxes), converted to f16 in the staging tile.
// Draft KV windowing: the page table is a ring (page of logical page lp is
// page_table[b][lp % pages_per_req]) and keys below kv_len - W are hidden.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dflash {
namespace att {

constexpr int KT = 64;          // keys per tile (one page)
constexpr int STAGES = 2;       // 2 x 32 KB: three CTAs of <= 128 threads fit on an SM
constexpr int TILE_BYTES = KT * 128 * 2;   // K (or V) tile: 64 keys x 128 dims
constexpr int STAGE_BYTES = 2 * TILE_BYTES;
constexpr int MAX_SPLITS = 16;  // splits of one (request, KV head) at most
constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 64 + (MAX_SPLITS + 1) * 128 * 4;
// FP8 layout: STAGES stages of [K codes 8 KB | V codes 8 KB], the 16-bit
// staging tile [K 16 KB | V 16 KB], the block keys [K 4 KB | V 4 KB] (16 rows
// of bf16), then the barriers; the split-merge weights reuse the staging tile.
constexpr int F8_TILE = KT * 128;
constexpr int F8_STAGE = 2 * F8_TILE;
constexpr int F8_STAGING = STAGES * F8_STAGE;
constexpr int F8_BLOCK = F8_STAGING + STAGE_BYTES;
constexpr int F8_BLK_ROWS = 16;
constexpr int F8_BARS = F8_BLOCK + 2 * F8_BLK_ROWS * 256;
constexpr int SMEM_F8 = 1024 + F8_BARS + 64;
static_assert(SMEM_F8 <= SMEM, "the FP8 layout fits the bf16 kernel's shared memory");
static_assert((MAX_SPLITS + 1) * 128 * 4 <= STAGE_BYTES, "merge weights fit the staging tile");
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr int kMaxCluster = 16;  // CTAs per (request, KV head) in the cluster kernel

struct Params {
  CUtensorMap tmK, tmV;          // cache: dims {D, KVH, n_pages*64}, box {64, 1, 64}
  CUtensorMap tmKb, tmVb;        // block keys: dims {D, KVH, B*S}, box {64, 1, 64}
  const bf16 *q;                 // [B*S, n_heads, D]
  bf16 *out;                     // [B*S, n_heads, D]
  const int *page_table;
  const int *kv_len;
  const int *item_start;         // [B*KVH + 1] prefix of splits per (b, g)
  const int *pps_ptr;            // pages per split (device scalar)
  float *part_o;                 // [max_items][R][D]
  float2 *part_ml;               // [max_items][R]
  int *tickets;                  // [B*KVH]
  unsigned int *err;
  int B, S, n_heads, kvh, pages_per_req, n_pages, window, R, max_items;
  float scale_log2;              // log2(e) / sqrt(D)
  int draft_window;              // 0 = off; W > 0: ring page table, keys below kv_len - W hidden
  float k_mul, v_mul;            // FP8: k_scale, v_scale
};

// First visible context position of query row j (of a request with kv
// committed rows): the draft window's bound and, on a sliding layer, the
// layer's own window (pq - pk < W).
__device__ __forceinline__ int first_visible(const Params &p, int kv, int j) {
  const int lw = p.draft_window > 0 ? max(0, kv - p.draft_window) : 0;
  return p.window > 0 ? max(lw, kv + j - p.window + 1) : lw;
}
// Cache page of logical page lp of request b.
__device__ __forceinline__ int page_of(const Params &p, int b, int lp) {
  return p.page_table[(size_t)b * p.pages_per_req + (p.draft_window > 0 ? lp % p.pages_per_req : lp)];
}
// kv_len clamped to the page table's capacity (no limit for a ring).
__device__ __forceinline__ int clamp_kv(const Params &p, int kv) {
  const int cap = p.pages_per_req * KT;
  return kv < 0 ? 0 : (p.draft_window == 0 && kv > cap ? cap : kv);
}

__device__ __forceinline__ uint32_t su32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try(b, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}
__device__ __forceinline__ void tma3(void *dst, const CUtensorMap *tm, uint64_t *bar, int x, int y,
                                     int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void mma16816_f16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Two E4M3 codes (bytes 0, 1 of w, or bytes 2, 3 with hi) as the f16 pair
// of their values (exact: every E4M3 value is an f16), lower byte in the
// lower half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w, bool hi) {
  const uint16_t pair = (uint16_t)(hi ? (w >> 16) : (w & 0xFFFFu));
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
  return r;
}
// bf16 pair -> f16 pair (round to nearest)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
  return pack_f16(f.x, f.y);
}
// Byte address of (row, 16-byte chunk c) in a tile of rows of 128 bytes with
// the 128-byte swizzle TMA applies (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int c) {
  return base + row * 128 + (((c ^ row) & 7) << 4);
}

// ---------------------------------------------------------------- work list
// Visible context range of a request with kv rows: [lo, kv), lo from the
// draft window and the layer window (the earliest query of the block sees
// the most); its pages.
__device__ __forceinline__ int visible_lo(int kv, int window, int draft_window) {
  const int lw = draft_window > 0 ? max(0, kv - draft_window) : 0;
  return window > 0 ? max(lw, kv - window + 1) : lw;
}

__global__ void attn_prep_kernel(const int *__restrict__ kv_len, int B, int kvh, int cap,
                                 int window, int draft_window, int target_items, int max_items,
                                 int *item_start, int *pps_out, unsigned int *err) {
  pdl_wait();
  __shared__ int s_total;
  if (threadIdx.x == 0) s_total = 0;
  __syncthreads();
  int local = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int kv = kv_len[b];
    kv = kv < 0 ? 0 : (kv > cap ? cap : kv);
    const int lo = visible_lo(kv, window, draft_window);
    const int pages = kv > lo ? (kv - 1) / KT - lo / KT + 1 : 0;
    local += pages;
  }
  atomicAdd(&s_total, local * kvh);
  __shared__ int s_maxpages;
  if (threadIdx.x == 0) s_maxpages = 0;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int kv = kv_len[b];
    kv = kv < 0 ? 0 : (kv > cap ? cap : kv);
    const int lo = visible_lo(kv, window, draft_window);
    atomicMax(&s_maxpages, kv > lo ? (kv - 1) / KT - lo / KT + 1 : 0);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int total = s_total;
    // about one item per resident CTA, at least two pages per split, at most MAX_SPLITS
    // splits per (request, head), and never more items than the scratch holds
    int pps = max(2, (total + target_items - 1) / target_items);
    while (B * kvh + total / pps + 1 > max_items) ++pps;
    pps = max(pps, (s_maxpages + MAX_SPLITS - 1) / MAX_SPLITS);
    *pps_out = pps;
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      int kv = kv_len[b];
      if (kv < 0 || kv > cap) raise_error(err, DFLASH_DERR_KV_CAPACITY);
      kv = kv < 0 ? 0 : (kv > cap ? cap : kv);
      const int lo = visible_lo(kv, window, draft_window);
      const int pages = kv > lo ? (kv - 1) / KT - lo / KT + 1 : 0;
      const int nsplit = max(1, (pages + pps - 1) / pps);
      for (int g = 0; g < kvh; ++g) {
        item_start[b * kvh + g] = acc;
        acc += nsplit;
      }
    }
    item_start[B * kvh] = acc;
  }
}

// Attention of the R query rows of (request b, KV head g) over context pages
// [pg0, pg1) of its visible range (first_page = first visible page) and, when
// has_block, the S block keys.  Leaves the unnormalised output, row maxima and
// row sums (already summed over the quad) in `a`.  `use` counts stage uses of
// the CTA's ring across calls.  All threads of the CTA take part.
struct Acc {
  float o[16][4];
  float m0, m1, l0, l1;
};

// One 64-key tile into ring stage u: context page `lp` of request b, head g
// (its cache page looked up in the page table), or the S block keys.  FP8:
// a context tile is one box of codes per tensor; the block keys go to their
// own 16-row region (barrier full[STAGES]) and are issued by issue_block.
template <bool FP8>
__device__ __forceinline__ void issue_tile(const Params &p, uint8_t *smem, uint64_t *full,
                                           uint32_t u, int b, int g, int lp, bool block) {
  uint64_t *bar = &full[u % STAGES];
  if (FP8) {
    uint8_t *st = smem + (u % STAGES) * F8_STAGE;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)),
                 "r"(F8_STAGE)
                 : "memory");
    int page = page_of(p, b, lp);
    if (page < 0 || page >= p.n_pages) {
      raise_error(p.err, DFLASH_DERR_PAGE_RANGE);
      page = 0;
    }
    tma3(st, &p.tmK, bar, 0, g, page * KT);
    tma3(st + F8_TILE, &p.tmV, bar, 0, g, page * KT);
    return;
  }
  uint8_t *st = smem + (u % STAGES) * STAGE_BYTES;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)),
               "r"(STAGE_BYTES)
               : "memory");
  if (!block) {
    int page = page_of(p, b, lp);
    if (page < 0 || page >= p.n_pages) {
      raise_error(p.err, DFLASH_DERR_PAGE_RANGE);
      page = 0;
    }
    tma3(st, &p.tmK, bar, 0, g, page * KT);
    tma3(st + TILE_BYTES / 2, &p.tmK, bar, 64, g, page * KT);
    tma3(st + TILE_BYTES, &p.tmV, bar, 0, g, page * KT);
    tma3(st + TILE_BYTES + TILE_BYTES / 2, &p.tmV, bar, 64, g, page * KT);
  } else {
    tma3(st, &p.tmKb, bar, 0, g, b * p.S);
    tma3(st + TILE_BYTES / 2, &p.tmKb, bar, 64, g, b * p.S);
    tma3(st + TILE_BYTES, &p.tmVb, bar, 0, g, b * p.S);
    tma3(st + TILE_BYTES + TILE_BYTES / 2, &p.tmVb, bar, 64, g, b * p.S);
  }
}
// FP8 layout: the S block keys of (b, g) as bf16, 16 rows per box.
__device__ __forceinline__ void issue_block_f8(const Params &p, uint8_t *smem, uint64_t *full, int b,
                                               int g) {
  uint64_t *bar = &full[STAGES];
  uint8_t *st = smem + F8_BLOCK;
  constexpr int BOX = F8_BLK_ROWS * 128;   // 16 rows x 64 dims of bf16
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)),
               "r"(4 * BOX)
               : "memory");
  tma3(st, &p.tmKb, bar, 0, g, b * p.S);
  tma3(st + BOX, &p.tmKb, bar, 64, g, b * p.S);
  tma3(st + 2 * BOX, &p.tmVb, bar, 0, g, b * p.S);
  tma3(st + 3 * BOX, &p.tmVb, bar, 64, g, b * p.S);
}

// FP8: E4M3 codes of stage `st` (K and V, 64 rows of 128 bytes, 128-byte
// swizzle) -> the f16 staging tile (two boxes of 64 dims per tensor, the same
// layout as a bf16 tile).  A 16-byte chunk of codes (dims
// 16c .. 16c+15 of one row) becomes two 16-byte chunks in box c / 4.
__device__ __forceinline__ void widen_f8(const uint8_t *st, uint8_t *staging) {
  for (int idx = threadIdx.x; idx < 2 * KT * 8; idx += blockDim.x) {
    const int tensor = idx >> 9, row = (idx >> 3) & 63, c = idx & 7;
    const uint4 w = *reinterpret_cast<const uint4 *>(st + tensor * F8_TILE + row * 128 +
                                                      (((c ^ row) & 7) << 4));
    uint4 lo, hi;
    lo.x = e4m3x2_to_f16x2(w.x, false);
    lo.y = e4m3x2_to_f16x2(w.x, true);
    lo.z = e4m3x2_to_f16x2(w.y, false);
    lo.w = e4m3x2_to_f16x2(w.y, true);
    hi.x = e4m3x2_to_f16x2(w.z, false);
    hi.y = e4m3x2_to_f16x2(w.z, true);
    hi.z = e4m3x2_to_f16x2(w.w, false);
    hi.w = e4m3x2_to_f16x2(w.w, true);
    uint8_t *box = staging + tensor * TILE_BYTES + (c >> 2) * (TILE_BYTES / 2) + row * 128;
    const int c0 = (c & 3) * 2;
    *reinterpret_cast<uint4 *>(box + (((c0 ^ row) & 7) << 4)) = lo;
    *reinterpret_cast<uint4 *>(box + ((((c0 + 1) ^ row) & 7) << 4)) = hi;
  }
}
// FP8: the bf16 block keys (16 rows) -> rows 0..15 of the f16 staging tile.
// Box rows of 128 bytes keep their 128-byte swizzle position (row % 8).
__device__ __forceinline__ void widen_block_f8(const uint8_t *blk, uint8_t *staging) {
  constexpr int BOX = F8_BLK_ROWS * 128;
  for (int idx = threadIdx.x; idx < 4 * F8_BLK_ROWS * 8; idx += blockDim.x) {
    const int box = idx >> 7, within = idx & 127;   // box: K lo, K hi, V lo, V hi
    const uint4 w = *reinterpret_cast<const uint4 *>(blk + box * BOX + within * 16);
    uint4 o;
    o.x = bf16x2_to_f16x2(w.x);
    o.y = bf16x2_to_f16x2(w.y);
    o.z = bf16x2_to_f16x2(w.z);
    o.w = bf16x2_to_f16x2(w.w);
    *reinterpret_cast<uint4 *>(staging + (box >> 1) * TILE_BYTES + (box & 1) * (TILE_BYTES / 2) +
                               within * 16) = o;
  }
}

// `pre`: tiles 0..pre-1 were already issued by the caller (context tiles,
// issued before the predecessor kernel finished).  FP8: the caller has also
// issued the block keys (issue_block_f8) when has_block; `buse` counts the
// block region's uses (its barrier phase).
// KS key groups: with KS = 2 (at most 32 query rows, i.e. two warps of
// rows) the CTA runs twice the warps and warp group kg takes keys
// 32 kg .. 32 kg + 31 of every tile; the two groups' partial softmax states
// are merged at the end, so the caller sees the result in warps 0 .. RW-1.
template <bool FP8, int KS>
__device__ __forceinline__ bool attend(const Params &p, uint8_t *smem, uint64_t *full, uint32_t &use,
                                       uint32_t &buse, int b, int g, int kv, int first_page, int pg0,
                                       int pg1, bool has_block, Acc &a, int pre = 0) {
  constexpr int NT = 8 / KS;                 // 8-key n-tiles of a tile per warp
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const int S = p.S, R = p.R, G = p.n_heads / p.kvh;
  const int RW = (R + 15) >> 4;              // warps of query rows
  const int warp = (threadIdx.x >> 5) % RW, kg = (threadIdx.x >> 5) / RW;
  const int key0 = kg * (KT / KS);           // first key of this warp's part of a tile
  const int nctx = max(0, pg1 - pg0);
  const int ntiles = nctx + (has_block ? 1 : 0);
  float(&o)[16][4] = a.o;
  float &m0 = a.m0, &m1 = a.m1, &l0 = a.l0, &l1 = a.l1;
  // query rows of this warp: r = warp*16 + grp (+8); row r -> head g*G + r/S, position j = r%S
  const int r0 = warp * 16 + grp, r1 = r0 + 8;
  uint32_t qa[8][4];
  {
    const bf16 *q = p.q;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = hh ? r1 : r0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int d = ks * 16 + half * 8 + tig * 2;
          uint32_t v = 0;
          if (r < R) {
            const int h = g * G + r / S, j = r % S;
            v = *reinterpret_cast<const uint32_t *>(q + ((size_t)(b * S + j) * p.n_heads + h) * 128 + d);
            if (FP8) v = bf16x2_to_f16x2(v);
          }
          qa[ks][half * 2 + hh] = v;
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  m0 = -INFINITY;
  m1 = -INFINITY;
  l0 = 0.f;
  l1 = 0.f;
  const int j0 = r0 % S, j1 = r1 % S;
  const int lo0 = first_visible(p, kv, j0), lo1 = first_visible(p, kv, j1);
  uint8_t *staging = smem + F8_STAGING;

  auto issue = [&](int t, uint32_t u) {
    issue_tile<FP8>(p, smem, full, u, b, g, first_page + pg0 + t, t >= pg1 - pg0);
  };
  // FP8: the ring carries only the context tiles; the block keys come last
  const int nring = FP8 ? nctx : ntiles;
  if (threadIdx.x == 0)
    for (int t = pre; t < STAGES && t < nring; ++t) issue(t, use + t);

  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const bool blk = t >= nctx;
    const uint32_t u = use + t;
    uint32_t kbase, vbase;
    float sl = p.scale_log2, vm = 1.f;   // logit scale (log2 units), P factor
    if (FP8) {
      if (!blk) {
        if (!mbar_wait(&full[u % STAGES], (u / STAGES) & 1)) ok = false;
        widen_f8(smem + (u % STAGES) * F8_STAGE, staging);
        sl = p.scale_log2 * p.k_mul;
        vm = p.v_mul;
      } else {
        if (!mbar_wait(&full[STAGES], buse & 1)) ok = false;
        ++buse;
        widen_block_f8(smem + F8_BLOCK, staging);
      }
      __syncthreads();   // staging complete; the stage is free again
      if (!blk && threadIdx.x == 0 && t + STAGES < nring) issue(t + STAGES, u + STAGES);
      kbase = su32(staging);
    } else {
      if (!mbar_wait(&full[u % STAGES], (u / STAGES) & 1)) ok = false;
      kbase = su32(smem + (u % STAGES) * STAGE_BYTES);
    }
    vbase = kbase + TILE_BYTES;
    // FP8 block tile: only its 16 rows are in the staging tile
    const bool short_tile = FP8 && blk;
    const int pos0 = (first_page + pg0 + t) * KT;   // position of key 0 of a context tile
    // ---- S = Q K^T (16 rows x 64 / KS keys per warp)
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (short_tile && key0 + nt * 8 >= F8_BLK_ROWS) continue;
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {          // 32 dims per ldmatrix.x4
        const int key = key0 + nt * 8 + (lane & 7);
        const int d = kc * 32 + (lane >> 3) * 8;
        const uint32_t addr = swz(kbase + (d >> 6) * (TILE_BYTES / 2), key, (d & 63) >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        if (FP8) {
          mma16816_f16(s[nt], qa[kc * 2], b0, b1);
          mma16816_f16(s[nt], qa[kc * 2 + 1], b2, b3);
        } else {
          mma16816(s[nt], qa[kc * 2], b0, b1);
          mma16816(s[nt], qa[kc * 2 + 1], b2, b3);
        }
      }
    }
    // ---- mask, online softmax.  A context tile that every row of the warp
    // sees whole (all but the last tile and the window edges) needs no mask.
    float mx0 = -INFINITY, mx1 = -INFINITY;
    const bool whole = __all_sync(0xffffffffu, !blk && pos0 + KT <= kv && pos0 >= lo0 &&
                                                   pos0 >= lo1 && r1 < R);
    if (whole) {
      // every score finite: the scale folds into the exponent (one FMA), and
      // the accumulators are rescaled only when a row maximum of the warp moved
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0 * sl), mn1 = fmaxf(m1, mx1 * sl);
      const bool moved = __any_sync(0xffffffffu, mn0 != m0 || mn1 != m1);
      const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);   // m = -inf at first: a = 0
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = exp2f(fmaf(s[nt][0], sl, -mn0));
        s[nt][1] = exp2f(fmaf(s[nt][1], sl, -mn0));
        s[nt][2] = exp2f(fmaf(s[nt][2], sl, -mn1));
        s[nt][3] = exp2f(fmaf(s[nt][3], sl, -mn1));
        ps0 += s[nt][0] + s[nt][1];
        ps1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
      if (moved) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          o[i][0] *= a0;
          o[i][1] *= a0;
          o[i][2] *= a1;
          o[i][3] *= a1;
        }
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = key0 + nt * 8 + tig * 2 + (e & 1);
          const bool row1 = e >= 2;
          bool vis;
          if (blk) {
            vis = key < S;
          } else {
            const int pos = pos0 + key;
            vis = pos < kv && pos >= (row1 ? lo1 : lo0);
          }
          if ((row1 ? r1 : r0) >= R) vis = false;
          const float v = vis ? s[nt][e] * sl : -INFINITY;
          s[nt][e] = v;
          if (row1) mx1 = fmaxf(mx1, v); else mx0 = fmaxf(mx0, v);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float a0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
      const float a1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = s[nt][0] == -INFINITY ? 0.f : exp2f(s[nt][0] - mn0);
        s[nt][1] = s[nt][1] == -INFINITY ? 0.f : exp2f(s[nt][1] - mn0);
        s[nt][2] = s[nt][2] == -INFINITY ? 0.f : exp2f(s[nt][2] - mn1);
        s[nt][3] = s[nt][3] == -INFINITY ? 0.f : exp2f(s[nt][3] - mn1);
        ps0 += s[nt][0] + s[nt][1];
        ps1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= a0;
        o[i][1] *= a0;
        o[i][2] *= a1;
        o[i][3] *= a1;
      }
    }
    // ---- O += P V (P from the S accumulators, V via transposed ldmatrix);
    // FP8 context tiles: P carries the V factor, f16 operands
#pragma unroll
    for (int kk = 0; kk < NT / 2; ++kk) {         // 16 keys per step
      if (short_tile && key0 + kk * 16 >= F8_BLK_ROWS) continue;
      uint32_t pa[4];
      if (FP8) {
        pa[0] = pack_f16(s[2 * kk][0] * vm, s[2 * kk][1] * vm);
        pa[1] = pack_f16(s[2 * kk][2] * vm, s[2 * kk][3] * vm);
        pa[2] = pack_f16(s[2 * kk + 1][0] * vm, s[2 * kk + 1][1] * vm);
        pa[3] = pack_f16(s[2 * kk + 1][2] * vm, s[2 * kk + 1][3] * vm);
      } else {
        pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
        pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
        pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      }
#pragma unroll
      for (int np = 0; np < 8; ++np) {            // pairs of 8-dim n-tiles
        const int key = key0 + kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int d = np * 16 + (lane >> 4) * 8;
        const uint32_t addr = swz(vbase + (d >> 6) * (TILE_BYTES / 2), key, (d & 63) >> 3);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        if (FP8) {
          mma16816_f16(o[2 * np], pa, b0, b1);
          mma16816_f16(o[2 * np + 1], pa, b2, b3);
        } else {
          mma16816(o[2 * np], pa, b0, b1);
          mma16816(o[2 * np + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();   // every warp is done with this stage (FP8: with the staging tile)
    if (!FP8 && threadIdx.x == 0 && t + STAGES < ntiles) issue(t + STAGES, u + STAGES);
  }
  use += nring;
  if (!ok && lane == 0) raise_error(p.err, DFLASH_DERR_TIMEOUT);

  // ---- finish: row sums across the quad
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (KS == 2) {
    // the second key group's (O, m, l) through shared memory (the stage
    // ring is idle: every issued tile has been consumed) into the first's
    float *x = reinterpret_cast<float *>(smem) + ((size_t)warp * 32 + lane) * 68;
    if (kg == 1) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<float4 *>(x + 4 * i) = make_float4(o[i][0], o[i][1], o[i][2], o[i][3]);
      *reinterpret_cast<float4 *>(x + 64) = make_float4(m0, m1, l0, l1);
    }
    __syncthreads();
    if (kg == 0) {
      const float4 ml = *reinterpret_cast<const float4 *>(x + 64);
      const float n0 = fmaxf(m0, ml.x), n1 = fmaxf(m1, ml.y);
      const float a0 = n0 == -INFINITY ? 0.f : exp2f(m0 - n0), b0 = n0 == -INFINITY ? 0.f : exp2f(ml.x - n0);
      const float a1 = n1 == -INFINITY ? 0.f : exp2f(m1 - n1), b1 = n1 == -INFINITY ? 0.f : exp2f(ml.y - n1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 w = *reinterpret_cast<const float4 *>(x + 4 * i);
        o[i][0] = o[i][0] * a0 + w.x * b0;
        o[i][1] = o[i][1] * a0 + w.y * b0;
        o[i][2] = o[i][2] * a1 + w.z * b1;
        o[i][3] = o[i][3] * a1 + w.w * b1;
      }
      l0 = l0 * a0 + ml.z * b0;
      l1 = l1 * a1 + ml.w * b1;
      m0 = n0;
      m1 = n1;
    }
    __syncthreads();   // the exchange area may be reused
  }
  return ok;
}

// ---------------------------------------------------------------- main kernel
// MAXT: threads per CTA this instantiation is built for; up to 128 threads
// (G*S <= 64 query rows) three CTAs share an SM, which is what hides the
// latency of the per-tile MMA/softmax chain.
template <int MAXT, bool FP8, int KS>
__global__ void __launch_bounds__(MAXT, MAXT <= 128 ? 3 : 1) attn_mma_kernel(const __grid_constant__ Params p) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + (FP8 ? F8_BARS : STAGES * STAGE_BYTES));
  int *s_flag = (int *)(full + STAGES + 1);
  // [MAX_SPLITS + 1][R] merge weights (FP8: in the staging tile, free between items)
  float *s_w = (float *)(smem + (FP8 ? F8_STAGING : STAGES * STAGE_BYTES + 64));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int grp = lane >> 2, tig = lane & 3;
  const int S = p.S, R = p.R, G = p.n_heads / p.kvh;
  const int pps = *p.pps_ptr;
  const int n_bg = p.B * p.kvh;
  const int total_items = p.item_start[n_bg];

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES + (FP8 ? 1 : 0); ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full[i])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t use = 0, buse = 0;   // stage uses so far (ring position and phase), block uses

  for (int item = blockIdx.x; item < total_items; item += gridDim.x) {
    // item -> (b, g, split)
    int lo_i = 0, hi_i = n_bg - 1;
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i + 1) >> 1;
      if (p.item_start[mid] <= item) lo_i = mid; else hi_i = mid - 1;
    }
    const int bg = lo_i, b = bg / p.kvh, g = bg % p.kvh;
    const int split = item - p.item_start[bg];
    const int nsplit = p.item_start[bg + 1] - p.item_start[bg];
    const int kv = clamp_kv(p, p.kv_len[b]);
    const int lo = visible_lo(kv, p.window, p.draft_window);
    const int first_page = lo / KT;
    const int pages = kv > lo ? (kv - 1) / KT - first_page + 1 : 0;
    const int pg0 = split * pps, pg1 = min(pages, pg0 + pps);
    const bool has_block = split == nsplit - 1;

    if (FP8 && has_block && threadIdx.x == 0) issue_block_f8(p, smem, full, b, g);
    Acc acc;
    attend<FP8, KS>(p, smem, full, use, buse, b, g, kv, first_page, pg0, pg1, has_block, acc);
    const int r0 = warp * 16 + grp, r1 = r0 + 8;
    float(&o)[16][4] = acc.o;
    const float m0 = acc.m0, m1 = acc.m1, l0 = acc.l0, l1 = acc.l1;
    if (nsplit == 1) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = hh ? r1 : r0;
        if (r >= R) continue;
        const float inv = 1.f / (hh ? l1 : l0);
        const int h = g * G + r / S, j = r % S;
        bf16 *dst = p.out + ((size_t)(b * S + j) * p.n_heads + h) * 128;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
          const int d = nt * 8 + tig * 2;
          *reinterpret_cast<__nv_bfloat162 *>(dst + d) =
              __floats2bfloat162_rn(o[nt][hh * 2] * inv, o[nt][hh * 2 + 1] * inv);
        }
      }
      continue;
    }
    float *po = p.part_o + (size_t)item * R * 128;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int r = hh ? r1 : r0;
      if (r >= R) continue;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        const int d = nt * 8 + tig * 2;
        *reinterpret_cast<float2 *>(po + r * 128 + d) = make_float2(o[nt][hh * 2], o[nt][hh * 2 + 1]);
      }
      if (tig == 0) p.part_ml[(size_t)item * R + r] = make_float2(hh ? m1 : m0, hh ? l1 : l0);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_flag = atomicAdd(&p.tickets[bg], 1) == nsplit - 1;
    __syncthreads();
    if (*s_flag) {
      __threadfence();
      const int base = p.item_start[bg];
      // per-row merge weights of the splits, then a float4 sweep over O
      for (int r = threadIdx.x; r < R; r += blockDim.x) {
        float mstar = -INFINITY;
        for (int sp = 0; sp < nsplit; ++sp)
          mstar = fmaxf(mstar, __ldcg(&p.part_ml[(size_t)(base + sp) * R + r].x));
        float den = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) {
          const float2 ml = __ldcg(&p.part_ml[(size_t)(base + sp) * R + r]);
          const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mstar);
          s_w[sp * R + r] = w;
          den += w * ml.y;
        }
        s_w[MAX_SPLITS * R + r] = 1.f / den;
      }
      __syncthreads();
#pragma unroll 4
      for (int idx = threadIdx.x; idx < R * 32; idx += blockDim.x) {
        const int r = idx >> 5, d = (idx & 31) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < nsplit; ++sp) {
          const float w = s_w[sp * R + r];
          const float4 v = __ldcg(reinterpret_cast<const float4 *>(
              &p.part_o[((size_t)(base + sp) * R + r) * 128 + d]));
          acc.x += w * v.x;
          acc.y += w * v.y;
          acc.z += w * v.z;
          acc.w += w * v.w;
        }
        const float inv = s_w[MAX_SPLITS * R + r];
        const int h = g * G + r / S, j = r % S;
        bf16 *dst = p.out + ((size_t)(b * S + j) * p.n_heads + h) * 128 + d;
        *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        *reinterpret_cast<__nv_bfloat162 *>(dst + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      }
      if (threadIdx.x == 0) p.tickets[bg] = 0;
    }
    __syncthreads();
  }
  pdl_trigger();
  (void)nwarps;
}

// ---------------------------------------------------------------- small batches
// One thread-block cluster of C CTAs per (request, KV head): CTA rank r takes
// the r-th of C equal slices of the context pages (the last rank also the
// block keys), then the C partial results are merged through distributed
// shared memory -- no scratch in global memory, no tickets, no prep kernel.
template <bool FP8, int KS>
__global__ void __launch_bounds__(256) attn_cluster_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t *full = (uint64_t *)(smem + (FP8 ? F8_BARS : STAGES * STAGE_BYTES));
  cg::cluster_group cl = cg::this_cluster();
  const int C = (int)cl.num_blocks();
  const int rank = (int)cl.block_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const int S = p.S, R = p.R, G = p.n_heads / p.kvh;
  const int bg = blockIdx.x / C, b = bg / p.kvh, g = bg % p.kvh;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES + (FP8 ? 1 : 0); ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full[i])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int kv_raw = p.kv_len[b];
  const int kv = clamp_kv(p, kv_raw);
  if (kv != kv_raw && threadIdx.x == 0 && rank == 0) raise_error(p.err, DFLASH_DERR_KV_CAPACITY);
  const int lo = visible_lo(kv, p.window, p.draft_window);
  const int first_page = lo / KT;
  const int pages = kv > lo ? (kv - 1) / KT - first_page + 1 : 0;
  const int pg0 = pages * rank / C, pg1 = pages * (rank + 1) / C;
  // The context pages, kv_len and the page table were written before the
  // previous kernel started (only Q and the block K/V come from it): their
  // first tiles go out before waiting for it.
  const int pre = min(STAGES, pg1 - pg0);
  if (threadIdx.x == 0)
    for (int t = 0; t < pre; ++t) issue_tile<FP8>(p, smem, full, t, b, g, first_page + pg0 + t, false);
  pdl_wait();
  if (FP8 && rank == C - 1 && threadIdx.x == 0) issue_block_f8(p, smem, full, b, g);
  uint32_t use = 0, buse = 0;
  Acc acc;
  attend<FP8, KS>(p, smem, full, use, buse, b, g, kv, first_page, pg0, pg1, rank == C - 1, acc, pre);
  // this CTA's partial (unnormalised O, row max, row sum) into its own shared memory;
  // the stage ring is free: attend() ends every tile with a CTA barrier
  float *po = reinterpret_cast<float *>(smem);                    // [R][128]
  float2 *pml = reinterpret_cast<float2 *>(smem + R * 128 * 4);   // [R]
  const int r0 = warp * 16 + grp, r1 = r0 + 8;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int r = hh ? r1 : r0;
    if (r >= R) continue;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
      *reinterpret_cast<float2 *>(po + r * 128 + nt * 8 + tig * 2) =
          make_float2(acc.o[nt][hh * 2], acc.o[nt][hh * 2 + 1]);
    if (tig == 0) pml[r] = make_float2(hh ? acc.m1 : acc.m0, hh ? acc.l1 : acc.l0);
  }
  cl.sync();
  // rank r merges rows [R*r/C, R*(r+1)/C) from every CTA of the cluster; all
  // remote loads of an item go out before any arithmetic
  const int rb = R * rank / C, re = R * (rank + 1) / C;
  const int nthr = blockDim.x;
  for (int idx = threadIdx.x; idx < (re - rb) * 32; idx += nthr) {
    const int r = rb + idx / 32, d = (idx % 32) * 4;
    float2 ml[kMaxCluster];
    float4 v[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (c >= C) break;
      ml[c] = cl.map_shared_rank(pml, c)[r];
      v[c] = *reinterpret_cast<const float4 *>(cl.map_shared_rank(po, c) + r * 128 + d);
    }
    float mstar = -INFINITY;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (c >= C) break;
      mstar = fmaxf(mstar, ml[c].x);
    }
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (c >= C) break;
      const float w = ml[c].x == -INFINITY ? 0.f : exp2f(ml[c].x - mstar);
      num.x += w * v[c].x;
      num.y += w * v[c].y;
      num.z += w * v[c].z;
      num.w += w * v[c].w;
      den += w * ml[c].y;
    }
    const float inv = 1.f / den;
    const int h = g * G + r / S, j = r % S;
    bf16 *dst = p.out + ((size_t)(b * S + j) * p.n_heads + h) * 128 + d;
    *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(num.x * inv, num.y * inv);
    *reinterpret_cast<__nv_bfloat162 *>(dst + 2) = __floats2bfloat162_rn(num.z * inv, num.w * inv);
  }
  cl.sync();   // peers may still be reading this CTA's shared memory
  __syncthreads();
  pdl_trigger();
}

}  // namespace att

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn att_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)ptr;
  }
  return fn;
}
// [rows, kvh, 128] bf16 viewed as dims {128, kvh, rows}; box {64, 1, box_rows}.
bool encode_kv(CUtensorMap *tm, const void *base, uint64_t rows, int kvh, uint32_t box_rows = 64) {
  EncodeTiledFn fn = att_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)kvh, rows};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)kvh * 128 * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// FP8 cache [rows, kvh, 128] bytes viewed as dims {128, kvh, rows}; box {128, 1, 64}:
// one 128-byte swizzle row per key.
bool encode_kv_f8(CUtensorMap *tm, const void *base, uint64_t rows, int kvh) {
  EncodeTiledFn fn = att_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)kvh, rows};
  cuuint64_t strides[2] = {128, (cuuint64_t)kvh * 128};
  cuuint32_t box[3] = {128, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

size_t attention_mma_scratch_items(int max_batch, int kvh) {
  return (size_t)max_batch * kvh + 8 * (size_t)kTcMaxCtas + 8;
}

bool attention_mma_uses_cluster(const AttnParams &a) {
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  return 4 * a.B * a.n_kv_heads <= 2 * sms;
}

cudaError_t prepare_attention_mma() {
  const void *kernels[] = {(const void *)att::attn_mma_kernel<128, false, 1>,
                           (const void *)att::attn_mma_kernel<128, false, 2>,
                           (const void *)att::attn_mma_kernel<256, false, 1>,
                           (const void *)att::attn_mma_kernel<128, true, 1>,
                           (const void *)att::attn_mma_kernel<128, true, 2>,
                           (const void *)att::attn_mma_kernel<256, true, 1>};
  for (const void *k : kernels) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, att::SMEM);
    if (e != cudaSuccess) return e;
  }
  const void *clusters[] = {(const void *)att::attn_cluster_kernel<false, 1>,
                            (const void *)att::attn_cluster_kernel<false, 2>,
                            (const void *)att::attn_cluster_kernel<true, 1>,
                            (const void *)att::attn_cluster_kernel<true, 2>};
  for (const void *k : clusters) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, att::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

namespace {
// Whether clusters of C CTAs of the cluster kernel (warps warps each) can be
// placed on this device at all; answered once per (C, warps).
bool cluster_fits(int C, int warps) {
  static int known[att::kMaxCluster + 1][9] = {};
  int &k = known[C][warps];
  if (k == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = att::SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    k = (cudaOccupancyMaxActiveClusters(&n, att::attn_cluster_kernel<false, 1>, &cfg) == cudaSuccess && n > 0)
            ? 1 : -1;
    cudaGetLastError();
  }
  return k > 0;
}
}  // namespace

cudaError_t launch_attention_mma(const AttnParams &a, const AttnScratch &w, cudaStream_t s) {
  if (a.B <= 0) return cudaSuccess;
  if (a.head_dim != 128 || a.page_size != att::KT) return cudaErrorInvalidValue;
  const int R = (a.n_heads / a.n_kv_heads) * a.S;
  // at most 32 query rows: two key groups per CTA (twice the warps)
  const int ks = R <= 32 ? 2 : 1;
  const int warps = (R + 15) / 16 * ks;
  if (warps > 8) return cudaErrorInvalidValue;
  if (a.fp8 && a.S > att::F8_BLK_ROWS) return cudaErrorInvalidValue;
  att::Params p;
  memset(&p, 0, sizeof(p));
  const uint64_t cache_rows = (uint64_t)a.n_pages * att::KT;
  const bool maps_ok =
      a.fp8 ? encode_kv_f8(&p.tmK, a.k_cache, cache_rows, a.n_kv_heads) &&
                  encode_kv_f8(&p.tmV, a.v_cache, cache_rows, a.n_kv_heads) &&
                  encode_kv(&p.tmKb, a.kb, (uint64_t)a.B * a.S, a.n_kv_heads, att::F8_BLK_ROWS) &&
                  encode_kv(&p.tmVb, a.vb, (uint64_t)a.B * a.S, a.n_kv_heads, att::F8_BLK_ROWS)
            : encode_kv(&p.tmK, a.k_cache, cache_rows, a.n_kv_heads) &&
                  encode_kv(&p.tmV, a.v_cache, cache_rows, a.n_kv_heads) &&
                  encode_kv(&p.tmKb, a.kb, (uint64_t)a.B * a.S, a.n_kv_heads) &&
                  encode_kv(&p.tmVb, a.vb, (uint64_t)a.B * a.S, a.n_kv_heads);
  if (!maps_ok) return cudaErrorInvalidValue;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  p.q = (const bf16 *)a.q;
  p.out = (bf16 *)a.out;
  p.page_table = a.page_table;
  p.kv_len = a.kv_len;
  p.err = a.err;
  p.B = a.B;
  p.S = a.S;
  p.n_heads = a.n_heads;
  p.kvh = a.n_kv_heads;
  p.pages_per_req = a.pages_per_req;
  p.n_pages = a.n_pages;
  p.window = a.window;
  p.R = R;
  p.scale_log2 = 1.4426950408889634f * a.scale;
  p.draft_window = a.draft_window;
  p.k_mul = a.k_scale;
  p.v_mul = a.v_scale;
  // Few (request, head) pairs: a cluster of C CTAs per pair, merged on chip.
  const int pairs = a.B * a.n_kv_heads;
  if (4 * pairs <= 2 * sms) {
    // as many CTAs per pair as fit in one wave (two clusters' CTAs share an SM)
    int C = 16;
    while (C > 4 && (C * pairs > 2 * sms || (C > 8 && (C * pairs > sms || !cluster_fits(C, warps)))))
      C >>= 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pairs * C);
    cfg.blockDim = dim3(warps * 32);
    cfg.dynamicSmemBytes = att::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (a.fp8)
      return ks == 2 ? cudaLaunchKernelEx(&cfg, att::attn_cluster_kernel<true, 2>, p)
                     : cudaLaunchKernelEx(&cfg, att::attn_cluster_kernel<true, 1>, p);
    return ks == 2 ? cudaLaunchKernelEx(&cfg, att::attn_cluster_kernel<false, 2>, p)
                   : cudaLaunchKernelEx(&cfg, att::attn_cluster_kernel<false, 1>, p);
  }
  const int max_items = (int)attention_mma_scratch_items(a.B, a.n_kv_heads);
  const int per_sm = warps <= 4 ? 3 : 1;   // resident CTAs per SM (shared memory / registers)
  const int cap = a.draft_window > 0 ? INT32_MAX : a.pages_per_req * att::KT;
  cudaError_t e = launch_pdl(att::attn_prep_kernel, dim3(1), dim3(256), 0, s, a.kv_len, a.B,
                             a.n_kv_heads, cap, a.window, a.draft_window, per_sm * sms,
                             max_items, w.item_start, w.pps, a.err);
  if (e != cudaSuccess) return e;
  p.item_start = w.item_start;
  p.pps_ptr = w.pps;
  p.part_o = w.part_o;
  p.part_ml = (float2 *)w.part_ml;
  p.tickets = w.tickets;
  p.max_items = max_items;
  const dim3 grid(per_sm * sms), block(warps * 32);
  if (a.fp8) {
    if (ks == 2) return launch_pdl(att::attn_mma_kernel<128, true, 2>, grid, block, att::SMEM, s, p);
    return warps <= 4 ? launch_pdl(att::attn_mma_kernel<128, true, 1>, grid, block, att::SMEM, s, p)
                      : launch_pdl(att::attn_mma_kernel<256, true, 1>, grid, block, att::SMEM, s, p);
  }
  if (ks == 2) return launch_pdl(att::attn_mma_kernel<128, false, 2>, grid, block, att::SMEM, s, p);
  return warps <= 4 ? launch_pdl(att::attn_mma_kernel<128, false, 1>, grid, block, att::SMEM, s, p)
                    : launch_pdl(att::attn_mma_kernel<256, false, 1>, grid, block, att::SMEM, s, p);
}

}  // namespace dflash
