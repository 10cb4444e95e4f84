// bf16 block attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// The same operation as the mma.sync kernel: non-causal attention of the S
// block queries of a request over [committed context ; the S block keys]
// ("Inside SGLang: DFlash and DFlash 2 Implementation", Step 4: two K/V
// sources inside draft attention; CSDN DFlash article, "draft model predict",
// is_causal=False), with the Kimi-K2.6 draft card's sliding window and the
// draft KV window.  Every (request b, KV head g) owns the R = G*S query rows
// of its query-head group (R <= 64 here); its context pages are cut into
// splits and the last split also takes the block keys.
//
// Per 64-key tile (one KV page of one head, K and V staged by TMA):
//   S   = Q K^T   tcgen05.mma M=128 N=64 K=128: A = Q, the R <= 64 query rows
//                 in 64 slots, slot 16w + t at A row 32w + t (lanes 0-15 of
//                 TMEM lane quarter w); B = the K tile; S lands in TMEM, lane =
//                 A row, column = key.
//   softmax       all four warps: thread t of warp w takes slot 16w + t % 16
//                 and keys 32 (t / 16) .. +31 (one .16x32bx2 TMEM load: a
//                 TMEM address is one per warp, and that shape gives the two
//                 half-warps the two column halves of the same 16 lanes); the
//                 row maximum is combined over the two halves with a shuffle;
//                 P = exp2 of the scaled logits minus the running maximum goes
//                 to shared memory as bf16 (64 slots x 64 keys, 128-byte
//                 swizzle), in the 8-row groups of A rows 32w+16 .. 32w+31,
//                 which hold no query.
//   O^T = V^T P^T tcgen05.mma M=128 N=64 K=64: A = the V tile read
//                 dims-major (MN-major operand: the staged [key][dim] rows as
//                 they are), B = P; lane = dim, column = slot.
//                 The PVs of an item accumulate in one TMEM O^T.  A row's
//                 running maximum m is raised only when a tile's maximum
//                 exceeds it by more than 8 (log2 units), so P <= 2^8; then,
//                 between the PVs of tiles t-1 and t, the four warps rescale
//                 the O^T columns of the rows that moved by exp2(m_old - m_new)
//                 (one vote per tile decides whether that pass runs).  The
//                 end result O / l does not depend on which m was used.
// The MMA of tile t+1's S overlaps the softmax of tile t (double-buffered S
// and P).
//
// Warp roles (192 threads, two CTAs per SM so that each scheduler has two
// softmax warps to switch between): warps 0-3 softmax and accumulation, warp
// 4 TMA producer and work-queue reader, warp 5 TMEM owner and MMA issuer,
// which issues whichever of the next S and the next PV is ready first.  Work
// items come from a device queue in largest-first order (built by the prep
// kernel), so the CTAs finish together.  A split that is not alone leaves
// (O, m, l) in scratch; the last split of a (b, g) to finish merges them
// (atomic ticket).
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace dflash {
namespace atc {

constexpr int KT = 64;                    // keys per tile (one page)
constexpr int NST = 2;                    // K slots and V slots (two CTAs share an SM)
constexpr int TILE = KT * 128 * 2;        // K (or V) of one tile: two boxes of 64 keys x 64 dims
constexpr int Q_KBLK = 128 * 128;         // one 64-dim K-block of the 128-row Q operand
constexpr int NSLOT = 64;                 // query slots: lanes 0-15 of each TMEM lane quarter
constexpr int MAX_SPLITS = 16;
constexpr int NQ = 4;                     // work-queue slots
// Q operand: 128 A rows, but only rows 32w .. 32w+15 (slot 16w + t at row
// 32w + t) hold queries; the 8-row groups of rows 32w+16 .. 32w+31 are free,
// and the two P buffers live there: P row q (8-row group q / 8) at
// P_OFF[pb] + (q / 8) * P_SBO, which lands in those free groups of both K-blocks.
constexpr int P_SBO = 4096;
constexpr int P_OFF0 = 2048, P_OFF1 = 3072;
constexpr int OFF_Q = 0;
constexpr int OFF_ST = OFF_Q + 2 * Q_KBLK;
constexpr int OFF_V = OFF_ST + NST * TILE;                   // the V ring after the K ring
constexpr int OFF_ALPHA = OFF_V + NST * TILE;                // [2][NSLOT] float
constexpr int OFF_ML = OFF_ALPHA + 3 * NSLOT * 4;            // [NSLOT] float2
constexpr int OFF_W = OFF_ML + NSLOT * 8;                    // [MAX_SPLITS + 1][NSLOT] float
constexpr int OFF_MISC = OFF_W + (MAX_SPLITS + 1) * NSLOT * 4;
// barriers: fullK[NST], fullV[NST], emptyK[NST], emptyV[NST], s_full[2],
// s_free[2], p_full[2], p_free[2], o_full[2], corr_done, o_read, q_full, done,
// item_full[NQ], item_empty[NQ]; then the queue entries [NQ][8] and a few words
constexpr int N_BARS = 4 * NST + 14 + 2 * NQ;
constexpr int SMEM = 1024 + OFF_MISC + N_BARS * 8 + NQ * 32 + 64;
static_assert(2 * (SMEM + 1024) <= 228 * 1024, "two CTAs per SM");
constexpr uint32_t TMEM_COLS = 256;       // S[2] at 0 / 64, the O^T accumulator at 128
// A row's running maximum is raised only when a tile's maximum exceeds it by
// more than TAU (log2 units): P <= 2^TAU otherwise, and the O^T column is
// rescaled (a correction between two PV MMAs) only when the maximum moves.
constexpr float TAU = 8.f;
constexpr uint32_t WAIT_LIMIT = 1u << 22;
constexpr int kThreads = 192;

struct Params {
  CUtensorMap tmK, tmV;          // cache: dims {D, KVH, n_pages*64}, box {64, 1, 64}
  CUtensorMap tmKb, tmVb;        // block keys: dims {D, KVH, B*S}, box {64, 1, 64}
  const bf16 *q;                 // [B*S, n_heads, D]
  bf16 *out;                     // [B*S, n_heads, D]
  const int *page_table;
  const int *kv_len;
  const int *item_start;         // [B*KVH + 1] prefix of splits per (b, g)
  const int *pps_ptr;            // [0] pages per split, [1] work-queue counter
  int *counter;                  // work-queue position (reset by the prep kernel)
  const int4 *queue;             // [items][2] the work queue, largest first (see Item)
  float *part_o;                 // [max_items][R][D]
  float2 *part_ml;               // [max_items][R]
  int *tickets;                  // [B*KVH]
  unsigned int *err;
  int B, S, n_heads, kvh, pages_per_req, n_pages, window, R;
  float scale_log2;              // log2(e) / sqrt(D)
  int draft_window;
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t su32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
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
// Bounded wait for the phase of parity `parity`; false = gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    if (mbar_try(b, parity)) return true;
    if (i > 64) __nanosleep(64);
  }
  return false;
}
// Non-blocking test of the phase of parity `parity`.
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// A role's wait: after its first timeout it waits no more (ok stays false),
// so that a broken pipeline ends in bounded time with the error raised.
__device__ __forceinline__ void role_wait(bool &ok, uint64_t *b, uint32_t parity) {
  if (ok && !mbar_wait(b, parity)) ok = false;
}
__device__ __forceinline__ void tma3(void *dst, const CUtensorMap *tm, uint64_t *bar, int x, int y,
                                     int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the tensor cores.
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(bar))
               : "memory");
}
// Each thread of the warp reads N consecutive 32-bit columns of its own TMEM
// lane (N = 8, 16 or 32).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float *v) {
  uint32_t r[N];
  if constexpr (N == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else if constexpr (N == 16) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
  } else {
    static_assert(N == 32, "x8, x16 or x32");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

// Lanes base .. base + 15 of the warp's lane quarter, 32 columns each: thread
// t < 16 reads lane base + t from column c, thread t >= 16 reads lane
// base + t - 16 from column c + 32 (shape .16x32bx2; taddr = base lane | c).
__device__ __forceinline__ void tmem_ld_halves32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32], 32;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Each thread of the warp writes 32 consecutive columns of its own TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
// 2^x by the hardware approximation (ex2.approx.ftz; results below 2^-126 flush to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptors (128-byte swizzle).  K-major: rows of 128
// bytes along K, 8-row core groups `sbo` bytes apart (1024 when packed).
// MN-major: 128-byte rows along M/N, one row per K index; `lbo` = bytes
// between 64-element blocks along M/N, 8-row groups along K 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr, uint32_t sbo = 1024) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16 instruction descriptor: bf16 A and B, fp32 D; a_mn = A is MN-major.
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ work items
__device__ __forceinline__ int visible_lo(int kv, int window, int draft_window) {
  const int lw = draft_window > 0 ? max(0, kv - draft_window) : 0;
  return window > 0 ? max(lw, kv - window + 1) : lw;
}
// First visible context position of a query at block position j.
__device__ __forceinline__ int first_visible(const Params &p, int kv, int j) {
  const int lw = p.draft_window > 0 ? max(0, kv - p.draft_window) : 0;
  return p.window > 0 ? max(lw, kv + j - p.window + 1) : lw;
}
__device__ __forceinline__ int clamp_kv(const Params &p, int kv) {
  const int cap = p.pages_per_req * KT;
  return kv < 0 ? 0 : (p.draft_window == 0 && kv > cap ? cap : kv);
}
// A work item as the prep kernel lays it out in the queue (two int4):
// {item, b * kvh + g, split, nsplit}, {kv, first visible page, first page of
// the split (relative), context pages of the split}.
struct Item {
  int item, b, g, bg, split, nsplit, kv, first_page, pg0, nctx, ntiles;
};
__device__ __forceinline__ Item unpack_item(const int *e, int kvh) {
  Item it;
  it.item = e[0];
  it.bg = e[1];
  it.split = e[2];
  it.nsplit = e[3];
  it.kv = e[4];
  it.first_page = e[5];
  it.pg0 = e[6];
  it.nctx = e[7];
  it.b = it.bg / kvh;
  it.g = it.bg % kvh;
  it.ntiles = it.nctx + (it.split == it.nsplit - 1 ? 1 : 0);
  return it;
}

// ------------------------------------------------------------------ prep
// Splits and the work queue.  pps = pages per split: about `target` items over
// the batch, at least two pages each, at most MAX_SPLITS splits per (request,
// head), never more items than the scratch holds.  item_start numbers the
// items request-major, then head, then split.  The queue lists the full
// splits (pps pages) first and then the last split of every (b, g) by
// decreasing size, so that the last items taken are the smallest.  One CTA of
// kPrepThreads threads, one request per thread (B <= kPrepThreads).
constexpr int kPrepThreads = 1024;

__device__ __forceinline__ int2 block_scan2(int2 v, int2 *s_warp, int2 &total) {
  // exclusive scan of (x, y) over the CTA
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int2 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, inc.x, o), y = __shfl_up_sync(0xffffffffu, inc.y, o);
    if (lane >= o) {
      inc.x += x;
      inc.y += y;
    }
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int2 w = lane < nw ? s_warp[lane] : make_int2(0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, w.x, o), y = __shfl_up_sync(0xffffffffu, w.y, o);
      if (lane >= o) {
        w.x += x;
        w.y += y;
      }
    }
    if (lane < nw) s_warp[lane] = w;   // inclusive warp prefixes
  }
  __syncthreads();
  total = s_warp[nw - 1];
  const int2 before = warp > 0 ? s_warp[warp - 1] : make_int2(0, 0);
  return make_int2(before.x + inc.x - v.x, before.y + inc.y - v.y);
}

__global__ void __launch_bounds__(kPrepThreads) attn_tc_prep_kernel(
    const int *__restrict__ kv_len, int B, int kvh, int cap, int window, int draft_window,
    int target_items, int max_items, int *item_start, int *pps_out, int4 *queue, unsigned int *err) {
  pdl_wait();
  __shared__ int s_rem[kPrepThreads];
  __shared__ int2 s_warp[32];
  __shared__ int s_total, s_max, s_pps;
  const int b = threadIdx.x;
  if (b == 0) {
    s_total = 0;
    s_max = 0;
  }
  __syncthreads();
  int pages = 0, kv = 0, first_page = 0;
  if (b < B) {
    kv = kv_len[b];
    if (kv < 0 || kv > cap) raise_error(err, DFLASH_DERR_KV_CAPACITY);
    kv = kv < 0 ? 0 : (kv > cap ? cap : kv);
    const int lo = visible_lo(kv, window, draft_window);
    first_page = lo / KT;
    pages = kv > lo ? (kv - 1) / KT - first_page + 1 : 0;
    atomicAdd(&s_total, pages * kvh);
    atomicMax(&s_max, pages);
  }
  __syncthreads();
  if (b == 0) {
    const int total = s_total;
    int pps = max(2, (total + target_items - 1) / target_items);
    const int room = max(1, max_items - B * kvh - 1);
    pps = max(pps, (total + room - 1) / room);
    pps = max(pps, (s_max + MAX_SPLITS - 1) / MAX_SPLITS);
    s_pps = pps;
    pps_out[0] = pps;
  }
  __syncthreads();
  const int pps = s_pps;
  const int nsplit = b < B ? max(1, (pages + pps - 1) / pps) : 0;
  const int rem = b < B ? pages - (nsplit - 1) * pps : -1;   // pages of the last split
  s_rem[b] = rem;
  int2 tot;
  const int2 ex = block_scan2(make_int2(nsplit * kvh, b < B ? (nsplit - 1) * kvh : 0), s_warp, tot);
  if (b < B) {
    for (int g = 0; g < kvh; ++g) item_start[b * kvh + g] = ex.x + g * nsplit;
    if (b == B - 1) item_start[B * kvh] = ex.x + nsplit * kvh;
    auto put = [&](int at, int g, int sp) {
      const int pg0 = sp * pps;
      queue[2 * at] = make_int4(ex.x + g * nsplit + sp, b * kvh + g, sp, nsplit);
      queue[2 * at + 1] = make_int4(kv, first_page, pg0, max(0, min(pages, pg0 + pps) - pg0));
    };
    // full splits: queue positions [0, tot.y) in request order
    int pos = ex.y;
    for (int g = 0; g < kvh; ++g)
      for (int sp = 0; sp + 1 < nsplit; ++sp) put(pos++, g, sp);
    // last splits: by decreasing size (ties: lower request first)
    int rank = 0;
    for (int o = 0; o < B; ++o) {
      const int r = s_rem[o];
      rank += (r > rem || (r == rem && o < b)) ? 1 : 0;
    }
    for (int g = 0; g < kvh; ++g) put(tot.y + rank * kvh + g, g, nsplit - 1);
  }
  if (b == 0) pps_out[1] = 0;   // queue position
}

// ------------------------------------------------------------------ main kernel
__global__ void __launch_bounds__(kThreads, 2) attn_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sQ = smem + OFF_Q;
  uint8_t *sST = smem + OFF_ST;
  float *s_alpha = (float *)(smem + OFF_ALPHA);
  float2 *s_ml = (float2 *)(smem + OFF_ML);
  float *s_w = (float *)(smem + OFF_W);
  uint8_t *sV = smem + OFF_V;
  uint64_t *bars = (uint64_t *)(smem + OFF_MISC);
  uint64_t *fullK = bars, *fullV = bars + NST, *emptyK = bars + 2 * NST, *emptyV = bars + 3 * NST;
  uint64_t *s_full = bars + 4 * NST, *s_free = s_full + 2, *p_full = s_free + 2;
  uint64_t *p_free = p_full + 2, *o_full = p_free + 2, *corr_done = o_full + 2;
  uint64_t *o_read = corr_done + 1, *q_full = o_read + 1, *done = q_full + 1;
  uint64_t *item_full = done + 1, *item_empty = item_full + NQ;
  int *s_items = (int *)(item_empty + NQ);          // [NQ][8] queue entries
  uint32_t *s_tmem = (uint32_t *)(s_items + NQ * 8);
  int *s_flag = (int *)(s_tmem + 1);
  int *s_corr = s_flag + 2;                         // [2] tile needs an O^T correction

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = p.S, R = p.R, G = p.n_heads / p.kvh;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&fullK[i], 1);
      mbar_init(&fullV[i], 1);
      mbar_init(&emptyK[i], 1);
      mbar_init(&emptyV[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&p_free[i], 1);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(corr_done, 128);
    mbar_init(o_read, 128);
    mbar_init(q_full, 128);
    mbar_init(done, 1);
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 129);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) tmem_alloc(s_tmem, TMEM_COLS);
  if (warp == 4 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tmK) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&p.tmV) : "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();   // Q, the block K/V and the work list come from the predecessors
  const int total_items = __ldg(&p.item_start[p.B * p.kvh]);
  bool ok = true;

  // consumers: queue entry k (item -1: no more work or a timeout)
  auto get_item = [&](uint32_t k) -> Item {
    role_wait(ok, &item_full[k % NQ], (k / NQ) & 1);
    Item it = unpack_item((const int *)&s_items[(k % NQ) * 8], p.kvh);
    if (!ok) it.item = -1;
    return it;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    // Two cursors over the same sequence of tiles: K tiles go out as soon as
    // a K slot is free (after that tile's S), V tiles as soon as a V slot is
    // free (after that tile's PV), the V cursor never ahead of the K cursor.
    // The K cursor also takes the queue entries, which stay in place until
    // the consumers have finished their items.
    if (lane == 0) {
      auto tile_page = [&](const Item &it, int t) {
        const int lp = it.first_page + it.pg0 + t;
        int page = __ldg(&p.page_table[(size_t)it.b * p.pages_per_req +
                                       (p.draft_window > 0 ? lp % p.pages_per_req : lp)]);
        if (page < 0 || page >= p.n_pages) {
          raise_error(p.err, DFLASH_DERR_PAGE_RANGE);
          page = 0;
        }
        return page;
      };
      auto issue = [&](const CUtensorMap *tm, const CUtensorMap *tmb, uint8_t *dst, uint64_t *bar,
                       const Item &it, int t) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)),
                     "r"(TILE)
                     : "memory");
        if (t < it.nctx) {
          const int page = tile_page(it, t);
          tma3(dst, tm, bar, 0, it.g, page * KT);
          tma3(dst + TILE / 2, tm, bar, 64, it.g, page * KT);
        } else {
          tma3(dst, tmb, bar, 0, it.g, it.b * S);
          tma3(dst + TILE / 2, tmb, bar, 64, it.g, it.b * S);
        }
      };
      uint32_t nf = 0;             // queue entries taken
      uint32_t kq = 0, vq = 0;     // entries of the K and V cursors
      int kt = 0, vt = 0;          // next tile of those entries
      uint32_t uK = 0, uV = 0;     // K and V tiles issued
      bool endK = false, endV = false, hasK = false, hasV = false;
      Item ik, iv;
      uint32_t idle = 0;
      while (ok && !(endK && endV)) {
        bool did = false;
        if (!endK && !hasK) {
          if (kq == nf && mbar_test(&item_empty[nf % NQ], ((nf / NQ) & 1) ^ 1)) {
            const int idx = atomicAdd(p.counter, 1);
            int *e = &s_items[(nf % NQ) * 8];
            if (idx < total_items) {
              const int4 d0 = __ldg(&p.queue[2 * idx]), d1 = __ldg(&p.queue[2 * idx + 1]);
              e[0] = d0.x; e[1] = d0.y; e[2] = d0.z; e[3] = d0.w;
              e[4] = d1.x; e[5] = d1.y; e[6] = d1.z; e[7] = d1.w;
            } else {
              e[0] = -1;
            }
            mbar_arrive(&item_full[nf % NQ]);
            ++nf;
            did = true;
          }
          if (kq < nf) {
            ik = unpack_item(&s_items[(kq % NQ) * 8], p.kvh);
            if (ik.item < 0) {
              endK = true;
            } else {
              hasK = true;
              kt = 0;
            }
          }
        }
        if (hasK && mbar_test(&emptyK[uK % NST], ((uK / NST) & 1) ^ 1)) {
          issue(&p.tmK, &p.tmKb, sST + (uK % NST) * TILE, &fullK[uK % NST], ik, kt);
          ++uK;
          did = true;
          if (++kt == ik.ntiles) {
            hasK = false;
            ++kq;
          }
        }
        if (!endV && !hasV && vq < nf) {
          iv = unpack_item(&s_items[(vq % NQ) * 8], p.kvh);
          if (iv.item < 0) {
            endV = true;
          } else {
            hasV = true;
            vt = 0;
          }
        }
        if (hasV && uV < uK && mbar_test(&emptyV[uV % NST], ((uV / NST) & 1) ^ 1)) {
          issue(&p.tmV, &p.tmVb, sV + (uV % NST) * TILE, &fullV[uV % NST], iv, vt);
          ++uV;
          did = true;
          if (++vt == iv.ntiles) {
            hasV = false;
            ++vq;
          }
        }
        if (did) {
          idle = 0;
        } else if (++idle > WAIT_LIMIT) {
          ok = false;
        } else if (idle > 64) {
          __nanosleep(32);
        }
      }
      if (!ok) {
        raise_error(p.err, DFLASH_DERR_TIMEOUT);
        // the consumers learn of the end through the queue
        if (!endK && kq == nf && mbar_wait(&item_empty[nf % NQ], ((nf / NQ) & 1) ^ 1)) {
          s_items[(nf % NQ) * 8] = -1;
          mbar_arrive(&item_full[nf % NQ]);
        }
      }
      // every copy this CTA issued has landed before it exits (the normal
      // path consumed them all already)
      for (uint32_t v = uK > (uint32_t)NST ? uK - NST : 0; v < uK; ++v) mbar_wait(&fullK[v % NST], (v / NST) & 1);
      for (uint32_t v = uV > (uint32_t)NST ? uV - NST : 0; v < uV; ++v) mbar_wait(&fullV[v % NST], (v / NST) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // Per item: S of tile 0, then whichever is ready first of the next tile's
    // S (its K/V staged, its S buffer read) and the next tile's O^T = V^T P^T
    // (its P written, its O^T buffer read), so that a late K/V tile never
    // holds back the PV that frees an earlier stage.
    if (lane == 0) {
      constexpr uint32_t ID_S = idesc(128, KT, false);
      constexpr uint32_t ID_PV = idesc(128, NSLOT, true);
      const uint32_t qa = su32(sQ);
      auto issue_s = [&](uint32_t uu) {
        tc_fence_after();
        const uint32_t kb = su32(sST + (uu % NST) * TILE);
#pragma unroll
        for (int kblk = 0; kblk < 2; ++kblk)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(tmem + (uu & 1) * 64, desc_kmajor(qa + kblk * Q_KBLK) + 2 * kk,
                      desc_kmajor(kb + kblk * (TILE / 2)) + 2 * kk, ID_S, (kblk | kk) ? 1u : 0u);
        umma_commit(&s_full[uu & 1]);
        umma_commit(&emptyK[uu % NST]);
      };
      // O^T += V^T P^T of tile v into the one accumulator (tile 0 of an item
      // overwrites it); the stage and the P buffer are free once it is done
      auto issue_pv = [&](uint32_t v, bool first) {
        tc_fence_after();
        const uint32_t vb = su32(sV + (v % NST) * TILE);
        const uint32_t pb = qa + ((v & 1) ? P_OFF1 : P_OFF0);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          umma_bf16(tmem + 128, desc_mnmajor(vb + kk * 2048, TILE / 2),
                    desc_kmajor(pb, P_SBO) + 2 * kk, ID_PV, (first && kk == 0) ? 0u : 1u);
        umma_commit(&o_full[v & 1]);
        umma_commit(&emptyV[v % NST]);
        umma_commit(&p_free[v & 1]);
      };
      uint32_t u = 0, ni = 0, ncorr = 0;
      for (uint32_t k = 0;; ++k) {
        const Item it = get_item(k);
        if (it.item < 0) break;
        mbar_arrive(&item_empty[k % NQ]);
        role_wait(ok, q_full, ni & 1);
        role_wait(ok, &fullK[u % NST], (u / NST) & 1);
        role_wait(ok, &s_free[u & 1], ((u >> 1) & 1) ^ 1);
        issue_s(u);
        int ns = 1, np = 0;   // tiles of this item with S issued / with PV issued
        uint32_t idle = 0;
        while (ok && np < it.ntiles) {
          bool did = false;
          if (ns < it.ntiles) {
            const uint32_t uu = u + ns;
            if (mbar_test(&fullK[uu % NST], (uu / NST) & 1) &&
                mbar_test(&s_free[uu & 1], ((uu >> 1) & 1) ^ 1)) {
              issue_s(uu);
              ++ns;
              did = true;
            }
          }
          // PV of tile np: its P written; then the O^T correction the softmax
          // asked for, or (tile 0) the previous item's O^T read out
          const uint32_t v = u + np;
          if (mbar_test(&p_full[v & 1], (v >> 1) & 1) && mbar_test(&fullV[v % NST], (v / NST) & 1)) {
            const bool corr = *(volatile int *)&s_corr[v & 1] != 0;
            const bool ready = np == 0 ? mbar_test(o_read, (ni & 1) ^ 1)
                                       : (!corr || mbar_test(corr_done, ncorr & 1));
            if (ready) {
              if (np > 0 && corr) ++ncorr;
              issue_pv(v, np == 0);
              ++np;
              did = true;
            }
          }
          if (did) {
            idle = 0;
          } else if (++idle > WAIT_LIMIT) {
            ok = false;
          } else if (idle > 64) {
            __nanosleep(32);
          }
        }
        u += it.ntiles;
        ++ni;
      }
      umma_commit(done);
      if (!mbar_wait(done, 0)) ok = false;   // every MMA done before TMEM is freed
      if (!ok) raise_error(p.err, DFLASH_DERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax + accumulation
    // Softmax role: thread (warp w, lane t) takes query slot 16w + t % 16 (A
    // row / TMEM lane 32w + t % 16) and keys 32 (t / 16) .. +31 of each tile.
    // Accumulation role: thread a owns output dim a (TMEM lane a of O^T).
    const int a = threadIdx.x;
    const int t16 = lane & 15, kh = lane >> 4;
    const int slot = warp * 16 + t16;
    const int arow = warp * 32 + t16;
    const bool live = warp * 16 < R;           // the warp's slots hold queries
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    auto bar_math = [] { asm volatile("bar.sync 1, 128;" ::: "memory"); };
    // barrier of the 128 math threads returning the OR of `v` over them
    auto bar_math_or = [](bool v) -> bool {
      uint32_t r;
      asm volatile(
          "{\n\t.reg .pred p, q;\n\t"
          "setp.ne.u32 p, %1, 0;\n\t"
          "bar.red.or.pred q, 1, 128, p;\n\t"
          "selp.u32 %0, 1, 0, q;\n\t}"
          : "=r"(r)
          : "r"((uint32_t)v)
          : "memory");
      return r != 0;
    };

    // A row `arow` of Q, K-block kh <- dims 64 kh .. 64 kh + 63 of the query
    // in `slot` (zeros past R)
    auto write_q = [&](int qb, int qg) {
      const uint4 *src = nullptr;
      if (slot < R) {
        const int h = qg * G + slot / S, j = slot % S;
        src = reinterpret_cast<const uint4 *>(p.q + ((size_t)(qb * S + j) * p.n_heads + h) * 128) +
              kh * 8;
      }
#pragma unroll
      for (int c0 = 0; c0 < 8; c0 += 4) {
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = src ? __ldg(src + c0 + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4 *>(sQ + kh * Q_KBLK + (arow >> 3) * 1024 + (arow & 7) * 128 +
                                     (((c0 + c) ^ (arow & 7)) << 4)) = v[c];
      }
      fence_async_smem();
      mbar_arrive(q_full);
    };
    // queue entry k for all 128 threads: one thread waits, a barrier
    // broadcasts (the loop bounds of every thread come from it)
    int *s_bcast = s_flag + 1;
    auto get_item_all = [&](uint32_t kk) -> Item {
      if (threadIdx.x == 0) *s_bcast = get_item(kk).item;
      bar_math();
      Item e = unpack_item(&s_items[(kk % NQ) * 8], p.kvh);
      e.item = *(volatile int *)s_bcast;
      return e;
    };

    uint32_t u = 0;
    uint32_t k = 0;
    Item it = get_item_all(0);
    if (it.item >= 0) write_q(it.b, it.g);
    while (it.item >= 0) {
      // the next queue entry, taken once this item's last S has been read
      Item nit;
      nit.item = -1;
      const int lo_q = first_visible(p, it.kv, slot % S);
      float m = -INFINITY, l = 0.f;
      const float sl = p.scale_log2;

      for (int t = 0; t < it.ntiles; ++t) {
        const uint32_t uu = u + t;
        // ---- softmax of tile t
        role_wait(ok, &s_full[uu & 1], (uu >> 1) & 1);
        tc_fence_after();
        bool need = false;   // this row's O^T column must be rescaled before PV of tile t
        if (live) {
          float sv[32];
          tmem_ld_halves32(tmem + lane_base + (uu & 1) * 64, sv);
          tc_fence_before();
          mbar_arrive(&s_free[uu & 1]);
          const bool blk = t >= it.nctx;
          const int key0 = 32 * kh;
          const int pos0 = (it.first_page + it.pg0 + t) * KT + key0;
          // every key of this thread visible (all but the edge tiles): no mask
          const bool whole = !blk && pos0 + 32 <= it.kv && pos0 >= lo_q;
          uint32_t vis = 0xffffffffu;
          if (!whole) {
            vis = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int pos = pos0 + i;
              const bool v = blk ? (key0 + i < S) : (pos < it.kv && pos >= lo_q);
              vis |= v ? (1u << i) : 0u;
            }
          }
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if ((vis >> i) & 1u) mx = fmaxf(mx, sv[i]);
          mx *= sl;
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          // the running maximum moves only by more than TAU; before the first
          // visible key of the row its O^T column is still zero
          float alpha = 1.f;
          if (mx > m + TAU) {
            if (m != -INFINITY) {
              alpha = ex2(m - mx);
              need = true;
            }
            m = mx;
          }
          float ps = 0.f;
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float p0 = (vis >> i) & 1u ? ex2(fmaf(sv[i], sl, -m)) : 0.f;
            const float p1 = (vis >> (i + 1)) & 1u ? ex2(fmaf(sv[i + 1], sl, -m)) : 0.f;
            ps += p0 + p1;
            __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
            packed[i / 2] = *reinterpret_cast<uint32_t *>(&h2);
          }
          l = fmaf(l, alpha, ps);
          // P buffer of this tile parity free again: PV of tile uu - 2 done
          role_wait(ok, &p_free[uu & 1], ((uu >> 1) & 1) ^ 1);
          // P row `slot`, keys key0 .. key0 + 31: 16-byte chunks 4 kh .. 4 kh + 3
          uint8_t *prow = sQ + ((uu & 1) ? P_OFF1 : P_OFF0) + (slot >> 3) * P_SBO + (slot & 7) * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int chunk = 4 * kh + c;
            *reinterpret_cast<uint4 *>(prow + ((chunk ^ (slot & 7)) << 4)) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          }
          if (kh == 0) s_alpha[(uu & 1) * NSLOT + slot] = alpha;
          fence_async_smem();
        } else {
          tc_fence_before();
          mbar_arrive(&s_free[uu & 1]);
        }
        // one vote over the 128 threads (also publishes alpha of tile t)
        const bool any = bar_math_or(need);
        if (threadIdx.x == 0) s_corr[uu & 1] = any ? 1 : 0;
        mbar_arrive(&p_full[uu & 1]);
        if (t == it.ntiles - 1) {
          // the last S of the item has been read: the next item's Q may go in
          nit = get_item_all(k + 1);
          if (nit.item >= 0) write_q(nit.b, nit.g);
        }
        if (any) {
          // O^T column q *= alpha_t[q] once PV of tile t - 1 is done (thread a: dim a)
          role_wait(ok, &o_full[(uu - 1) & 1], ((uu - 1) >> 1) & 1);
          tc_fence_after();
          const float4 *al4 = reinterpret_cast<const float4 *>(s_alpha + (uu & 1) * NSLOT);
#pragma unroll
          for (int c0 = 0; c0 < NSLOT; c0 += 32) {
            float ov[32];
            tmem_ld<32>(tmem + lane_base + 128 + c0, ov);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 al = al4[(c0 + i) >> 2];
              ov[i] *= al.x;
              ov[i + 1] *= al.y;
              ov[i + 2] *= al.z;
              ov[i + 3] *= al.w;
            }
            tmem_st32(tmem + lane_base + 128 + c0, ov);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          mbar_arrive(corr_done);
        }
      }
      // ---- O^T of the item (thread a: dim a, every slot) once its last PV is done
      float o[NSLOT];
      {
        const uint32_t v = u + it.ntiles - 1;
        role_wait(ok, &o_full[v & 1], (v >> 1) & 1);
        tc_fence_after();
        tmem_ld<32>(tmem + lane_base + 128, o);
        tmem_ld<32>(tmem + lane_base + 128 + 32, o + 32);
        tc_fence_before();
        mbar_arrive(o_read);
      }
      // ---- row sums over the two key halves of each slot; (m, l) per slot
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (live && kh == 0) s_ml[slot] = make_float2(m, l);
      bar_math();
      const int d = a;   // output dim of this thread
      if (it.nsplit == 1) {
#pragma unroll
        for (int q = 0; q < NSLOT; ++q) {
          if (q >= R) break;
          const float inv = 1.f / s_ml[q].y;
          const int h = it.g * G + q / S, jq = q % S;
          p.out[((size_t)(it.b * S + jq) * p.n_heads + h) * 128 + d] = __float2bfloat16_rn(o[q] * inv);
        }
      } else {
        float *po = p.part_o + (size_t)it.item * R * 128;
#pragma unroll
        for (int q = 0; q < NSLOT; ++q) {
          if (q >= R) break;
          po[q * 128 + d] = o[q];
        }
        if (d < R) p.part_ml[(size_t)it.item * R + d] = s_ml[d];
        __threadfence();
        bar_math();
        if (threadIdx.x == 0) *s_flag = atomicAdd(&p.tickets[it.bg], 1) == it.nsplit - 1;
        bar_math();
        if (*s_flag) {
          __threadfence();
          const int base = __ldg(&p.item_start[it.bg]);
          for (int r = threadIdx.x; r < R; r += 128) {
            float mstar = -INFINITY;
            for (int sp = 0; sp < it.nsplit; ++sp)
              mstar = fmaxf(mstar, __ldcg(&p.part_ml[(size_t)(base + sp) * R + r].x));
            float den = 0.f;
            for (int sp = 0; sp < it.nsplit; ++sp) {
              const float2 ml = __ldcg(&p.part_ml[(size_t)(base + sp) * R + r]);
              const float w = ml.x == -INFINITY ? 0.f : exp2f(ml.x - mstar);
              s_w[sp * NSLOT + r] = w;
              den += w * ml.y;
            }
            s_w[MAX_SPLITS * NSLOT + r] = 1.f / den;
          }
          bar_math();
          for (int idx = threadIdx.x; idx < R * 32; idx += 128) {
            const int r = idx >> 5, dd = (idx & 31) * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sp = 0; sp < it.nsplit; ++sp) {
              const float w = s_w[sp * NSLOT + r];
              const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                  &p.part_o[((size_t)(base + sp) * R + r) * 128 + dd]));
              acc.x += w * v.x;
              acc.y += w * v.y;
              acc.z += w * v.z;
              acc.w += w * v.w;
            }
            const float inv = s_w[MAX_SPLITS * NSLOT + r];
            const int h = it.g * G + r / S, jq = r % S;
            bf16 *dst = p.out + ((size_t)(it.b * S + jq) * p.n_heads + h) * 128 + dd;
            *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
            *reinterpret_cast<__nv_bfloat162 *>(dst + 2) =
                __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
          }
          if (threadIdx.x == 0) p.tickets[it.bg] = 0;
        }
      }
      bar_math();   // s_ml, s_w and the flag may be reused
      mbar_arrive(&item_empty[k % NQ]);
      u += it.ntiles;
      ++k;
      it = nit;
    }
    if (!ok && lane == 0) raise_error(p.err, DFLASH_DERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();   // every global write of this CTA is done
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace atc

// ---------------------------------------------------------------------- host
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tc_encoder() {
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
// [rows, kvh, 128] bf16 viewed as dims {128, kvh, rows}; box {64, 1, 64}, 128-byte swizzle.
bool encode_kv_tc(CUtensorMap *tm, const void *base, uint64_t rows, int kvh) {
  EncodeTiledFn fn = tc_encoder();
  if (!fn) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)kvh, rows};
  cuuint64_t strides[2] = {128 * 2, (cuuint64_t)kvh * 128 * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool attention_tc_eligible(const AttnParams &a) {
  const int R = (a.n_heads / a.n_kv_heads) * a.S;
  return !a.fp8 && a.head_dim == 128 && a.page_size == atc::KT && R >= 1 && R <= atc::NSLOT &&
         a.B <= atc::kPrepThreads && a.n_heads % a.n_kv_heads == 0;
}

cudaError_t prepare_attention_tc() {
  return cudaFuncSetAttribute(atc::attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              atc::SMEM);
}

cudaError_t launch_attention_tc(const AttnParams &a, const AttnScratch &w, cudaStream_t s) {
  if (a.B <= 0) return cudaSuccess;
  if (!attention_tc_eligible(a)) return cudaErrorInvalidValue;
  const int R = (a.n_heads / a.n_kv_heads) * a.S;
  atc::Params p;
  memset(&p, 0, sizeof(p));
  const uint64_t cache_rows = (uint64_t)a.n_pages * atc::KT;
  if (!(encode_kv_tc(&p.tmK, a.k_cache, cache_rows, a.n_kv_heads) &&
        encode_kv_tc(&p.tmV, a.v_cache, cache_rows, a.n_kv_heads) &&
        encode_kv_tc(&p.tmKb, a.kb, (uint64_t)a.B * a.S, a.n_kv_heads) &&
        encode_kv_tc(&p.tmVb, a.vb, (uint64_t)a.B * a.S, a.n_kv_heads)))
    return cudaErrorInvalidValue;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  const int max_items = (int)attention_mma_scratch_items(a.B, a.n_kv_heads);
  const int cap = a.draft_window > 0 ? INT32_MAX : a.pages_per_req * atc::KT;
  // about one item per CTA (two CTAs per SM): measured against four and eight
  // per SM, fewer items cut the per-item start and the split merges; one per
  // SM left large items that unbalanced the CTAs at block size 8
  cudaError_t e = launch_pdl(atc::attn_tc_prep_kernel, dim3(1), dim3(atc::kPrepThreads), 0, s,
                             a.kv_len, a.B, a.n_kv_heads, cap, a.window, a.draft_window,
                             2 * sms, max_items, w.item_start, w.pps, reinterpret_cast<int4 *>(w.order), a.err);
  if (e != cudaSuccess) return e;
  p.q = (const bf16 *)a.q;
  p.out = (bf16 *)a.out;
  p.page_table = a.page_table;
  p.kv_len = a.kv_len;
  p.item_start = w.item_start;
  p.pps_ptr = w.pps;
  p.counter = w.pps + 1;
  p.queue = reinterpret_cast<const int4 *>(w.order);
  p.part_o = w.part_o;
  p.part_ml = (float2 *)w.part_ml;
  p.tickets = w.tickets;
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
  const dim3 grid(2 * sms), block(atc::kThreads);   // two CTAs per SM
  return launch_pdl(atc::attn_tc_kernel, grid, block, atc::SMEM, s, p);
}

}  // namespace dflash
