// Blackwell (sm_103a) tensor-core GEMM for every bf16 contraction of the draft
// pass: fc (K-split over the selected target layers), context K/V of all
// layers, QKV, O, gate/up (paired tiles, SwiGLU), down and lm_head (argmax).
//
//   Y[m, n] = sum_k A[m, k] * W[n, k]      A: tokens x K, W: features x K
//
// Operand roles are swapped for the tensor core ("swap-AB"): the weight tile
// (128 output features) is the MMA's M operand and the token tile (BN = 16..256
// rows) its N operand, so a draft block of 16 tokens still uses full 128-row
// MMAs.  The accumulator D[feature][token] lives in TMEM.
//
// Structure (one CTA per SM, persistent):
//   warp 0      TMA producer: W and A tiles (128B-swizzled, K-major) into a
//               ring of shared-memory slots (one k-block of one 128-row weight
//               tile plus its activation tile; a paired gate/up k-block uses
//               two consecutive slots), mbarrier transaction counts.
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16 (bf16 in,
//               fp32 accumulate), tcgen05.commit frees a stage / publishes an
//               accumulator.  Two accumulator buffers let the epilogue of one
//               tile overlap the MMAs of the next.
//   warps 2..5  epilogue: tcgen05.ld to registers, shared-memory staging, the
//               shared epilogue ops (norm/RoPE/scatter, SwiGLU, argmax, ...).
// A launch runs a *program* of up to kMaxPhases dependent GEMMs (e.g. O-proj,
// gate/up, down, the next layer's QKV): between phases all CTAs meet at a
// grid barrier (the launch is cooperative, so every CTA is resident), and the
// producer streams the next phase's weights into free ring slots before it
// waits -- the weight stream does not stop at a GEMM boundary.
// Work split (stream-K): per phase, the flattened (tile, k-block) iteration
// space is cut into equal contiguous ranges, one per CTA.  A tile covered by
// one CTA is finished directly.  A tile shared by several CTAs is finished by
// its owner, the CTA holding its first k-block -- for that CTA the tile is
// the last segment of its range, so the owner merges after all its other
// work.  The other contributors publish fp32 shares and a count; the owner
// waits for the count (every CTA is resident), pulls the shares into shared
// memory by bulk copy, adds them to its own share in CTA order -- a fixed
// order, so results are deterministic -- and runs the epilogue.
// Every mbarrier wait is bounded; a wait that gives up raises
// DFLASH_DERR_TIMEOUT and the CTA winds down instead of hanging.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "epilogue.cuh"
#include "inject_rows.cuh"
#include "kernels.h"

namespace dflash {
namespace tc {

constexpr int BK = 64;            // k elements per stage: one 128-byte swizzle row
constexpr int THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr uint32_t WAIT_LIMIT = 1u << 22;
// Trace slots per CTA: 0..7 launch-level stamps, then 4 per phase (inputs
// ready at the producer, first MMA, last MMA, epilogue done).
constexpr int kTraceSlots = 8 + 4 * kMaxPhases;

// One GEMM of a program: its operands, epilogues and stream-K schedule.
struct Phase {
  CUtensorMap tmA[kMaxSrc];       // activations, box {BK, BN}
  CUtensorMap tmW[kMaxSeg];       // weights, box {BK, 128}
  EpiParams epi[kMaxSeg];
  int seg_ntiles[kMaxSeg];        // 128-feature tiles per segment (pairs count once)
  int seg_half[kMaxSeg];          // pair: row offset of the second half
  int nseg, pair;
  int nstep;                      // features between consecutive tiles of a segment
  int M, K, KB, m_tiles, tiles;
  int bnt;                        // token rows per tile in this phase
  int k_per_src;
  int counter_off;                // this phase's tickets start here
  int G;                          // CTAs sharing this phase (<= gridDim.x, <= total_iters)
  long long total_iters;
  int nfull;                      // whole tiles per CTA in full waves (see cta_sched)
  // M_dev: row count on the device (<= M); the schedule fields above are then
  // recomputed in the kernel from it (nfeat feature tiles per token tile)
  const int *M_dev;
  int nfeat;
};

struct Params {
  Phase ph[kMaxPhases];
  int nph;
  ProgramEmbed emb;               // phase 0 is the embedding when emb.M > 0
  ProgramFinalize fin;            // draft ids by the last CTA out when fin.M > 0
  ProgramInject inj;              // injection row map in phase 0 when inj.rows > 0
  ProgramNorm nrm;                // GEMM-free phase nrm_phase normalises rows when nrm.M > 0
  int nrm_phase;
  float *partials;                // [gridDim.x][2][<= 2*BN][128]
  int *counters;                  // tickets of every phase, zero between launches
  unsigned int *grid_bar;         // [2] phase arrivals, exits; zero between launches
  unsigned int *err;
  unsigned long long *trace;      // optional [gridDim.x][kTraceSlots] timestamps (ns), test entries only
};
static_assert(sizeof(Params) <= 32000, "kernel parameter block limit");

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t su32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
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
    if (i > 64) __nanosleep(128);
  }
  return false;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, uint64_t *bar, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(su32(dst)),
      "l"((uint64_t)tm), "r"(su32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          su32(dst)),
      "l"((uint64_t)src), "r"(bytes), "r"(su32(bar))
      : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
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
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(bar))
               : "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Each thread of the warp writes 16 consecutive 32-bit columns of its own TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void stamp(const Params &p, int slot) {
  if (p.trace) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[blockIdx.x * kTraceSlots + slot] = t;
  }
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Named-barrier AND-reduction over the 128 epilogue threads (uniform result).
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row core groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
  d |= (uint64_t)1 << 16;                     // leading-dimension offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride-dimension offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}
// Instruction descriptor of kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ schedule
// A phase's work is the (tile, k-block) space.  With several token tiles
// (m_tiles > 1) and at least G tiles, it starts with nfull full waves of
// whole tiles: wave w gives tile w*G + c to CTA c, so the m_tiles CTAs that
// share a weight tile (consecutive tiles in the raster order
// tile = feature tile * m_tiles + token tile) stream the same weight
// k-blocks at the same time and all but the first read them from L2.  The
// remaining tiles (the tail: at least half a wave when there are full waves)
// are split stream-K: their flattened (tile,
// k-block) iterations are cut into Gt = min(G, tail iterations) equal
// contiguous ranges, so every CTA that takes part holds at least one
// iteration (a split tile's contributors are exactly the CTAs between its
// first and last).  In the
// schedule's own numbering CTA c's whole tiles are contiguous: schedule tile
// s < nfull*G is tile (s % nfull) * G + s / nfull; tail tiles keep their
// index.  Only tail tiles are ever split.
struct Range {
  long long b, e;
};
struct Sched {
  Range whole, tail;   // schedule iterations (tile * KB + k-block) of this CTA
};
// The scalars of a phase that the inner loops use, read once per phase into
// registers.
struct PhaseScalars {
  int KB, k_per_src, m_tiles, nseg, pair, M, G, bnt, nfull, Gt, nstep;
  long long total, tail_base, tail_total;
  int seg_ntiles[kMaxSeg];
};
__device__ __forceinline__ PhaseScalars load_scalars(const Phase &ph) {
  PhaseScalars ps;
  ps.KB = ph.KB;
  ps.k_per_src = ph.k_per_src;
  ps.m_tiles = ph.m_tiles;
  ps.nseg = ph.nseg;
  ps.pair = ph.pair;
  ps.M = ph.M;
  ps.G = ph.G;
  ps.bnt = ph.bnt;
  ps.nfull = ph.nfull;
  ps.nstep = ph.nstep;
  ps.total = ph.total_iters;
  if (ph.M_dev) {
    // row count written by the previous kernel (the caller has waited for
    // it): the same schedule the host computes for a known M
    const int M = min(ph.M, max(0, __ldcg(ph.M_dev)));
    ps.M = M;
    ps.m_tiles = (M + ph.bnt - 1) / ph.bnt;
    const int tiles = ph.nfeat * ps.m_tiles;
    ps.total = (long long)tiles * ph.KB;
    ps.G = (int)max(1LL, min((long long)gridDim.x, ps.total));
    ps.nfull = ps.m_tiles > 1 && ph.nseg > 0 ? tiles / ps.G : 0;
    if (ps.nfull > 0 && 2 * (tiles - ps.nfull * ps.G) < ps.G) --ps.nfull;
  }
  ps.tail_base = (long long)ps.nfull * ps.G * ph.KB;
  ps.tail_total = ps.total - ps.tail_base;
  ps.Gt = (int)(ps.tail_total < ps.G ? (ps.tail_total > 0 ? ps.tail_total : 1) : ps.G);
#pragma unroll
  for (int i = 0; i < kMaxSeg; ++i) ps.seg_ntiles[i] = ph.seg_ntiles[i];
  return ps;
}
// CTA c's whole tiles and its share of the tail (empty ranges for CTAs
// that sit the phase out).
__device__ __forceinline__ Sched cta_sched(const PhaseScalars &ps, int c) {
  Sched s;
  if (c >= ps.G) {
    s.whole = {0, 0};
    s.tail = {0, 0};
    return s;
  }
  s.whole.b = (long long)c * ps.nfull * ps.KB;
  s.whole.e = s.whole.b + (long long)ps.nfull * ps.KB;
  if (c < ps.Gt) {
    s.tail.b = ps.tail_base + ps.tail_total * c / ps.Gt;
    s.tail.e = ps.tail_base + ps.tail_total * (c + 1) / ps.Gt;
  } else {
    s.tail = {0, 0};
  }
  return s;
}
// The tile a schedule tile stands for.
__device__ __forceinline__ int sched_tile(const PhaseScalars &ps, int s) {
  if (s >= ps.nfull * ps.G) return s;
  return (s % ps.nfull) * ps.G + s / ps.nfull;
}
// The CTA whose tail range holds tail iteration it (it >= tail_base).
__device__ __forceinline__ int cta_of_tail_iter(const PhaseScalars &ps, long long it) {
  return (int)(((it - ps.tail_base + 1) * ps.Gt - 1) / ps.tail_total);
}

// tile -> (segment, feature tile, token tile), with register-only indexing
template <int BN>
__device__ __forceinline__ void locate(const PhaseScalars &ps, int tile, int &seg, int &n0, int &m0) {
  int nt = tile / ps.m_tiles;
  m0 = (tile - nt * ps.m_tiles) * ps.bnt;
  seg = 0;
#pragma unroll
  for (int i = 0; i < kMaxSeg - 1; ++i) {
    if (seg == i && i < ps.nseg - 1 && nt >= ps.seg_ntiles[i]) {
      nt -= ps.seg_ntiles[i];
      seg = i + 1;
    }
  }
  n0 = nt * ps.nstep;
}

template <int BN, bool PAIRABLE>
struct Cfg {
  static constexpr int P = PAIRABLE ? 2 : 1;              // accumulators per tile
  static constexpr int W_BYTES = 128 * BK * 2;
  static constexpr int A_BYTES = BN * BK * 2;
  static constexpr int SLOT_BYTES = W_BYTES + A_BYTES;
  // SPLIT (256-token tiles with pairs in the program): a paired k-block takes
  // one slot, [W_gate | W_up | activations of PT = 128 tokens], and its
  // accumulator (tokens in lanes, gate then up features in 256 columns) fills
  // one 256-column buffer; plain phases keep
  // [W | activations of 256 tokens].  Smaller tiles pair two slots (the
  // activation tile rides in the first).
  static constexpr bool SPLIT = PAIRABLE && BN == 256;
  static constexpr int PT = SPLIT ? BN / 2 : BN;          // token rows of a paired tile
  static constexpr int CH = SPLIT ? 16 : (BN < 32 ? BN : 32);   // epilogue token chunk
  static constexpr int CH_PLAIN = SPLIT ? 32 : CH;        // ... of a plain phase
  // large tiles: an owner adds the other shares into its TMEM accumulator
  // with direct loads (a 256-token share does not fit the merge area)
  static constexpr bool TMEM_MERGE = BN >= 128;
  // stream-K merge area: shares of a (row chunk, half) of a split tile, one
  // bulk copy each.  The epilogue's fp32 staging tiles (one chunk per half)
  // live in it too: the last slot holds the gate half of a paired tile while
  // the up half's shares come into the slots before it, the first slot the up
  // half (written once its merge is done); a tile's staging is consumed before
  // the next merge starts.
  static constexpr int CHUNK_BYTES = CH * 128 * 4;
  static constexpr int MERGE_MIN = BN >= 128 ? 16 * 1024 : 48 * 1024;   // deeper ring at large tiles
  static constexpr int MERGE_BYTES = MERGE_MIN > P * CHUNK_BYTES ? MERGE_MIN : P * CHUNK_BYTES;
  static constexpr int MERGE_SLOTS = MERGE_BYTES / CHUNK_BYTES;
  static constexpr int BAR_BYTES = 2048;   // mbarriers, TMEM slot, epilogue scratch, row scales
  static constexpr int BUDGET = 225 * 1024;
  static constexpr int SLOTS_RAW =
      (BUDGET - 1024 - MERGE_BYTES - BAR_BYTES) / SLOT_BYTES;
  static constexpr int SLOTS = SLOTS_RAW > 24 ? 24 : SLOTS_RAW;
  static constexpr int SMEM = 1024 + SLOTS * SLOT_BYTES + MERGE_BYTES + BAR_BYTES;
  static constexpr int ACC_COLS = SPLIT ? BN : P * BN;    // one accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS <= 32 ? 32 : (2 * ACC_COLS <= 64 ? 64 :
                                   (2 * ACC_COLS <= 128 ? 128 : (2 * ACC_COLS <= 256 ? 256 : 512)));
  static_assert(SLOTS >= (PAIRABLE && !SPLIT ? 4 : 3), "two k-blocks (paired: two slots each) must fit");
  static_assert(MERGE_SLOTS >= P, "merge area: the staging tiles and, paired, one share");
  static_assert(2 * ACC_COLS <= 512, "accumulators exceed TMEM");
  static_assert(2 * SLOTS * 8 + 6 * 8 <= 496, "barrier region");
};

// Bounded acquire-spin on a grid barrier word (no sleep between polls: the
// wait is on the critical path of every phase change; one 4-byte L2 read per
// poll and CTA); false = gave up after ~2^22 polls (seconds).
__device__ __forceinline__ bool grid_wait(const unsigned int *bar, unsigned int target) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
    if (v >= target) return true;
  }
  return false;
}
// Bounded acquire-spin until a counter reaches `target`; false = gave up.
__device__ __forceinline__ bool counter_wait(const int *ctr, int target) {
  for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
  }
  return false;
}
// Later bulk-async (TMA) reads must observe what generic stores made visible.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// MMAs of k-blocks kb0..kb1-1 of one tile into the accumulator at d0.  NS
// 1: one weight tile per slot; 2: a gate/up pair in two slots sharing the
// activation tile of the first; 3: a gate/up pair in one slot (SPLIT
// layout).  The pair layout is a compile-time constant so that the MMAs of a
// k-block issue back to back (a run-time choice here measurably slowed every
// GEMM).
template <class C, int NS, int BN>
__device__ __forceinline__ bool mma_kblocks(uint32_t &it, int kb0, int kb1, uint32_t d0,
                                            uint8_t *slots, uint64_t *full, uint64_t *empty,
                                            const Params &p) {
  if constexpr (NS == 3) {
    // [W_gate | W_up] is one 256-row operand (the up rows follow the gate rows
    // 16 KB on, 8-row groups 1 KB apart): one M=128 (tokens) x N=256 MMA per
    // k-step reads the token tile once; D lanes are tokens, columns 0..127
    // the gate features and 128..255 the up features
    constexpr uint32_t idesc = idesc_bf16(128, 2 * C::PT);
    for (int kb = kb0; kb < kb1; ++kb) {
      const int s0 = it % C::SLOTS;
      if (!mbar_wait(&full[s0], (it / C::SLOTS) & 1)) return false;
      if (it == 0) stamp(p, 4);
      tc_fence_after();
      const uint32_t st0 = su32(slots + s0 * C::SLOT_BYTES);
      const uint64_t wdesc = sw128_desc(st0);
      const uint64_t adesc = sw128_desc(st0 + 2 * C::W_BYTES);
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk) {
        const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
        umma_bf16(d0, adesc + 2 * kk, wdesc + 2 * kk, idesc, acc);
      }
      umma_commit(&empty[s0]);
      it += 1;
    }
    return true;
  }
  constexpr uint32_t idesc = idesc_bf16(128, BN);
  for (int kb = kb0; kb < kb1; ++kb) {
    const int s0 = it % C::SLOTS;
    if (!mbar_wait(&full[s0], (it / C::SLOTS) & 1)) return false;
    if (it == 0) stamp(p, 4);
    tc_fence_after();
    const uint32_t st0 = su32(slots + s0 * C::SLOT_BYTES);
    const uint64_t adesc = sw128_desc(st0 + C::W_BYTES);
    const uint64_t wdesc0 = sw128_desc(st0);
    int s1 = 0;
    uint64_t wdesc1 = 0;
    if (NS == 2) {
      s1 = (it + 1) % C::SLOTS;
      wdesc1 = sw128_desc(su32(slots + s1 * C::SLOT_BYTES));
    }
#pragma unroll
    for (int kk = 0; kk < BK / 16; ++kk) {
      const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
      umma_bf16(d0, wdesc0 + 2 * kk, adesc + 2 * kk, idesc, acc);
      if (NS == 2) umma_bf16(d0 + BN, wdesc1 + 2 * kk, adesc + 2 * kk, idesc, acc);
    }
    umma_commit(&empty[s0]);
    if (NS == 2) umma_commit(&empty[s1]);
    it += NS;
  }
  return true;
}
// Activation tile of one k-block into slot s (K-split over the A sources).
template <class C, int NS>
__device__ __forceinline__ void issue_a(const Phase &ph, const PhaseScalars &ps, uint8_t *slots,
                                        int s, int k, int m0, uint64_t *full, uint64_t pol) {
  const int src = k / ps.k_per_src;
  constexpr int off = NS == 3 ? 2 * C::W_BYTES : C::W_BYTES;   // after the weight tile(s)
  tma_load_2d(slots + s * C::SLOT_BYTES + off, &ph.tmA[src], &full[s], k - src * ps.k_per_src, m0,
              pol);
}
// The activations of phase ph_i may be read: the preceding kernel (phase 0)
// or every CTA's previous phase has written them.  false = the grid barrier
// wait gave up.
__device__ __forceinline__ bool phase_inputs_ready(const Params &p, int ph_i, int G) {
  if (ph_i == 0) {
    stamp(p, 2);
    pdl_wait();
    stamp(p, 3);
    stamp(p, 8);
    return true;
  }
  const bool ok = grid_wait(p.grid_bar, (unsigned)(ph_i * G));
  fence_proxy_async();   // later TMA reads see the other CTAs' generic stores
  stamp(p, 8 + 4 * ph_i);
  return ok;
}

// TMA producer of one phase: this CTA's (tile, k-block) range, NS slots per
// k-block.  The weights never depend on earlier work: they go out as soon as a
// slot is free.  Activations wait for the phase's inputs (the previous kernel,
// or every CTA's previous phase), at the latest when the next slot to fill
// still holds a weight-only k-block of this phase (waiting for it would never
// end); until then their (slot, k, row) wait in pend_*.  false = a wait gave up.
template <class C, int NS, int BN>
__device__ __forceinline__ bool produce_phase(const Params &p, const Phase &ph,
                                              const PhaseScalars &ps, int ph_i, int cta,
                                              uint32_t &it, uint8_t *slots, uint64_t *full,
                                              uint64_t *empty, int *pend_s, int *pend_k,
                                              int *pend_m, uint64_t pol_w, uint64_t pol_a) {
  // a GEMM-free phase (embedding, normalisation) loads nothing: its inputs
  // are never needed here, and the next phase's weights may stream at once
  if (ps.total == 0) return true;
  const Sched S = cta_sched(ps, cta);
  const uint32_t it0 = it;
  bool ready = false;
  int npend = 0;
  // full waves exist only with 256-token tiles (smaller tiles hold every row)
  constexpr bool FW = BN == 256;
  for (int part = FW ? 0 : 1; part < 2; ++part) {
  const Range R = part ? S.tail : S.whole;
  long long left = R.e - R.b;
  int tile = (int)(R.b / ps.KB), kb = (int)(R.b - (long long)tile * ps.KB) - 1;
  int seg = 0, n0 = 0, m0 = 0, half = 0;
  const CUtensorMap *tmw = &ph.tmW[0];
  if (left > 0) {
    locate<BN>(ps, FW ? sched_tile(ps, tile) : tile, seg, n0, m0);
    tmw = &ph.tmW[seg];
    if (NS >= 2) half = ph.seg_half[seg];
  }
  while (left > 0) {
    --left;
    if (++kb == ps.KB) {
      kb = 0;
      ++tile;
      locate<BN>(ps, FW ? sched_tile(ps, tile) : tile, seg, n0, m0);
      tmw = &ph.tmW[seg];
      if (NS >= 2) half = ph.seg_half[seg];
    }
    const int k = kb * BK;
    constexpr int SPK = NS == 2 ? 2 : 1;   // slots per k-block
    if (!ready && it + SPK - it0 > (uint32_t)C::SLOTS) {
      const bool ok = phase_inputs_ready(p, ph_i, gridDim.x);
      for (int j = 0; j < npend; ++j)
        issue_a<C, NS>(ph, ps, slots, pend_s[j], pend_k[j], pend_m[j], full, pol_a);
      npend = 0;
      ready = true;
      if (!ok) return false;
    }
    // slot uses below SLOTS find a never-used slot: nothing to wait for
    if (it >= (uint32_t)C::SLOTS && !mbar_wait(&empty[it % C::SLOTS], ((it / C::SLOTS) & 1) ^ 1))
      return false;
    if (NS == 2 && it + 1 >= (uint32_t)C::SLOTS &&
        !mbar_wait(&empty[(it + 1) % C::SLOTS], (((it + 1) / C::SLOTS) & 1) ^ 1))
      return false;
    const int s0 = it % C::SLOTS;
    if (NS == 3) {
      // [W_gate | W_up | activations of PT tokens] in one slot
      mbar_expect_tx(&full[s0], 2 * C::W_BYTES + C::PT * BK * 2);
      tma_load_2d(slots + s0 * C::SLOT_BYTES, tmw, &full[s0], k, n0, pol_w);
      tma_load_2d(slots + s0 * C::SLOT_BYTES + C::W_BYTES, tmw, &full[s0], k, half + n0, pol_w);
    } else {
      mbar_expect_tx(&full[s0], NS * C::W_BYTES + C::A_BYTES);
      tma_load_2d(slots + s0 * C::SLOT_BYTES, tmw, &full[s0], k, n0, pol_w);
    }
    if (NS == 2) {
      const int s1 = (it + 1) % C::SLOTS;
      tma_load_2d(slots + s1 * C::SLOT_BYTES, tmw, &full[s0], k, half + n0, pol_w);
      mbar_arrive(&full[s1]);   // keeps the second slot's phase count in step
    }
    if (ready) {
      issue_a<C, NS>(ph, ps, slots, s0, k, m0, full, pol_a);
    } else {
      pend_s[npend] = s0;
      pend_k[npend] = k;
      pend_m[npend] = m0;
      ++npend;
    }
    it += SPK;
  }
  }
  if (!ready) {
    const bool ok = phase_inputs_ready(p, ph_i, gridDim.x);
    for (int j = 0; j < npend; ++j)
      issue_a<C, NS>(ph, ps, slots, pend_s[j], pend_k[j], pend_m[j], full, pol_a);
    if (!ok) return false;
  }
  return true;
}

__device__ __forceinline__ InjectArgs inject_args(const ProgramInject &j) {
  InjectArgs a;
  a.B = j.B;
  a.row_offset = j.row_offset;
  a.n_rows = j.n_rows;
  a.kv_len = j.kv_len;
  a.page_table = j.page_table;
  a.pages_per_req = j.pages_per_req;
  a.n_pages = j.n_pages;
  a.page_size = j.page_size;
  a.max_position = j.max_position;
  a.draft_window = j.draft_window;
  return a;
}

// Row bookkeeping of the block embedding (once per row): its position,
// range checks and the cleared argmax key.
__device__ __forceinline__ void embed_row_setup(const ProgramEmbed &e, unsigned int *err, int m,
                                                bool bad_id) {
  const int b = m / e.S, j = m - b * e.S;
  const int pos = e.kv_len[b] + j;
  const bool bad_pos = pos < 0 || pos >= e.max_position;
  if (bad_id) raise_error(err, DFLASH_DERR_TOKEN_RANGE);
  if (bad_pos) raise_error(err, DFLASH_DERR_POSITION);
  e.row_pos[m] = bad_pos ? 0 : pos;
  e.keys[m] = 0ull;
}

// The block embedding of a program's first phase ("Inside SGLang", Step 3:
// input id = anchor at j = 0, else mask_token_id; position = prefix length +
// j), with the first layer's deferred RMSNorm operand: x, x * g and the sum
// of squares of every 128-feature part of x.  Work item = (row, 256-feature
// chunk): a lane holds 8 features (16-byte loads of the table row and the
// gain) and a warp takes four items per step, issuing all of their loads
// before using any -- the loads' latency, not bandwidth, bounds this phase.
// Lanes 0-15 hold the chunk's first 128-feature part, 16-31 its second.
// (Feature counts that are not a multiple of 256, or unaligned buffers:
// one (row, 128-feature part) item per warp and step.)
__device__ __forceinline__ void program_embed(const ProgramEmbed &e, unsigned int *err, int gwarp,
                                              int nwarps, int lane) {
  const bool vec = (e.H & 255) == 0 && (((uintptr_t)e.table | (uintptr_t)e.gain |
                                          (uintptr_t)e.x | (uintptr_t)e.xg) & 15) == 0;
  if (vec) {
    constexpr int U = 4;
    const int chunks = e.H >> 8, items = e.M * chunks;
    for (int base = gwarp; base < items; base += nwarps * U) {
      int m[U], t[U], id[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int item = base + k * nwarps;
        const bool live = item < items;
        m[k] = live ? item / chunks : 0;
        t[k] = live ? item - m[k] * chunks : 0;
        const int b = m[k] / e.S, j = m[k] - b * e.S;
        id[k] = !live ? 0 : (j == 0 ? e.anchor[b] : e.mask_id);
      }
      uint4 tv[U], gv[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const bool live = base + k * nwarps < items;
        const bool bad = id[k] < 0 || id[k] >= e.vocab;
        const int c = t[k] * 256 + lane * 8;
        tv[k] = make_uint4(0u, 0u, 0u, 0u);
        gv[k] = tv[k];
        if (live && !bad)
          tv[k] = *reinterpret_cast<const uint4 *>((const bf16 *)e.table + (int64_t)id[k] * e.H + c);
        if (live) gv[k] = *reinterpret_cast<const uint4 *>((const bf16 *)e.gain + c);
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (base + k * nwarps >= items) continue;   // the same for the whole warp
        if (t[k] == 0 && lane == 0) embed_row_setup(e, err, m[k], id[k] < 0 || id[k] >= e.vocab);
        const int c = t[k] * 256 + lane * 8;
        const bf16 *vb = reinterpret_cast<const bf16 *>(&tv[k]);
        const bf16 *gb = reinterpret_cast<const bf16 *>(&gv[k]);
        float v[8];
        uint4 o;
        __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[i] = __bfloat162float(vb[i]);
          ss += v[i] * v[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o2[i] = __floats2bfloat162_rn(v[2 * i] * __bfloat162float(gb[2 * i]),
                                        v[2 * i + 1] * __bfloat162float(gb[2 * i + 1]));
        float *xr = e.x + (int64_t)m[k] * e.H + c;
        reinterpret_cast<float4 *>(xr)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(xr)[1] = make_float4(v[4], v[5], v[6], v[7]);
        *reinterpret_cast<uint4 *>((bf16 *)e.xg + (int64_t)m[k] * e.H + c) = o;
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if ((lane & 15) == 0) e.ssq[(int64_t)(2 * t[k] + (lane >> 4)) * e.ssq_ld + m[k]] = ss;
      }
    }
    return;
  }
  const int parts = e.H >> 7;
  for (int item = gwarp; item < e.M * parts; item += nwarps) {
    const int m = item / parts, t = item - m * parts;
    const int b = m / e.S, j = m - b * e.S;
    const int id = j == 0 ? e.anchor[b] : e.mask_id;
    const bool bad_id = id < 0 || id >= e.vocab;
    if (t == 0 && lane == 0) embed_row_setup(e, err, m, bad_id);
    const int c = t * 128 + lane * 4;
    const bf16 *src = (const bf16 *)e.table + (int64_t)(bad_id ? 0 : id) * e.H + c;
    const bf16 *gp = (const bf16 *)e.gain + c;
    float v[4], g[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = bad_id ? 0.f : __bfloat162float(src[k]);
      g[k] = __bfloat162float(gp[k]);
    }
    float *xr = e.x + (int64_t)m * e.H + c;
    bf16 *xgr = (bf16 *)e.xg + (int64_t)m * e.H + c;
    *reinterpret_cast<float4 *>(xr) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<__nv_bfloat162 *>(xgr) = __floats2bfloat162_rn(v[0] * g[0], v[1] * g[1]);
    *reinterpret_cast<__nv_bfloat162 *>(xgr + 2) = __floats2bfloat162_rn(v[2] * g[2], v[3] * g[3]);
    const float ss = warp_sum((v[0] * v[0] + v[1] * v[1]) + (v[2] * v[2] + v[3] * v[3]));
    if (lane == 0) e.ssq[(int64_t)t * e.ssq_ld + m] = ss;
  }
}

// The final RMSNorm as a GEMM-free phase of the program ("Inside SGLang",
// Step 4: the lm_head reads the draft's final-normed hidden state): the
// rows are rounded to bf16 after the row scale, so the lm_head's operand is
// exactly the normalised hidden state the caller may receive.  Work item =
// (row, 256-feature chunk), each lane 8 features; a warp takes four items
// per step and issues all their loads (sums of squares, x, gains) before
// using any, since the loads' latency bounds this phase.
__device__ __forceinline__ void program_norm(const ProgramNorm &q, int gwarp, int nwarps, int lane) {
  constexpr int U = 4;
  const int chunks = q.H >> 8, parts = q.H >> 7, items = q.M * chunks;
  for (int base = gwarp; base < items; base += nwarps * U) {
    float ss[U];
    float4 xa[U], xb[U];
    uint4 gw[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int item = base + k * nwarps;
      const bool live = item < items;
      const int m = live ? item / chunks : 0;
      const int c0 = (item - m * chunks) * 256 + lane * 8;
      ss[k] = 0.f;
      xa[k] = xb[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      gw[k] = make_uint4(0u, 0u, 0u, 0u);
      if (live) {
        for (int t = lane; t < parts; t += 32) ss[k] += __ldcg(q.ssq + (int64_t)t * q.ssq_ld + m);
        const float4 *xr = reinterpret_cast<const float4 *>(q.x + (int64_t)m * q.H + c0);
        xa[k] = __ldcg(xr);
        xb[k] = __ldcg(xr + 1);
        gw[k] = *reinterpret_cast<const uint4 *>((const bf16 *)q.gain + c0);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int item = base + k * nwarps;
      if (item >= items) continue;   // the same for the whole warp
      const int m = item / chunks, c0 = (item - m * chunks) * 256 + lane * 8;
      const float r = rsqrtf(warp_sum(ss[k]) / (float)q.H + q.eps);
      const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&gw[k]);
      const float2 g0 = __bfloat1622float2(g2[0]), g1 = __bfloat1622float2(g2[1]);
      const float2 g2f = __bfloat1622float2(g2[2]), g3 = __bfloat1622float2(g2[3]);
      const float4 a = xa[k], b = xb[k];
      uint4 o;
      __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
      o2[0] = __floats2bfloat162_rn(a.x * r * g0.x, a.y * r * g0.y);
      o2[1] = __floats2bfloat162_rn(a.z * r * g1.x, a.w * r * g1.y);
      o2[2] = __floats2bfloat162_rn(b.x * r * g2f.x, b.y * r * g2f.y);
      o2[3] = __floats2bfloat162_rn(b.z * r * g3.x, b.w * r * g3.y);
      *reinterpret_cast<uint4 *>((bf16 *)q.out + (int64_t)m * q.H + c0) = o;
      if (q.out2) *reinterpret_cast<uint4 *>((bf16 *)q.out2 + (int64_t)m * q.H + c0) = o;
    }
  }
}

// The epilogue of a finished tile read from TMEM: CHc tokens at a time
// through the fp32 staging tiles (the gate or only half at the end of the
// merge area, the up half at its start).
template <class C, int CHc, typename T>
__device__ __forceinline__ void finish_tile(const EpiParams &e, uint32_t tacc, int bnt, int np,
                                            int rows, int m0, int n0, int tid, int f, float *merge,
                                            int *s_int, float *s_rstd) {
  if (C::SPLIT && np == 2 && e.op == EPI_QKV) {
    // Head-pair tile of the 256-token layout (QKV, 128-wide heads): TMEM lane
    // f is token m0 + f, columns 0..127 head n0 / 128 and bnt.. the next head.
    // A thread holds its token's whole head rows, so the per-head RMSNorm
    // needs no exchange between threads and the rotary partners (d, d + 64)
    // are the thread's own columns; each head row leaves in 16-byte stores.
    // The arithmetic is head_ops_d128's: the deferred norm's row scale, the
    // head RMSNorm and its gain, then the rotation.
    const bool live = f < rows;
    const int m = m0 + (live ? f : 0);
    const float sc = e.ssq_in && live ? s_rstd[f] : 1.f;
    const float4 *rope =
        reinterpret_cast<const float4 *>(e.rope + (int64_t)(live ? e.row_pos[m] : 0) * 64);
    // the token's (cos, sin) row (512 bytes) comes into L1 while the sums of
    // squares are formed
#pragma unroll
    for (int j = 0; j < 4; ++j) prefetch_l1(rope + 8 * j);
    const int kvd = e.n_kv_heads * 128;
    float rstd[2];
    T *dst[2];
    const T *gain[2];
    bool nr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float ss[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c0 = 0; c0 < 128; c0 += 32) {
        float v[32];
        tmem_ld16(tacc + h * bnt + c0, v);
        tmem_ld16(tacc + h * bnt + c0 + 16, v + 16);
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float x = v[k] * sc;
          ss[k & 3] += x * x;
        }
      }
      const int hg = (n0 >> 7) + h;
      const int kind = hg < e.n_heads ? 0 : (hg < e.n_heads + e.n_kv_heads ? 1 : 2);
      const int head = kind == 0 ? hg : (kind == 1 ? hg - e.n_heads : hg - e.n_heads - e.n_kv_heads);
      nr[h] = kind != 2;
      rstd[h] = rsqrtf(((ss[0] + ss[1]) + (ss[2] + ss[3])) / 128.f + e.eps);
      gain[h] = (const T *)(kind == 0 ? e.q_gain : e.k_gain);
      dst[h] = kind == 0 ? (T *)e.q_out + (int64_t)m * e.n_heads * 128 + head * 128
                         : (T *)(kind == 1 ? e.k_out : e.v_out) + (int64_t)m * kvd + head * 128;
    }
    for (int c0 = 0; c0 < 64; c0 += 16) {
      // (cos, sin) of elements c0 .. c0+15: two per float4
      float4 cs[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) cs[j] = rope[(c0 >> 1) + j];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float lo[16], hi[16];
        tmem_ld16(tacc + h * bnt + c0, lo);
        tmem_ld16(tacc + h * bnt + 64 + c0, hi);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          lo[k] *= sc;
          hi[k] *= sc;
        }
        if (nr[h]) {
          // the gains are the same for every thread (broadcast loads)
          uint4 gw[4];
          gw[0] = reinterpret_cast<const uint4 *>(gain[h] + c0)[0];
          gw[1] = reinterpret_cast<const uint4 *>(gain[h] + c0)[1];
          gw[2] = reinterpret_cast<const uint4 *>(gain[h] + 64 + c0)[0];
          gw[3] = reinterpret_cast<const uint4 *>(gain[h] + 64 + c0)[1];
          const T *gl = reinterpret_cast<const T *>(gw), *gh = gl + 16;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float c = (k & 1) ? cs[k >> 1].z : cs[k >> 1].x;
            const float sn = (k & 1) ? cs[k >> 1].w : cs[k >> 1].y;
            const float a = lo[k] * rstd[h] * to_f32(gl[k]), b = hi[k] * rstd[h] * to_f32(gh[k]);
            lo[k] = a * c - b * sn;
            hi[k] = b * c + a * sn;
          }
        }
        uint4 pk[4];
        T *pt = reinterpret_cast<T *>(pk);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          pt[k] = from_f32<T>(lo[k]);
          pt[16 + k] = from_f32<T>(hi[k]);
        }
        if (live) {
          reinterpret_cast<uint4 *>(dst[h] + c0)[0] = pk[0];
          reinterpret_cast<uint4 *>(dst[h] + c0)[1] = pk[1];
          reinterpret_cast<uint4 *>(dst[h] + 64 + c0)[0] = pk[2];
          reinterpret_cast<uint4 *>(dst[h] + 64 + c0)[1] = pk[3];
        }
      }
    }
    return;
  }
  if (C::SPLIT && np == 2) {
    // gate/up pair tile of the 256-token layout: TMEM lane f is token m0 + f,
    // columns 0..127 the gate and bnt.. the up features n0 .. n0+127; each
    // thread writes its token's 128 outputs (16-byte stores), scaled by the
    // token's deferred-RMSNorm factor
    const bool live = f < rows;
    const float sc = e.ssq_in && live ? s_rstd[f] : 1.f;
    const int nvalid = e.N / 2;
    T *dst = (T *)e.out_act + (int64_t)(m0 + (live ? f : 0)) * e.ld + n0;
    for (int c0 = 0; c0 < 128; c0 += 16) {
      float gv[16], uv[16];
      tmem_ld16(tacc + c0, gv);
      tmem_ld16(tacc + bnt + c0, uv);
      uint4 pk[2];
      T *pt = reinterpret_cast<T *>(pk);
#pragma unroll
      for (int k = 0; k < 16; ++k) pt[k] = from_f32<T>(silu(gv[k] * sc) * (uv[k] * sc));
      if (live && n0 + c0 + 16 <= nvalid) {
        reinterpret_cast<uint4 *>(dst + c0)[0] = pk[0];
        reinterpret_cast<uint4 *>(dst + c0)[1] = pk[1];
      } else if (live) {
        for (int k = 0; k < 16; ++k)
          if (n0 + c0 + k < nvalid) dst[c0 + k] = pt[k];
      }
    }
    return;
  }
  if (e.op == EPI_ARGMAX && e.ssq_in == nullptr && np == 1 && (bnt & 31) == 0) {
    // lm_head argmax straight from TMEM: thread f holds vocabulary row n0 + f
    // for 32 tokens at a time; a transpose-reduce over the warp's lanes (at
    // offset s every lane keeps half of its 2s candidates and trades the other
    // half with lane ^ s) leaves lane l with the warp's best key of token
    // c0 + l; the four warps meet in shared memory, one atomic per token.
    unsigned long long *xk = reinterpret_cast<unsigned long long *>(merge);   // [4][32]
    const int lane = tid & 31, ew = tid >> 5;
    const int n = n0 + f;
    const bool fvalid = n < e.N;
    for (int c0 = 0; c0 < bnt; c0 += 32) {
      float v[32];
      tmem_ld16(tacc + c0, v);
      tmem_ld16(tacc + c0 + 16, v + 16);
      unsigned long long k[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) k[t] = fvalid ? argmax_key(v[t], n) : 0ull;
#pragma unroll
      for (int sft = 16; sft >= 1; sft >>= 1) {
        const bool up = (lane & sft) != 0;
#pragma unroll
        for (int i = 0; i < sft; ++i) {
          const unsigned long long send = up ? k[i] : k[i + sft];
          const unsigned long long keep = up ? k[i + sft] : k[i];
          const unsigned long long got = __shfl_xor_sync(0xffffffffu, send, sft);
          k[i] = got > keep ? got : keep;
        }
      }
      xk[ew * 32 + lane] = k[0];
      epi_bar();
      if (ew == 0) {
        unsigned long long b = xk[lane];
#pragma unroll
        for (int w = 1; w < 4; ++w) {
          const unsigned long long o = xk[w * 32 + lane];
          b = o > b ? o : b;
        }
        if (c0 + lane < rows && b) atomicMax(e.argmax_keys + m0 + c0 + lane, b);
      }
      epi_bar();
    }
    return;
  }
  if (e.op == EPI_RESID_NORM && e.ssq_in == nullptr && np == 1 && (bnt & 31) == 0 &&
      sizeof(T) == 2 && n0 + 128 <= e.N) {
    // Residual + next norm's operand straight from TMEM (no staging through
    // shared memory): thread f owns feature n0 + f.  The tile goes in units of
    // 16 tokens; the residual rows of the next unit are loaded into registers
    // before this unit's stores and the unit after that is prefetched into L1,
    // so the loads' latency (long while the TMA stream keeps L2 busy) overlaps
    // the stores.  Per 32 tokens the sums of squares of the 128 features come
    // from a warp transpose-reduce and the four warps in shared memory.
    float *red = merge;   // [4][32]
    const int lane = tid & 31, ew = tid >> 5;
    const int n = n0 + f;
    const float g = to_f32(((const T *)e.norm_gain)[n]);
    const int units = bnt >> 4;
    auto row = [&](int u, int t) { return (int64_t)(m0 + 16 * u + t) * e.ld + n; };
    auto load_unit = [&](int u, float *x) {
#pragma unroll
      for (int t = 0; t < 16; ++t) x[t] = 16 * u + t < rows ? e.out_f32[row(u, t)] : 0.f;
    };
    auto prefetch_unit = [&](int u) {   // lane t < 16: row t of the unit (one line per warp)
      if (u < units && lane < 16 && 16 * u + lane < rows) prefetch_l1(e.out_f32 + row(u, lane));
    };
    float xn[16];
    prefetch_unit(1);
    load_unit(0, xn);
    for (int c0 = 0; c0 < bnt; c0 += 32) {
      float sq[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int u = (c0 >> 4) + h;
        float xo[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) xo[t] = xn[t];
        prefetch_unit(u + 2);
        if (u + 1 < units) load_unit(u + 1, xn);
        float v[16];
        tmem_ld16(tacc + 16 * u, v);
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float y = v[t] + xo[t];
          if (16 * u + t < rows) {
            e.out_f32[row(u, t)] = y;
            ((T *)e.out_act)[row(u, t)] = from_f32<T>(y * g);
          }
          sq[16 * h + t] = y * y;
        }
      }
#pragma unroll
      for (int sft = 16; sft >= 1; sft >>= 1) {
        const bool up = (lane & sft) != 0;
#pragma unroll
        for (int i = 0; i < sft; ++i) {
          const float send = up ? sq[i] : sq[i + sft];
          const float keep = up ? sq[i + sft] : sq[i];
          sq[i] = keep + __shfl_xor_sync(0xffffffffu, send, sft);
        }
      }
      red[ew * 32 + lane] = sq[0];
      epi_bar();
      if (ew == 0 && c0 + lane < rows)
        e.ssq_out[(int64_t)(n0 >> 7) * e.ssq_ld + m0 + c0 + lane] =
            (red[lane] + red[32 + lane]) + (red[64 + lane] + red[96 + lane]);
      epi_bar();
    }
    return;
  }
  float *st0 = merge + (C::MERGE_BYTES - CHc * 128 * 4) / 4, *st1 = merge;
  for (int c0 = 0; c0 < bnt; c0 += CHc) {
    float v[CHc];
    for (int q = 0; q < np; ++q) {
      tmem_ld16(tacc + q * bnt + c0, v);
      if (CHc == 32) tmem_ld16(tacc + q * bnt + c0 + 16, v + 16);
      float *dst = q ? st1 : st0;
#pragma unroll
      for (int t = 0; t < CHc; ++t) dst[t * 128 + f] = v[t];
    }
    epi_bar();
    if (c0 < rows)
      run_epilogue<T>(e, st0, np == 2 ? st1 : nullptr, 128, m0 + c0, min(CHc, rows - c0), n0, tid,
                      128, s_int, [] { epi_bar(); }, s_rstd + c0);
    epi_bar();
  }
}

// Owner of a split tile, large tiles: the other contributors' fp32 shares
// are added, in CTA order (deterministic), to this CTA's accumulator in
// TMEM -- 32 tokens and up to two shares per batch of loads, all in flight
// together -- so the tile then finishes like an unsplit one.
template <class C>
__device__ __forceinline__ void tmem_merge(const Params &p, const PhaseScalars &ps, int tile,
                                           int c_first, int others, uint32_t tacc, int bnt, int np,
                                           int f) {
  constexpr int GT = 32, KMAX = 2;
  for (int q = 0; q < np; ++q) {
    for (int g0 = 0; g0 < bnt; g0 += GT) {
      float acc[GT];
      tmem_ld16(tacc + q * bnt + g0, acc);
      tmem_ld16(tacc + q * bnt + g0 + 16, acc + 16);
      for (int k0 = 0; k0 < others; k0 += KMAX) {
        float v[KMAX][GT];
#pragma unroll
        for (int kk = 0; kk < KMAX; ++kk) {
          if (k0 + kk < others) {
            const int c = c_first + 1 + k0 + kk;
            const long long cfirst_tile = (ps.tail_base + ps.tail_total * c / ps.Gt) / ps.KB;
            const int w = tile == cfirst_tile ? 0 : 1;
            const float *sh = p.partials + ((size_t)c * 2 + w) * (C::ACC_COLS * 128) +
                              (size_t)(q * bnt + g0) * 128 + f;
#pragma unroll
            for (int t = 0; t < GT; ++t) v[kk][t] = __ldcg(sh + t * 128);
          }
        }
#pragma unroll
        for (int kk = 0; kk < KMAX; ++kk) {
          if (k0 + kk < others) {
#pragma unroll
            for (int t = 0; t < GT; ++t) acc[t] += v[kk][t];
          }
        }
      }
      tmem_st16(tacc + q * bnt + g0, acc);
      tmem_st16(tacc + q * bnt + g0 + 16, acc + 16);
    }
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

template <int BN, bool PAIRABLE, typename T>
__global__ void __launch_bounds__(THREADS, 1) gemm_tc_kernel(const __grid_constant__ Params p) {
  using C = Cfg<BN, PAIRABLE>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *slots = smem;
  float *merge = (float *)(smem + C::SLOTS * C::SLOT_BYTES);
  uint8_t *barbase = smem + C::SLOTS * C::SLOT_BYTES + C::MERGE_BYTES;
  uint64_t *bars = (uint64_t *)barbase;
  uint64_t *full = bars, *empty = bars + C::SLOTS;
  uint64_t *acc_full = bars + 2 * C::SLOTS, *acc_empty = acc_full + 2;
  uint64_t *mma_done = acc_empty + 2;
  uint64_t *merge_bar = mma_done + 1;
  uint32_t *tmem_slot = (uint32_t *)(barbase + 496);
  int *s_int = (int *)(barbase + 512);        // kEpiScratchInts ints
  float *s_rstd = (float *)(barbase + 1024);  // [BN] deferred-norm row scales

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;

  if (threadIdx.x == 0) stamp(p, 0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::SLOTS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(mma_done, 1);
    mbar_init(merge_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if (warp == 0 && lane == 0) {
    for (int k = 0; k < p.nph; ++k) {
      for (int i = 0; i < p.ph[k].nseg; ++i) prefetch_tmap(&p.ph[k].tmW[i]);
      for (int i = 0; i < kMaxSrc && i * p.ph[k].k_per_src < p.ph[k].K; ++i)
        prefetch_tmap(&p.ph[k].tmA[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) stamp(p, 1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      uint32_t it = 0;   // slot uses so far
      bool ok = true;
      // k-blocks whose weights went out before their activations could:
      // (slot, k, token row), at most one ring's worth
      int pend_s[C::SLOTS], pend_k[C::SLOTS], pend_m[C::SLOTS];
      for (int ph_i = 0; ph_i < p.nph && ok; ++ph_i) {
        const Phase &ph = p.ph[ph_i];
        if (ph.M_dev) pdl_wait();   // the row count comes from the previous kernel
        const PhaseScalars ps = load_scalars(ph);
        if constexpr (PAIRABLE)
          ok = ps.pair ? produce_phase<C, C::SPLIT ? 3 : 2, BN>(p, ph, ps, ph_i, cta, it, slots,
                                                                full, empty, pend_s, pend_k,
                                                                pend_m, pol_w, pol_a)
                       : produce_phase<C, 1, BN>(p, ph, ps, ph_i, cta, it, slots, full, empty,
                                                 pend_s, pend_k, pend_m, pol_w, pol_a);
        else
          ok = produce_phase<C, 1, BN>(p, ph, ps, ph_i, cta, it, slots, full, empty, pend_s,
                                       pend_k, pend_m, pol_w, pol_a);
      }
      if (!ok) raise_error(p.err, DFLASH_DERR_TIMEOUT);
      // drain: no TMA write may still be in flight when the CTA winds down
      for (uint32_t j = 0; j < (uint32_t)C::SLOTS && j < it; ++j) {
        const uint32_t q = it - 1 - j;
        mbar_wait(&full[q % C::SLOTS], (q / C::SLOTS) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      int seg_i = 0;
      bool ok = true;
      for (int ph_i = 0; ph_i < p.nph && ok; ++ph_i) {
        if (p.ph[ph_i].M_dev) pdl_wait();
        const PhaseScalars ps = load_scalars(p.ph[ph_i]);
        const Sched S = cta_sched(ps, cta);
        const int ns = ps.pair ? 2 : 1;
        for (int part = BN == 256 ? 0 : 1; part < 2 && ok; ++part) {
        const Range R = part ? S.tail : S.whole;
        for (long long i = R.b; i < R.e && ok; ++seg_i) {
          const int kb0 = (int)(i % ps.KB);
          const int kb1 = (int)(kb0 + (R.e - i) < ps.KB ? kb0 + (R.e - i) : ps.KB);
          const int buf = seg_i & 1;
          const uint32_t aph = (seg_i >> 1) & 1;
          if (!mbar_wait(&acc_empty[buf], aph ^ 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d0 = tmem + buf * C::ACC_COLS;
          if constexpr (PAIRABLE)
            ok = ns == 2 ? mma_kblocks<C, C::SPLIT ? 3 : 2, BN>(it, kb0, kb1, d0, slots, full,
                                                                 empty, p)
                         : mma_kblocks<C, 1, BN>(it, kb0, kb1, d0, slots, full, empty, p);
          else
            ok = mma_kblocks<C, 1, BN>(it, kb0, kb1, d0, slots, full, empty, p);
          if (!ok) break;
          umma_commit(&acc_full[buf]);
          if (i == R.b && part == (S.whole.e > S.whole.b ? 0 : 1))
            stamp(p, 9 + 4 * ph_i);   // first segment's MMAs issued
          i += kb1 - kb0;
        }
        }
        if (S.whole.e > S.whole.b || S.tail.e > S.tail.b) stamp(p, 10 + 4 * ph_i);
      }
      if (!ok) raise_error(p.err, DFLASH_DERR_TIMEOUT);
      // every MMA issued by this thread must be complete before TMEM is freed
      umma_commit(mma_done);
      mbar_wait(mma_done, 0);
      stamp(p, 5);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - EPI_WARP0;                 // 0..3
    const int tid = ew * 32 + lane;                  // 0..127
    const int quarter = warp & 3;                    // TMEM lane quarter this warp may access
    const int f = quarter * 32 + lane;               // output feature row of this thread
    // staging tiles in the merge area: gate (or only) half in its last slot, up half in its first
    float *st0 = merge + (C::MERGE_SLOTS - 1) * (C::CHUNK_BYTES / 4), *st1 = merge;
    int seg_i = 0;
    uint32_t merge_phase = 0;   // completed phases of merge_bar
    bool alive = true;
    for (int ph_i = 0; ph_i < p.nph && alive; ++ph_i) {
      const Phase &ph = p.ph[ph_i];
      if (ph_i == 0 || ph.M_dev) pdl_wait();
      const PhaseScalars ps = load_scalars(ph);
      const int np = ps.pair ? 2 : 1;
      // this phase reads what the previous kernel / every CTA's previous phase
      // wrote; for the latter one thread spins with acquire semantics and the
      // named barrier orders the other epilogue threads after it
      if (ph_i > 0 && !epi_all(tid == 0 ? grid_wait(p.grid_bar, (unsigned)(ph_i * G)) : true)) {
        if (tid == 0) raise_error(p.err, DFLASH_DERR_TIMEOUT);
        alive = false;
        break;
      }
      if (ph_i == 0 && p.emb.M > 0)
        program_embed(p.emb, p.err, cta * 4 + ew, G * 4, lane);
      if (ph_i == p.nrm_phase && p.nrm.M > 0) program_norm(p.nrm, cta * 4 + ew, G * 4, lane);
      if (ph_i == 0 && p.inj.rows > 0) {
        // the K/V phase's row map (read only after the grid barrier)
        InjectArgs a = inject_args(p.inj);
        for (int r = cta * 128 + tid; r < p.inj.rows; r += G * 128) {
          int slot, pos;
          inject_map_row(a, p.inj.row0 + r, [&](int b) { return a.kv_len[b]; },
                         [&](int b) { return a.row_offset[b]; }, [&](int b) { return a.n_rows[b]; },
                         slot, pos, p.err);
          p.inj.row_slot[r] = slot;
          p.inj.row_pos[r] = pos;
        }
      }
      int rstd_m0 = -1, rstd_seg = -1;   // rows whose deferred-norm scales are in s_rstd
      const Sched S = cta_sched(ps, cta);
      for (int part = BN == 256 ? 0 : 1; part < 2 && alive; ++part) {
      const Range R = part ? S.tail : S.whole;
      for (long long i = R.b; i < R.e; ++seg_i) {
        const int stile = (int)(i / ps.KB);          // schedule tile
        const int tile = BN == 256 ? sched_tile(ps, stile) : stile;
        const int kb0 = (int)(i - (long long)stile * ps.KB);
        const int kb1 = (int)(kb0 + (R.e - i) < ps.KB ? kb0 + (R.e - i) : ps.KB);
        i += kb1 - kb0;
        int seg, n0, m0;
        locate<BN>(ps, tile, seg, n0, m0);
        const EpiParams e = ph.epi[seg];
        const int bnt = ps.bnt;   // token rows of this phase's tiles
        const int rows = min(bnt, ps.M - m0);
        const int buf = seg_i & 1;
        const uint32_t aph = (seg_i >> 1) & 1;
        // row scales of a deferred RMSNorm, computed while the MMAs still run
        if (e.ssq_in != nullptr && (m0 != rstd_m0 || seg != rstd_seg)) {
          epi_bar();   // the previous tile's epilogue is done with s_rstd
          compute_rstd(e, m0, rows, s_rstd, lane, ew, 4);
          rstd_m0 = m0;
          rstd_seg = seg;
        }
        const bool ok = epi_all(mbar_wait(&acc_full[buf], aph));
        if (!ok) {
          if (tid == 0) raise_error(p.err, DFLASH_DERR_TIMEOUT);
          alive = false;
          break;
        }
        tc_fence_after();
        if (tid == 0 && seg_i == 0) stamp(p, 6);
        const uint32_t tacc = tmem + ((uint32_t)(quarter * 32) << 16) + buf * C::ACC_COLS;
        const bool whole = kb0 == 0 && kb1 == ps.KB;
        bool finish = whole;            // this CTA runs the tile's epilogue from TMEM
        int *owner_ticket = nullptr;    // reset after that epilogue (merged in TMEM)
        if (!whole) {
          // Split tile.  Its owner is the CTA holding the tile's first k-block:
          // the tile is the last segment of that CTA's range, so the owner
          // merges after all its other work.  Every other contributor
          // publishes its fp32 share and moves on.
          // (only tail tiles are split, and they keep their index)
          const int c_first = cta_of_tail_iter(ps, (long long)tile * ps.KB);
          const int c_last = cta_of_tail_iter(ps, (long long)(tile + 1) * ps.KB - 1);
          int *ticket = p.counters + ph.counter_off + tile;   // shares published so far
          if (cta != c_first) {
            const long long first_tile = R.b / ps.KB;
            const int which = tile == first_tile ? 0 : 1;
            float *mine = p.partials + ((size_t)cta * 2 + which) * (C::ACC_COLS * 128);
            for (int c0 = 0; c0 < bnt; c0 += C::CH) {
              float v[32];
              for (int q = 0; q < np; ++q) {
                tmem_ld16(tacc + q * bnt + c0, v);
                if (C::CH == 32) tmem_ld16(tacc + q * bnt + c0 + 16, v + 16);
#pragma unroll
                for (int t = 0; t < C::CH; ++t) mine[(q * bnt + c0 + t) * 128 + f] = v[t];
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            // publish: the barrier orders every thread's share before thread
            // 0's fence (cumulative), the count goes out after it
            epi_bar();
            if (tid == 0) {
              __threadfence();
              atomicAdd(ticket, 1);
            }
          } else if (C::TMEM_MERGE) {
            // Owner, large tiles: the other shares (every CTA is resident)
            // are added into this CTA's accumulator, then the tile finishes
            // like an unsplit one.
            const int others = c_last - c_first;
            if (!epi_all(tid == 0 ? counter_wait(ticket, others) : true) && tid == 0)
              raise_error(p.err, DFLASH_DERR_TIMEOUT);
            tmem_merge<C>(p, ps, tile, c_first, others, tacc, bnt, np, f);
            finish = true;
            owner_ticket = ticket;
          } else {
            // Owner: the other shares (every CTA is resident) come into the
            // merge area by bulk copy -- one memory round trip for up to
            // MERGE_SLOTS shares -- and are added to the owner's own share,
            // read from TMEM, in CTA order (a fixed order: deterministic).
            const int others = c_last - c_first;
            if (!epi_all(tid == 0 ? counter_wait(ticket, others) : true) && tid == 0)
              raise_error(p.err, DFLASH_DERR_TIMEOUT);
            for (int c0 = 0; c0 < bnt; c0 += C::CH) {
              for (int q = 0; q < np; ++q) {
                float acc[32];
                tmem_ld16(tacc + q * bnt + c0, acc);
                if (C::CH == 32) tmem_ld16(tacc + q * bnt + c0 + 16, acc + 16);
                // the up half's shares keep clear of the gate half's staging tile
                const int mslots = q ? C::MERGE_SLOTS - 1 : C::MERGE_SLOTS;
                for (int k0 = 0; k0 < others; k0 += mslots) {
                  const int kn = min(mslots, others - k0);
                  if (tid == 0) {
                    fence_proxy_async();   // the shares were written by generic stores
                    // and this area was last written / read by generic accesses
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_expect_tx(merge_bar, kn * C::CHUNK_BYTES);
                    for (int k = 0; k < kn; ++k) {
                      const int c = c_first + 1 + k0 + k;
                      const long long cfirst_tile =
                          (ps.tail_base + ps.tail_total * c / ps.Gt) / ps.KB;
                      const int w = tile == cfirst_tile ? 0 : 1;
                      bulk_g2s(merge + k * (C::CHUNK_BYTES / 4),
                               p.partials + ((size_t)c * 2 + w) * (C::ACC_COLS * 128) +
                                   (size_t)(q * bnt + c0) * 128,
                               C::CHUNK_BYTES, merge_bar);
                    }
                  }
                  if (!epi_all(mbar_wait(merge_bar, merge_phase & 1)) && tid == 0)
                    raise_error(p.err, DFLASH_DERR_TIMEOUT);
                  ++merge_phase;
                  for (int k = 0; k < kn; ++k) {
#pragma unroll
                    for (int t = 0; t < C::CH; ++t) acc[t] += merge[k * (C::CHUNK_BYTES / 4) + t * 128 + f];
                  }
                  epi_bar();   // the merge area may be refilled
                }
                float *dst = q ? st1 : st0;
#pragma unroll
                for (int t = 0; t < C::CH; ++t) dst[t * 128 + f] = acc[t];
              }
              epi_bar();
              if (c0 < rows)
                run_epilogue<T>(e, st0, np == 2 ? st1 : nullptr, 128, m0 + c0,
                                min(C::CH, rows - c0), n0, tid, 128, s_int, [] { epi_bar(); },
                                s_rstd + c0);
              epi_bar();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            if (tid == 0) *ticket = 0;   // ready for the next launch
          }
          epi_bar();
        }
        if (finish) {
          if (C::SPLIT && !ps.pair)
            finish_tile<C, C::CH_PLAIN, T>(e, tacc, bnt, np, rows, m0, n0, tid, f, merge, s_int,
                                           s_rstd);
          else
            finish_tile<C, C::CH, T>(e, tacc, bnt, np, rows, m0, n0, tid, f, merge, s_int, s_rstd);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[buf]);
          if (owner_ticket && tid == 0) *owner_ticket = 0;   // ready for the next launch
        }
      }
      }
      if (!alive) break;
      if (tid == 0) stamp(p, 11 + 4 * ph_i);
      if (ph_i + 1 < p.nph) {
        // this CTA's share of the phase is written: count it in the grid
        // barrier (same publication pattern as a split tile's share)
        epi_bar();
        if (tid == 0) {
          __threadfence();
          atomicAdd(&p.grid_bar[0], 1u);
        }
      }
    }
  }
  if (warp == EPI_WARP0 && lane == 0) stamp(p, 7);
  tc_fence_before();
  __syncthreads();
  if (p.nph > 1 || p.fin.M > 0 || p.inj.advance) {
    // the last CTA out clears the barrier words for the next program and
    // turns the argmax keys every CTA has contributed to into draft ids
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned int old = atomicAdd(&p.grid_bar[1], 1u);
      s_int[0] = old == (unsigned int)G - 1;
      if (old == (unsigned int)G - 1) {
        p.grid_bar[0] = 0;
        p.grid_bar[1] = 0;
        __threadfence();
      }
    }
    __syncthreads();
    if (s_int[0] && p.inj.advance) {
      // every CTA has read the old lengths (row map, phase 0) and is done
      const InjectArgs a = inject_args(p.inj);
      for (int b = threadIdx.x; b < p.inj.B; b += blockDim.x)
        inject_advance(a, b, p.inj.total_rows,
                       a.draft_window > 0 ? (int64_t)INT32_MAX : (int64_t)a.pages_per_req * a.page_size,
                       p.err);
    }
    if (s_int[0] && p.fin.M > 0) {
      for (int m = threadIdx.x; m < p.fin.M; m += blockDim.x) {
        const int j = m % p.fin.S;
        p.fin.draft_ids[m] = j == 0 ? p.fin.anchor[m / p.fin.S] : argmax_key_index(__ldcg(p.fin.keys + m));
      }
    }
  }
  pdl_trigger();   // every global write of this CTA is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace tc

// ---------------------------------------------------------------------- host
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

// 2D bf16 tensor [rows, cols] (row stride ld elements), box {BK, box_rows}, 128B swizzle.
bool encode_2d(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint64_t ld,
               uint32_t box_rows) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)tc::BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_num_sms = 0;

template <int BN, bool PAIRABLE>
cudaError_t launch_cfg(tc::Params &p, int G, bool coop, cudaStream_t s) {
  using C = tc::Cfg<BN, PAIRABLE>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(tc::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = coop ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, tc::gemm_tc_kernel<BN, PAIRABLE, bf16>, p);
}

template <int BN, bool PAIRABLE>
cudaError_t set_attr() {
  using C = tc::Cfg<BN, PAIRABLE>;
  return cudaFuncSetAttribute(tc::gemm_tc_kernel<BN, PAIRABLE, bf16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
}

int pick_bn(int M) {
  return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}
// Token rows of a tile: a paired phase of a 256-token program uses the SPLIT
// layout's 128-token tiles.
int tile_rows(int BN, bool pair) { return pair && BN == 256 ? 128 : BN; }

bool g_head_pairs = true;

// A QKV GEMM of 128-wide heads in a 256-token program runs as head pairs:
// tiles of two consecutive heads (256 features) by 128 tokens in the SPLIT
// layout, so that the epilogue finds whole head rows in each TMEM lane.
bool head_pairs(const GemmProblem &P, int BN) {
  const EpiParams &e = P.seg[0].epi;
  return g_head_pairs && BN == 256 && P.nseg == 1 && e.op == EPI_QKV && e.head_dim == 128 &&
         P.seg[0].N == e.N && e.N % 256 == 0;
}

// One phase of a program from a problem description; returns its tile count.
bool build_phase(tc::Phase &ph, const GemmProblem &P, int BN, int counter_off) {
  memset(&ph, 0, sizeof(ph));
  if (P.K % tc::BK || P.A.k_per_src % tc::BK) return false;
  const bool swiglu = P.seg[0].epi.op == EPI_SWIGLU;
  const bool hp = head_pairs(P, BN);
  const bool pair = swiglu || hp;
  const int bnt = tile_rows(BN, pair);
  for (int j = 0; j < P.A.n_src; ++j)
    if (!encode_2d(&ph.tmA[j], P.A.ptr[j], (uint64_t)P.M, (uint64_t)P.A.k_per_src, (uint64_t)P.A.ld, bnt))
      return false;
  int ntiles = 0;
  for (int i = 0; i < P.nseg; ++i) {
    const GemmSeg &g = P.seg[i];
    if (!encode_2d(&ph.tmW[i], g.W, (uint64_t)g.N, (uint64_t)P.K, (uint64_t)g.ldw, 128))
      return false;
    ph.epi[i] = g.epi;
    // a gate/up pair: gate rows n0.., up rows N/2 + n0..; a head pair: rows
    // n0 .. n0+255 (tiles 256 features apart)
    const int n = pair ? g.N / 2 : g.N;
    ph.seg_ntiles[i] = (n + 127) / 128;
    ph.seg_half[i] = swiglu ? g.N / 2 : hp ? 128 : 0;
    ntiles += ph.seg_ntiles[i];
  }
  ph.nseg = P.nseg;
  ph.pair = pair ? 1 : 0;
  ph.nstep = hp ? 256 : 128;
  ph.M_dev = P.M_dev;
  ph.nfeat = ntiles;
  ph.M = P.M;
  ph.K = P.K;
  ph.KB = P.K / tc::BK;
  ph.bnt = bnt;
  ph.m_tiles = (P.M + bnt - 1) / bnt;
  ph.tiles = ntiles * ph.m_tiles;
  ph.k_per_src = P.A.k_per_src;
  ph.counter_off = counter_off;
  ph.total_iters = (long long)ph.tiles * ph.KB;
  return true;
}

}  // namespace

// Partial-tile scratch: per CTA two slots of (pair ? 2 : 1) * BN * 128 fp32, at most 256 * 128.
int gemm_tc_trace_slots() { return tc::kTraceSlots; }

void gemm_tc_set_head_pairs(bool on) { g_head_pairs = on; }

size_t gemm_tc_partials_bytes() { return (size_t)kTcMaxCtas * 2 * 256 * 128 * 4; }

int gemm_tc_tiles(int n_tiles, int M, bool pair) {
  const int bnt = tile_rows(pick_bn(M), pair);
  return n_tiles * ((M + bnt - 1) / bnt);
}

int gemm_tc_num_sms() {
  if (!g_num_sms) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 1;
  }
  return g_num_sms;
}

cudaError_t prepare_gemm_tc() {
  cudaError_t e;
#define DFLASH_TC_ATTR(bn, pr) \
  if ((e = set_attr<bn, pr>()) != cudaSuccess) return e;
  DFLASH_TC_ATTR(16, false) DFLASH_TC_ATTR(32, false) DFLASH_TC_ATTR(64, false)
  DFLASH_TC_ATTR(128, false) DFLASH_TC_ATTR(256, false) DFLASH_TC_ATTR(16, true)
  DFLASH_TC_ATTR(32, true) DFLASH_TC_ATTR(64, true) DFLASH_TC_ATTR(128, true)
  DFLASH_TC_ATTR(256, true)
#undef DFLASH_TC_ATTR
  return cudaSuccess;
}

cudaError_t launch_gemm_program(const GemmProblem *probs, int n, float *partials, int *counters,
                                int max_tiles, unsigned int *grid_bar, unsigned int *err,
                                cudaStream_t s, unsigned long long *trace,
                                const ProgramEmbed *embed, const ProgramFinalize *fin,
                                const ProgramInject *inject, const ProgramNorm *norm) {
  const int lead = embed ? 1 : 0;   // the embedding phase comes first
  const int extra = norm ? 1 : 0;   // the normalisation phase comes before the last GEMM
  if (n <= 0 || n > kMaxGemmPhases || n + lead + extra > kMaxPhases) return cudaErrorInvalidValue;
  if ((n + lead + extra > 1 || fin || inject) && !grid_bar) return cudaErrorInvalidValue;
  if (norm && (norm->M != probs[0].M || norm->H % 256 || norm->H <= 0 || !norm->x || !norm->ssq ||
               !norm->gain || !norm->out))
    return cudaErrorInvalidValue;
  if (inject && n + lead < 2) return cudaErrorInvalidValue;   // the map is read by a later phase
  if (embed && (embed->M != probs[0].M || embed->H % 128 || embed->M <= 0))
    return cudaErrorInvalidValue;
  const int M = probs[0].M;
  if (M <= 0) return cudaSuccess;
  const int BN = pick_bn(M);
  bool any_pair = false;
  for (int i = 0; i < n; ++i) {
    if (probs[i].M != M || probs[i].nseg <= 0) return cudaErrorInvalidValue;
    any_pair |= probs[i].seg[0].epi.op == EPI_SWIGLU || head_pairs(probs[i], BN);
  }
  tc::Params p;
  memset(&p, 0, sizeof(p));
  int off = 0;
  long long most = 0;
  if (lead) {
    p.ph[0].nseg = 0;   // no GEMM work: the epilogue warps embed the block
    p.ph[0].M = M;
    p.ph[0].KB = 1;
    p.ph[0].m_tiles = 1;
    p.emb = *embed;
  }
  p.nrm_phase = -1;
  for (int i = 0; i < n; ++i) {
    int k = lead + i;
    if (norm && i == n - 1) {
      // GEMM-free: no tiles, the epilogue warps normalise the rows
      p.ph[k].nseg = 0;
      p.ph[k].M = M;
      p.ph[k].KB = 1;
      p.ph[k].m_tiles = 1;
      p.nrm = *norm;
      p.nrm_phase = k;
      ++k;
    }
    if (!build_phase(p.ph[k], probs[i], BN, off)) return cudaErrorInvalidValue;
    off += p.ph[k].tiles;
    most = std::max(most, p.ph[k].total_iters);
  }
  if (off > max_tiles) return cudaErrorInvalidValue;
  if (fin) p.fin = *fin;
  if (inject) p.inj = *inject;
  n += lead + extra;
  p.nph = n;
  p.partials = partials;
  p.counters = counters;
  p.grid_bar = grid_bar;
  p.err = err;
  p.trace = trace;
  const int G = (int)std::min<long long>(std::min(gemm_tc_num_sms(), kTcMaxCtas), most);
  for (int i = 0; i < n; ++i) {
    tc::Phase &ph = p.ph[i];
    ph.G = (int)std::max<long long>(1, std::min<long long>(G, ph.total_iters));
    // full waves of whole tiles when several token tiles share each weight tile;
    // a tail of fewer than half a wave of tiles would be split many ways
    // (every tail tile merged from many shares at the end of the phase), so
    // the last full wave joins the tail then
    ph.nfull = ph.m_tiles > 1 && ph.nseg > 0 ? ph.tiles / ph.G : 0;
    if (ph.nfull > 0 && 2 * (ph.tiles - ph.nfull * ph.G) < ph.G) --ph.nfull;
  }
  const bool coop = n > 1;
  if (any_pair) {
    switch (BN) {
      case 16: return launch_cfg<16, true>(p, G, coop, s);
      case 32: return launch_cfg<32, true>(p, G, coop, s);
      case 64: return launch_cfg<64, true>(p, G, coop, s);
      case 128: return launch_cfg<128, true>(p, G, coop, s);
      case 256: return launch_cfg<256, true>(p, G, coop, s);
    }
  } else {
    switch (BN) {
      case 16: return launch_cfg<16, false>(p, G, coop, s);
      case 32: return launch_cfg<32, false>(p, G, coop, s);
      case 64: return launch_cfg<64, false>(p, G, coop, s);
      case 128: return launch_cfg<128, false>(p, G, coop, s);
      case 256: return launch_cfg<256, false>(p, G, coop, s);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(const GemmProblem &P, float *partials, int *counters, int max_tiles,
                           unsigned int *err, cudaStream_t s, unsigned long long *trace) {
  if (P.M <= 0 || P.nseg <= 0) return cudaSuccess;
  return launch_gemm_program(&P, 1, partials, counters, max_tiles, nullptr, err, s, trace);
}

}  // namespace dflash
