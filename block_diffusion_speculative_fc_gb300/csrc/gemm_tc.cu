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
//               ring of shared-memory stages, mbarrier transaction counts.
//   warp 1      TMEM allocator and MMA issuer: tcgen05.mma kind::f16 (bf16 in,
//               fp32 accumulate), tcgen05.commit frees a stage / publishes an
//               accumulator.  Two accumulator buffers let the epilogue of one
//               tile overlap the MMAs of the next.
//   warps 2..5  epilogue: tcgen05.ld to registers, shared-memory staging, the
//               shared epilogue ops (norm/RoPE/scatter, SwiGLU, argmax, ...).
// Work split (stream-K): the flattened (tile, k-block) iteration space is cut
// into gridDim.x equal contiguous ranges.  A tile covered by one CTA is
// finished directly; a tile shared by several CTAs has each write an fp32
// partial, and the last to arrive (atomic ticket, no waiting on other CTAs)
// sums the partials in CTA order -- a fixed order, so results are
// deterministic -- and runs the epilogue.
// Every mbarrier wait is bounded; a wait that gives up raises
// DFLASH_DERR_TIMEOUT and the CTA winds down instead of hanging.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dflash {
namespace tc {

constexpr int BK = 64;            // k elements per stage: one 128-byte swizzle row
constexpr int THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr uint32_t WAIT_LIMIT = 1u << 22;

struct Params {
  CUtensorMap tmA[kMaxSrc];       // activations, box {BK, BN}
  CUtensorMap tmW[kMaxSeg];       // weights, box {BK, 128}
  EpiParams epi[kMaxSeg];
  int seg_ntiles[kMaxSeg];        // 128-feature tiles per segment (pairs count once)
  int seg_half[kMaxSeg];          // pair: row offset of the "up" half
  int nseg;
  int M, K, KB, m_tiles, tiles;
  int k_per_src;
  long long total_iters;
  float *partials;                // [gridDim.x][2][P][BN][128]
  int *counters;                  // [tiles]
  unsigned int *err;
  unsigned long long *trace;      // optional [gridDim.x][8] phase timestamps (ns), test builds only
};

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
__device__ __forceinline__ void stamp(const Params &p, int slot) {
  if (p.trace) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.trace[blockIdx.x * 8 + slot] = t;
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
struct Range {
  long long b, e;
};
__device__ __forceinline__ Range cta_range(long long total, int G, int c) {
  return {total * c / G, total * (c + 1) / G};
}
__device__ __forceinline__ int cta_of_iter(long long it, long long total, int G) {
  return (int)(((it + 1) * G - 1) / total);
}

template <int BN, bool PAIR>
struct Cfg {
  static constexpr int P = PAIR ? 2 : 1;
  static constexpr int W_BYTES = 128 * BK * 2;
  static constexpr int A_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = P * W_BYTES + A_BYTES;
  static constexpr int CH = BN < 32 ? BN : 32;          // epilogue token chunk
  static constexpr int STAGING_BYTES = P * CH * 128 * 4;
  static constexpr int BAR_BYTES = 768 + 1024;   // mbarriers, TMEM slot, flag, epilogue scratch, row scales
  static constexpr int BUDGET = 225 * 1024;
  static constexpr int STAGES_RAW = (BUDGET - 1024 - STAGING_BYTES - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 12 ? 12 : STAGES_RAW;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + BAR_BYTES;
  static constexpr int ACC_COLS = P * BN;                // one accumulator buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS <= 32 ? 32 : (2 * ACC_COLS <= 64 ? 64 :
                                   (2 * ACC_COLS <= 128 ? 128 : (2 * ACC_COLS <= 256 ? 256 : 512)));
  static_assert(STAGES >= 2, "not enough shared memory for two stages");
  static_assert(2 * ACC_COLS <= 512, "accumulators exceed TMEM");
};

template <int BN, bool PAIR, typename T>
__global__ void __launch_bounds__(THREADS, 1) gemm_tc_kernel(const __grid_constant__ Params p) {
  using C = Cfg<BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *stages = smem;
  float *staging = (float *)(smem + C::STAGES * C::STAGE_BYTES);
  uint64_t *bars = (uint64_t *)(smem + C::STAGES * C::STAGE_BYTES + C::STAGING_BYTES);
  uint64_t *full = bars, *empty = bars + C::STAGES;
  uint64_t *acc_full = bars + 2 * C::STAGES, *acc_empty = acc_full + 2;
  uint64_t *mma_done = acc_empty + 2;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  int *flag = (int *)(tmem_slot + 1);
  int *s_int = (int *)((uint8_t *)bars + 256);   // kEpiScratchInts ints
  float *s_rstd = (float *)((uint8_t *)bars + 768);   // [BN] deferred-norm row scales

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const Range R = cta_range(p.total_iters, G, cta);

  if (threadIdx.x == 0) stamp(p, 0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(mma_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.nseg; ++i) prefetch_tmap(&p.tmW[i]);
    for (int i = 0; i < kMaxSrc && i * p.k_per_src < p.K; ++i) prefetch_tmap(&p.tmA[i]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) stamp(p, 1);

  // tile -> (segment, feature tile, token tile)
  auto locate = [&](int tile, int &seg, int &n0, int &m0) {
    int nt = tile / p.m_tiles;
    m0 = (tile % p.m_tiles) * BN;
    seg = 0;
    while (seg < p.nseg - 1 && nt >= p.seg_ntiles[seg]) nt -= p.seg_ntiles[seg++];
    n0 = nt * 128;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      // walk this CTA's (tile, k-block) range incrementally: one division up
      // front, a tile lookup only when the tile changes
      struct Walker {
        long long left;
        int tile, kb, seg, n0, m0, k;
      };
      auto start = [&](Walker &w, long long at) {
        w.left = R.e - at;
        w.tile = (int)(at / p.KB);
        w.kb = (int)(at % p.KB) - 1;
        locate(w.tile, w.seg, w.n0, w.m0);
      };
      auto advance = [&](Walker &w) -> bool {
        if (w.left <= 0) return false;
        --w.left;
        if (++w.kb == p.KB) {
          w.kb = 0;
          ++w.tile;
          locate(w.tile, w.seg, w.n0, w.m0);
        }
        w.k = w.kb * BK;
        return true;
      };
      Walker ld;
      start(ld, R.b);
      int &seg = ld.seg, &n0 = ld.n0, &m0 = ld.m0, &k = ld.k;
      auto next = [&]() -> bool { return advance(ld); };
      auto load_w = [&](int s) {
        uint8_t *st = stages + s * C::STAGE_BYTES;
        mbar_expect_tx(&full[s], C::STAGE_BYTES);
        tma_load_2d(st, &p.tmW[seg], &full[s], k, n0, pol_w);
        if (PAIR) tma_load_2d(st + C::W_BYTES, &p.tmW[seg], &full[s], k, p.seg_half[seg] + n0, pol_w);
      };
      auto load_a = [&](int s, int kk, int mm) {
        const int src = kk / p.k_per_src;
        tma_load_2d(stages + s * C::STAGE_BYTES + C::P * C::W_BYTES, &p.tmA[src], &full[s],
                    kk - src * p.k_per_src, mm, pol_a);
      };
      // Weights do not depend on the previous kernel: fill the whole ring with
      // them first, then wait for the predecessor and add the activations.
      int it = 0;
      int pend_k[C::STAGES], pend_m[C::STAGES];
      while (it < C::STAGES && next()) {
        load_w(it);
        pend_k[it] = k;
        pend_m[it] = m0;
        ++it;
      }
      stamp(p, 2);
      pdl_wait();
      stamp(p, 3);
      for (int j = 0; j < it; ++j) load_a(j, pend_k[j], pend_m[j]);
      bool ok = true;
      while (next()) {
        const int s = it % C::STAGES;
        if (!mbar_wait(&empty[s], ((it / C::STAGES) & 1) ^ 1)) {
          ok = false;
          break;
        }
        load_w(s);
        load_a(s, k, m0);
        ++it;
      }
      if (!ok) raise_error(p.err, DFLASH_DERR_TIMEOUT);
      // drain: no TMA write may still be in flight when the CTA winds down
      for (int j = 0; j < C::STAGES && j < it; ++j) {
        const int q = it - 1 - j;
        mbar_wait(&full[q % C::STAGES], (q / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, BN);
      int it = 0, seg_i = 0;
      bool ok = true;
      for (long long i = R.b; i < R.e && ok; ++seg_i) {
        const int kb0 = (int)(i % p.KB);
        const int kb1 = (int)(kb0 + (R.e - i) < p.KB ? kb0 + (R.e - i) : p.KB);
        const int buf = seg_i & 1;
        const uint32_t aph = (seg_i >> 1) & 1;
        if (!mbar_wait(&acc_empty[buf], aph ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem + buf * C::ACC_COLS;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % C::STAGES;
          if (!mbar_wait(&full[s], (it / C::STAGES) & 1)) {
            ok = false;
            break;
          }
          if (it == 0) stamp(p, 4);
          tc_fence_after();
          const uint32_t st = su32(stages + s * C::STAGE_BYTES);
          const uint64_t bdesc = sw128_desc(st + C::P * C::W_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
            umma_bf16(d0, sw128_desc(st) + 2 * kk, bdesc + 2 * kk, idesc, acc);
            if (PAIR) umma_bf16(d0 + BN, sw128_desc(st + C::W_BYTES) + 2 * kk, bdesc + 2 * kk, idesc, acc);
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&acc_full[buf]);
        i += kb1 - kb0;
      }
      if (!ok) raise_error(p.err, DFLASH_DERR_TIMEOUT);
      // every MMA issued by this thread must be complete before TMEM is freed
      umma_commit(mma_done);
      mbar_wait(mma_done, 0);
      stamp(p, 5);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();                                      // reads the predecessor's outputs
    const int ew = warp - EPI_WARP0;                 // 0..3
    const int tid = ew * 32 + lane;                  // 0..127
    const int quarter = warp & 3;                    // TMEM lane quarter this warp may access
    const int f = quarter * 32 + lane;               // output feature row of this thread
    float *st0 = staging, *st1 = staging + C::CH * 128;
    int seg_i = 0;
    int rstd_m0 = -1, rstd_seg = -1;   // rows whose deferred-norm scales are in s_rstd
    for (long long i = R.b; i < R.e; ++seg_i) {
      const int tile = (int)(i / p.KB);
      const int kb0 = (int)(i % p.KB);
      const int kb1 = (int)(kb0 + (R.e - i) < p.KB ? kb0 + (R.e - i) : p.KB);
      i += kb1 - kb0;
      int seg, n0, m0;
      locate(tile, seg, n0, m0);
      const EpiParams &e = p.epi[seg];
      const int rows = min(BN, p.M - m0);
      const int buf = seg_i & 1;
      const uint32_t aph = (seg_i >> 1) & 1;
      // row scales of a deferred RMSNorm, computed while the MMAs still run
      const bool need_rstd = e.ssq_in != nullptr && (m0 != rstd_m0 || seg != rstd_seg);
      if (need_rstd) {
        epi_bar();   // the previous tile's epilogue is done with s_rstd
        compute_rstd(e, m0, rows, s_rstd, lane, ew, 4);
        rstd_m0 = m0;
        rstd_seg = seg;
      }
      const bool ok = epi_all(mbar_wait(&acc_full[buf], aph));
      if (!ok) {
        if (tid == 0) raise_error(p.err, DFLASH_DERR_TIMEOUT);
        break;
      }
      tc_fence_after();
      if (tid == 0 && seg_i == 0) stamp(p, 6);
      const uint32_t tacc = tmem + ((uint32_t)(quarter * 32) << 16) + buf * C::ACC_COLS;
      const bool whole = kb0 == 0 && kb1 == p.KB;
      if (whole) {
        for (int c0 = 0; c0 < BN; c0 += C::CH) {
          float v[32];
#pragma unroll
          for (int q = 0; q < C::P; ++q) {
            tmem_ld16(tacc + q * BN + c0, v);
            if (C::CH == 32) tmem_ld16(tacc + q * BN + c0 + 16, v + 16);
            float *dst = q ? st1 : st0;
#pragma unroll
            for (int t = 0; t < C::CH; ++t) dst[t * 128 + f] = v[t];
          }
          epi_bar();
          if (c0 < rows)
            run_epilogue<T>(e, st0, PAIR ? st1 : nullptr, 128, m0 + c0, min(C::CH, rows - c0), n0,
                            tid, 128, s_int, [] { epi_bar(); }, s_rstd + c0);
          epi_bar();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else {
        // partial tile: publish this CTA's share, last arriver finishes the tile
        const long long first_tile = R.b / p.KB;
        const int which = tile == first_tile ? 0 : 1;
        float *mine = p.partials + ((size_t)cta * 2 + which) * (C::P * BN * 128);
        for (int c0 = 0; c0 < BN; c0 += C::CH) {
          float v[32];
#pragma unroll
          for (int q = 0; q < C::P; ++q) {
            tmem_ld16(tacc + q * BN + c0, v);
            if (C::CH == 32) tmem_ld16(tacc + q * BN + c0 + 16, v + 16);
#pragma unroll
            for (int t = 0; t < C::CH; ++t) mine[(q * BN + c0 + t) * 128 + f] = v[t];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        __threadfence();
        epi_bar();
        const long long kb_total = p.total_iters;
        const int c_first = cta_of_iter((long long)tile * p.KB, kb_total, G);
        const int c_last = cta_of_iter((long long)(tile + 1) * p.KB - 1, kb_total, G);
        if (tid == 0) {
          const int old = atomicAdd(&p.counters[tile], 1);
          *flag = old == c_last - c_first;
        }
        epi_bar();
        const bool last = *flag != 0;
        if (last) {
          __threadfence();
          for (int c0 = 0; c0 < BN; c0 += C::CH) {
#pragma unroll
            for (int q = 0; q < C::P; ++q) {
              float acc[32];
#pragma unroll
              for (int t = 0; t < C::CH; ++t) acc[t] = 0.f;
              // contributors in CTA order, two at a time so that twice the
              // loads are in flight; the summation order stays fixed
              auto slot_of = [&](int c) {
                const long long cfirst_tile = (p.total_iters * c / G) / p.KB;
                const int w = tile == cfirst_tile ? 0 : 1;
                return p.partials + ((size_t)c * 2 + w) * (C::P * BN * 128) + (q * BN + c0) * 128 + f;
              };
              int c = c_first;
              for (; c < c_last; c += 2) {
                const float *a = slot_of(c), *b2 = slot_of(c + 1);
                float va[32], vb[32];
#pragma unroll
                for (int t = 0; t < C::CH; ++t) {
                  va[t] = __ldcg(a + t * 128);
                  vb[t] = __ldcg(b2 + t * 128);
                }
#pragma unroll
                for (int t = 0; t < C::CH; ++t) acc[t] = (acc[t] + va[t]) + vb[t];
              }
              if (c == c_last) {
                const float *a = slot_of(c);
#pragma unroll
                for (int t = 0; t < C::CH; ++t) acc[t] += __ldcg(a + t * 128);
              }
              float *dst = q ? st1 : st0;
#pragma unroll
              for (int t = 0; t < C::CH; ++t) dst[t * 128 + f] = acc[t];
            }
            epi_bar();
            if (c0 < rows)
              run_epilogue<T>(e, st0, PAIR ? st1 : nullptr, 128, m0 + c0, min(C::CH, rows - c0),
                              n0, tid, 128, s_int, [] { epi_bar(); }, s_rstd + c0);
            epi_bar();
          }
          if (tid == 0) p.counters[tile] = 0;   // ready for the next launch
        }
        epi_bar();
      }
    }
  }
  if (warp == EPI_WARP0 && lane == 0) stamp(p, 7);
  tc_fence_before();
  __syncthreads();
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

template <int BN, bool PAIR>
cudaError_t launch_cfg(tc::Params &p, int G, cudaStream_t s) {
  using C = tc::Cfg<BN, PAIR>;
  auto kern = tc::gemm_tc_kernel<BN, PAIR, bf16>;
  return launch_pdl(kern, dim3(G), dim3(tc::THREADS), C::SMEM, s, p);
}

template <int BN, bool PAIR>
cudaError_t set_attr() {
  using C = tc::Cfg<BN, PAIR>;
  return cudaFuncSetAttribute(tc::gemm_tc_kernel<BN, PAIR, bf16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
}

}  // namespace

// Partial-tile scratch: per CTA two slots of (pair ? 2 : 1) * BN * 128 fp32, at most 256 * 128.
size_t gemm_tc_partials_bytes() { return (size_t)kTcMaxCtas * 2 * 256 * 128 * 4; }

int gemm_tc_tiles(int n_tiles, int M, bool pair) {
  int BN = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  if (pair && BN > 128) BN = 128;
  return n_tiles * ((M + BN - 1) / BN);
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
#undef DFLASH_TC_ATTR
  return cudaSuccess;
}

cudaError_t launch_gemm_tc(const GemmProblem &P, float *partials, int *counters, int max_tiles,
                           unsigned int *err, cudaStream_t s, unsigned long long *trace) {
  if (P.M <= 0 || P.nseg <= 0) return cudaSuccess;
  if (P.K % tc::BK) return cudaErrorInvalidValue;
  const bool pair = P.seg[0].epi.op == EPI_SWIGLU;
  int BN = P.M <= 16 ? 16 : P.M <= 32 ? 32 : P.M <= 64 ? 64 : P.M <= 128 ? 128 : 256;
  if (pair && BN > 128) BN = 128;
  tc::Params p;
  memset(&p, 0, sizeof(p));
  for (int j = 0; j < P.A.n_src; ++j)
    if (!encode_2d(&p.tmA[j], P.A.ptr[j], (uint64_t)P.M, (uint64_t)P.A.k_per_src, (uint64_t)P.A.ld, BN))
      return cudaErrorInvalidValue;
  int ntiles = 0;
  for (int i = 0; i < P.nseg; ++i) {
    const GemmSeg &g = P.seg[i];
    if (!encode_2d(&p.tmW[i], g.W, (uint64_t)g.N, (uint64_t)P.K, (uint64_t)g.ldw, 128))
      return cudaErrorInvalidValue;
    p.epi[i] = g.epi;
    const int n = pair ? g.N / 2 : g.N;
    p.seg_ntiles[i] = (n + 127) / 128;
    p.seg_half[i] = pair ? g.N / 2 : 0;
    ntiles += p.seg_ntiles[i];
  }
  p.nseg = P.nseg;
  p.M = P.M;
  p.K = P.K;
  p.KB = P.K / tc::BK;
  p.m_tiles = (P.M + BN - 1) / BN;
  p.tiles = ntiles * p.m_tiles;
  if (p.tiles > max_tiles) return cudaErrorInvalidValue;
  p.k_per_src = P.A.k_per_src;
  p.total_iters = (long long)p.tiles * p.KB;
  p.partials = partials;
  p.counters = counters;
  p.err = err;
  p.trace = trace;
  const int G = (int)std::min<long long>(std::min(gemm_tc_num_sms(), kTcMaxCtas), p.total_iters);
  switch (BN | (pair ? 1 : 0)) {
    case 16: return launch_cfg<16, false>(p, G, s);
    case 32: return launch_cfg<32, false>(p, G, s);
    case 64: return launch_cfg<64, false>(p, G, s);
    case 128: return launch_cfg<128, false>(p, G, s);
    case 256: return launch_cfg<256, false>(p, G, s);
    case 17: return launch_cfg<16, true>(p, G, s);
    case 33: return launch_cfg<32, true>(p, G, s);
    case 65: return launch_cfg<64, true>(p, G, s);
    case 129: return launch_cfg<128, true>(p, G, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash
