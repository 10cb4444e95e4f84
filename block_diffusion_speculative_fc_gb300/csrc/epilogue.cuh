// GEMM epilogues shared by every GEMM kernel of the library.
//
// A GEMM hands over an fp32 tile Y[r][c] (r = token row m0 + r, c = output
// feature n0 + c, 128 features wide, at most 32 rows) staged in shared
// memory; the epilogue turns it into the step's output:
//   EPI_QKV       per-head RMSNorm of q and k, RoPE of q and k, plain v
//                 ("Inside SGLang", Step 4: DFlashAttention computes block
//                 Q/K/V, normalizes Q/K, applies RoPE).
//   EPI_KV_CACHE  k-norm and RoPE of k, plain v, written to the paged cache
//                 row of each context row (CSDN DFlash article,
//                 "fused_kv_materialize": K RMSNorm + K RoPE + V relayout
//                 for all layers, heads and tokens).
//   EPI_SWIGLU    silu(gate) * up of a paired gate/up tile.
//   EPI_ARGMAX    greedy token choice without materialising logits.
//   EPI_TOPK      the K best tokens of every row, per 128-token tile (DFlash 2
//                 candidates), again without materialising logits.
//   EPI_RESID / EPI_STORE_*  residual add / plain stores.
// The tile is tiny and sits on the critical path of short launches, so every
// op issues its global loads in batches before using them (one memory round
// trip per batch rather than one per element).
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace dflash {

constexpr int kEpiMaxRows = 32;

// Bring a line into L1 ahead of its use: the epilogues touch a row of global
// memory per item, and issuing every line of a chunk first turns one memory
// round trip per item into one per chunk, with no registers held meanwhile.
__device__ __forceinline__ void prefetch_l1(const void *p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Rotate-half RoPE on one head held by a warp (component i pairs with
// i + D/2), optionally preceded by a per-head RMSNorm.  g_lo/g_hi: this lane's
// gains for i = lane + 32k and i + D/2; cs: this lane's (cos, sin).
template <typename T, int NP>
__device__ __forceinline__ void head_epilogue(const float *src, int D, bool norm, bool rope,
                                              const float *g_lo, const float *g_hi, float eps,
                                              const float2 *cs, T *dst, int lane) {
  const int half = D >> 1;
  float lo[NP], hi[NP];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const int i = lane + 32 * k;
    lo[k] = i < half ? src[i] : 0.f;
    hi[k] = i < half ? src[i + half] : 0.f;
    ss += lo[k] * lo[k] + hi[k] * hi[k];
  }
  float rstd = 1.f;
  if (norm) {
    ss = warp_sum(ss);
    rstd = rsqrtf(ss / (float)D + eps);
  }
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const int i = lane + 32 * k;
    if (i >= half) continue;
    float a = lo[k], b = hi[k];
    if (norm) {
      a *= rstd * g_lo[k];
      b *= rstd * g_hi[k];
    }
    if (rope) {
      const float x = a * cs[k].x - b * cs[k].y;
      const float y = b * cs[k].x + a * cs[k].y;
      a = x;
      b = y;
    }
    dst[i] = from_f32<T>(a);
    dst[i + half] = from_f32<T>(b);
  }
}

// Per-head epilogues for D = 64 * NP.  One warp per (row, head) item; row
// positions / cache slots come from shared memory, gains are loaded once.
template <typename T, int NP, class Sync>
__device__ void head_ops(const EpiParams &e, const float *t0, int ldt, int m0, int rows, int n0,
                         int lane, int warp, int nwarps, const int *s_pos, const int *s_slot,
                         Sync sync) {
  const int D = e.head_dim;
  const int hpt = 128 / D;
  const int kvd = e.n_kv_heads * D;
  const bool qkv = e.op == EPI_QKV;
  for (int item = warp; item < rows * hpt; item += nwarps) {
    const int r = item / hpt, hh = item % hpt;
    const int f0 = n0 + hh * D;
    if (f0 >= e.N) continue;
    const int m = m0 + r;
    const int hg = f0 / D;
    // kind: 0 = q, 1 = k, 2 = v
    int kind, head;
    if (qkv) {
      kind = hg < e.n_heads ? 0 : (hg < e.n_heads + e.n_kv_heads ? 1 : 2);
      head = kind == 0 ? hg : (kind == 1 ? hg - e.n_heads : hg - e.n_heads - e.n_kv_heads);
    } else {
      kind = hg < e.n_kv_heads ? 1 : 2;
      head = kind == 1 ? hg : hg - e.n_kv_heads;
    }
    T *dst;
    if (qkv) {
      dst = kind == 0 ? (T *)e.q_out + (int64_t)m * e.n_heads * D + head * D
                      : (T *)(kind == 1 ? e.k_out : e.v_out) + (int64_t)m * kvd + head * D;
    } else {
      const int slot = s_slot[r];
      if (slot < 0) continue;
      dst = (T *)(kind == 1 ? e.k_cache : e.v_cache) + (int64_t)slot * kvd + head * D;
    }
    const bool nr = kind != 2;
    float g_lo[NP], g_hi[NP];
    float2 cs[NP];
    if (nr) {
      const T *gain = (const T *)(kind == 0 ? e.q_gain : e.k_gain);
      const float2 *rope_row = e.rope + (int64_t)s_pos[r] * (D >> 1);
#pragma unroll
      for (int k = 0; k < NP; ++k) {
        const int i = lane + 32 * k;
        g_lo[k] = to_f32(gain[i]);
        g_hi[k] = to_f32(gain[i + (D >> 1)]);
        cs[k] = rope_row[i];
      }
    }
    head_epilogue<T, NP>(t0 + r * ldt + hh * D, D, nr, nr, g_lo, g_hi, e.eps, cs, dst, lane);
  }
  (void)sync;
}

// The per-head epilogues for D = 128 with wide accesses: a tile is one head,
// a half-warp takes a row, lane l owns elements 4l..4l+3 and their rotary
// partners 64+4l..64+4l+3 (8-byte stores), and the head's RMSNorm reduces
// over the 16 lanes.  Same arithmetic as head_epilogue.
template <typename T>
__device__ void head_ops_d128(const EpiParams &e, const float *t0, int ldt, int m0, int rows,
                              int n0, int lane, int warp, int nwarps, const int *s_pos,
                              const int *s_slot, const float *rs) {
  if (n0 >= e.N) return;
  const int kvd = e.n_kv_heads * 128;
  const bool qkv = e.op == EPI_QKV;
  const int hg = n0 >> 7;
  int kind, head;
  if (qkv) {
    kind = hg < e.n_heads ? 0 : (hg < e.n_heads + e.n_kv_heads ? 1 : 2);
    head = kind == 0 ? hg : (kind == 1 ? hg - e.n_heads : hg - e.n_heads - e.n_kv_heads);
  } else {
    kind = hg < e.n_kv_heads ? 1 : 2;
    head = kind == 1 ? hg : hg - e.n_kv_heads;
  }
  const bool nr = kind != 2;
  const int hl = lane & 15, hw = lane >> 4;
  float glo[4] = {1.f, 1.f, 1.f, 1.f}, ghi[4] = {1.f, 1.f, 1.f, 1.f};
  if (nr) {
    const T *gain = (const T *)(kind == 0 ? e.q_gain : e.k_gain);
    const uint2 a = *reinterpret_cast<const uint2 *>(gain + 4 * hl);
    const uint2 b = *reinterpret_cast<const uint2 *>(gain + 64 + 4 * hl);
    const T *pa = reinterpret_cast<const T *>(&a), *pb = reinterpret_cast<const T *>(&b);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      glo[k] = to_f32(pa[k]);
      ghi[k] = to_f32(pb[k]);
    }
  }
  // the RoPE rows of this warp's rows (512 bytes each, four lines) go to L1
  // before any is used
  if (nr && (hl & 3) == 0)
    for (int r = 2 * warp + hw; r < rows; r += 2 * nwarps)
      prefetch_l1(e.rope + (int64_t)s_pos[r] * 64 + 4 * hl);
  // whole warps iterate together (the norm shuffles over 16 lanes)
  for (int rb = 2 * warp; rb < rows; rb += 2 * nwarps) {
    const int r = rb + hw;
    const bool act = r < rows;
    float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f};
    if (act) {
      const float4 a = *reinterpret_cast<const float4 *>(t0 + r * ldt + 4 * hl);
      const float4 b = *reinterpret_cast<const float4 *>(t0 + r * ldt + 64 + 4 * hl);
      const float sc = rs ? rs[r] : 1.f;   // the deferred RMSNorm's row scale
      lo[0] = a.x * sc; lo[1] = a.y * sc; lo[2] = a.z * sc; lo[3] = a.w * sc;
      hi[0] = b.x * sc; hi[1] = b.y * sc; hi[2] = b.z * sc; hi[3] = b.w * sc;
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) ss += lo[k] * lo[k] + hi[k] * hi[k];
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (!act) continue;
    const int m = m0 + r;
    T *dst;
    int64_t cache_off = 0;   // element offset of this head row in the cache
    if (qkv) {
      dst = kind == 0 ? (T *)e.q_out + (int64_t)m * e.n_heads * 128 + head * 128
                      : (T *)(kind == 1 ? e.k_out : e.v_out) + (int64_t)m * kvd + head * 128;
    } else {
      const int slot = s_slot[r];
      if (slot < 0) continue;
      cache_off = (int64_t)slot * kvd + head * 128;
      dst = (T *)(kind == 1 ? e.k_cache : e.v_cache) + cache_off;
    }
    if (nr) {
      const float rstd = rsqrtf(ss / 128.f + e.eps);
      const float4 *rope = reinterpret_cast<const float4 *>(e.rope + (int64_t)s_pos[r] * 64 + 4 * hl);
      const float4 c01 = rope[0], c23 = rope[1];   // (cos, sin) of elements 4l .. 4l+3
      const float cs_c[4] = {c01.x, c01.z, c23.x, c23.z}, cs_s[4] = {c01.y, c01.w, c23.y, c23.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = lo[k] * rstd * glo[k], b = hi[k] * rstd * ghi[k];
        lo[k] = a * cs_c[k] - b * cs_s[k];
        hi[k] = b * cs_c[k] + a * cs_s[k];
      }
    }
    if (!qkv && e.kv_fp8) {
      // FP8 E4M3 cache (CSDN article, Kimi-K2.6 draft card: one byte per
      // K/V element): the code of x / scale, four bytes per store
      const float sc = kind == 1 ? e.k_scale : e.v_scale;
      uint8_t *d8 = (uint8_t *)(kind == 1 ? e.k_cache : e.v_cache) + cache_off;
      *reinterpret_cast<uint32_t *>(d8 + 4 * hl) =
          e4m3x2(lo[0], lo[1], sc) | (e4m3x2(lo[2], lo[3], sc) << 16);
      *reinterpret_cast<uint32_t *>(d8 + 64 + 4 * hl) =
          e4m3x2(hi[0], hi[1], sc) | (e4m3x2(hi[2], hi[3], sc) << 16);
      continue;
    }
    uint2 plo, phi;
    T *ql = reinterpret_cast<T *>(&plo), *qh = reinterpret_cast<T *>(&phi);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      ql[k] = from_f32<T>(lo[k]);
      qh[k] = from_f32<T>(hi[k]);
    }
    *reinterpret_cast<uint2 *>(dst + 4 * hl) = plo;
    *reinterpret_cast<uint2 *>(dst + 64 + 4 * hl) = phi;
  }
}

// t0: fp32 tile [rows][ldt] (features n0 .. n0+127); t1: the "up" tile of a
// SwiGLU pair.  All `nthreads` threads of the caller take part (a multiple of
// 128); the caller synchronises before (tile complete) and after (tile reuse).
// The tiles may be modified in place.  s_int: shared scratch of at least
// kEpiScratchInts ints; sync(): barrier over the participating threads.
constexpr int kEpiScratchInts = 3 * kEpiMaxRows;

// Row scales 1/sqrt(sum_t ssq[t][m] / H + eps) of the deferred RMSNorm for
// rows m0 .. m0+rows-1 into rstd[0..rows): a thread per row, the slots of a
// row summed in four interleaved chains, every load issued before the sums
// (consecutive threads read consecutive rows of a slot: coalesced).
__device__ __forceinline__ void compute_rstd(const EpiParams &e, int m0, int rows, float *rstd,
                                             int lane, int warp, int nwarps) {
  const int nthr = nwarps * 32;
  for (int r = warp * 32 + lane; r < rows; r += nthr) {
    const float *p = e.ssq_in + m0 + r;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    int q = 0;
#pragma unroll 8
    for (; q + 4 <= e.ssq_parts; q += 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) a[k] += p[(int64_t)(q + k) * e.ssq_ld];
    }
    for (; q < e.ssq_parts; ++q) a[0] += p[(int64_t)q * e.ssq_ld];
    rstd[r] = rsqrtf(((a[0] + a[1]) + (a[2] + a[3])) * e.inv_h + e.norm_eps);
  }
}

// Element-wise epilogues with wide accesses: a thread takes 8 consecutive
// features of one row (16-byte stores of bf16, two float4 of fp32), and the
// per-row sum of squares of the fused-norm ops reduces over the 16 lanes that
// share the row.  Applies to whole 128-feature tiles whose rows are 16-byte
// aligned; returns false (scalar path) otherwise.  Same arithmetic and output
// as the scalar path.
template <typename T>
__device__ __forceinline__ bool elementwise_vec(const EpiParams &e, const float *t0,
                                                const float *t1, int ldt, int m0, int rows,
                                                int n0, int tid, int nthreads, const float *rs) {
  const int op = e.op;
  if (op != EPI_STORE_F32 && op != EPI_RESID && op != EPI_STORE_ACT && op != EPI_SWIGLU &&
      op != EPI_RESID_NORM && op != EPI_STORE_NORM)
    return false;
  const int nvalid = op == EPI_SWIGLU ? e.N / 2 : e.N;
  const bool f32_out = op == EPI_STORE_F32 || op == EPI_RESID || op == EPI_RESID_NORM;
  const bool act_out = op == EPI_STORE_ACT || op == EPI_SWIGLU || op == EPI_RESID_NORM ||
                       op == EPI_STORE_NORM;
  const bool norm_out = op == EPI_RESID_NORM || op == EPI_STORE_NORM;
  if (sizeof(T) != 2) return false;   // bf16 outputs (the tensor-core path)
  if (n0 + 128 > nvalid || (e.ld & 7) || (nthreads & 31) || (ldt & 3)) return false;
  if (f32_out && ((uintptr_t)e.out_f32 & 15)) return false;
  if (act_out && ((uintptr_t)e.out_act & 15)) return false;
  if (norm_out && ((uintptr_t)e.norm_gain & 15)) return false;
  const int total = rows << 4;
  const int lane = tid & 31;
  if (op == EPI_RESID || op == EPI_RESID_NORM)   // residual rows to L1 first (4 items a line)
    for (int it = tid; it < total; it += nthreads)
      if ((it & 3) == 0)
        prefetch_l1(e.out_f32 + (int64_t)(m0 + (it >> 4)) * e.ld + n0 + ((it & 15) << 3));
  // whole warps iterate together (the row reduction shuffles); an item past
  // the end belongs to a 16-lane group that is past the end as a whole
  for (int it = tid; it - lane < total; it += nthreads) {
    const bool act = it < total;
    const int r = it >> 4, c8 = (it & 15) << 3;
    float ss = 0.f;
    if (act) {
      const float4 *src = reinterpret_cast<const float4 *>(t0 + r * ldt + c8);
      const float4 a = src[0], b = src[1];
      float y[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      const float sc = rs ? rs[r] : 1.f;   // the deferred RMSNorm's row scale
#pragma unroll
      for (int k = 0; k < 8; ++k) y[k] *= sc;
      const int64_t o = (int64_t)(m0 + r) * e.ld + n0 + c8;
      if (op == EPI_SWIGLU) {
        const float4 *u = reinterpret_cast<const float4 *>(t1 + r * ldt + c8);
        const float4 ua = u[0], ub = u[1];
        const float up[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = silu(y[k]) * (up[k] * sc);
      }
      if (op == EPI_RESID || op == EPI_RESID_NORM) {
        const float4 *old = reinterpret_cast<const float4 *>(e.out_f32 + o);
        const float4 oa = old[0], ob = old[1];
        y[0] += oa.x; y[1] += oa.y; y[2] += oa.z; y[3] += oa.w;
        y[4] += ob.x; y[5] += ob.y; y[6] += ob.z; y[7] += ob.w;
      }
      if (f32_out) {
        float4 *dst = reinterpret_cast<float4 *>(e.out_f32 + o);
        dst[0] = make_float4(y[0], y[1], y[2], y[3]);
        dst[1] = make_float4(y[4], y[5], y[6], y[7]);
      }
      if (act_out) {
        float z[8];
        if (norm_out) {
          const uint4 graw = *reinterpret_cast<const uint4 *>((const T *)e.norm_gain + n0 + c8);
          const T *g = reinterpret_cast<const T *>(&graw);
#pragma unroll
          for (int k = 0; k < 8; ++k) z[k] = y[k] * to_f32(g[k]);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) z[k] = y[k];
        }
        uint4 packed;
        T *pk = reinterpret_cast<T *>(&packed);
#pragma unroll
        for (int k = 0; k < 8; ++k) pk[k] = from_f32<T>(z[k]);
        *reinterpret_cast<uint4 *>((T *)e.out_act + o) = packed;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) ss += y[k] * y[k];
    }
    if (norm_out) {
      // sum of squares of this row's 128 features over the 16 lanes of the
      // row (every lane of the warp takes part in the shuffles)
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (act && (it & 15) == 0) e.ssq_out[(int64_t)(n0 >> 7) * e.ssq_ld + m0 + r] = ss;
    }
  }
  return true;
}

template <typename T, class Sync>
__device__ void run_epilogue(const EpiParams &e, float *t0, float *t1, int ldt, int m0, int rows,
                             int n0, int tid, int nthreads, int *s_int, Sync sync,
                             const float *rstd_pre = nullptr) {
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  // deferred RMSNorm of the A operand: every row scales by its rstd
  // (rstd_pre: row scales the caller already computed, indexed from m0).
  // The wide element-wise and per-head paths apply it as they read the tile;
  // the others scale the tile in place first.
  const float *rs = nullptr;
  if (e.ssq_in) {
    rs = rstd_pre;
    if (!rs) {
      float *s_rstd = reinterpret_cast<float *>(s_int + 2 * kEpiMaxRows);
      compute_rstd(e, m0, rows, s_rstd, lane, warp, nwarps);
      sync();
      rs = s_rstd;
    }
  }
  if (elementwise_vec<T>(e, t0, t1, ldt, m0, rows, n0, tid, nthreads, rs)) return;
  const bool heads = e.op == EPI_QKV || e.op == EPI_KV_CACHE;
  const bool wide = sizeof(T) == 2 && (ldt & 3) == 0 && (nthreads & 31) == 0 &&
                    ((uintptr_t)e.q_gain & 7) == 0 && ((uintptr_t)e.k_gain & 7) == 0;
  const bool heads_wide = heads && e.head_dim == 128 && wide;
  if (rs && !heads_wide) {
    for (int idx = tid; idx < rows * 128; idx += nthreads) {
      const int r = idx >> 7, c = idx & 127;
      t0[r * ldt + c] *= rs[r];
      if (t1) t1[r * ldt + c] *= rs[r];
    }
    sync();
  }
  switch (e.op) {
    case EPI_STORE_F32:
    case EPI_RESID:
    case EPI_STORE_ACT:
    case EPI_SWIGLU:
    case EPI_RESID_NORM:
    case EPI_STORE_NORM: {
      const int nvalid = e.op == EPI_SWIGLU ? e.N / 2 : e.N;
      const int c = tid & 127, rg = tid >> 7, ng = nthreads >> 7;
      const int n = n0 + c;
      const bool norm_out = e.op == EPI_RESID_NORM || e.op == EPI_STORE_NORM;
      const float g = (norm_out && n < nvalid) ? to_f32(((const T *)e.norm_gain)[n]) : 0.f;
      constexpr int BATCH = 16;
      if (n < nvalid) {
        for (int rb = rg; rb < rows; rb += BATCH * ng) {
          float y[BATCH];
#pragma unroll
          for (int k = 0; k < BATCH; ++k) {
            const int r = rb + k * ng;
            y[k] = r < rows ? t0[r * ldt + c] : 0.f;
          }
          if (e.op == EPI_RESID || e.op == EPI_RESID_NORM) {
            float old[BATCH];
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
              const int r = rb + k * ng;
              old[k] = r < rows ? e.out_f32[(int64_t)(m0 + r) * e.ld + n] : 0.f;
            }
#pragma unroll
            for (int k = 0; k < BATCH; ++k) y[k] += old[k];
          }
#pragma unroll
          for (int k = 0; k < BATCH; ++k) {
            const int r = rb + k * ng;
            if (r >= rows) continue;
            const int64_t o = (int64_t)(m0 + r) * e.ld + n;
            switch (e.op) {
              case EPI_STORE_F32:
              case EPI_RESID:
                e.out_f32[o] = y[k];
                break;
              case EPI_STORE_ACT:
                ((T *)e.out_act)[o] = from_f32<T>(y[k]);
                break;
              case EPI_SWIGLU:
                ((T *)e.out_act)[o] = from_f32<T>(silu(y[k]) * t1[r * ldt + c]);
                break;
              case EPI_RESID_NORM:
                e.out_f32[o] = y[k];
                ((T *)e.out_act)[o] = from_f32<T>(y[k] * g);
                t0[r * ldt + c] = y[k] * y[k];
                break;
              case EPI_STORE_NORM:
                ((T *)e.out_act)[o] = from_f32<T>(y[k] * g);
                t0[r * ldt + c] = y[k] * y[k];
                break;
            }
          }
        }
      }
      if (norm_out) {
        // per-row sum of squares of the 128 features of this tile
        sync();
        for (int r = warp; r < rows; r += nwarps) {
          float v = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int cc = lane + 32 * k;
            v += (n0 + cc < nvalid) ? t0[r * ldt + cc] : 0.f;
          }
          v = warp_sum(v);
          if (lane == 0) e.ssq_out[(int64_t)(n0 >> 7) * e.ssq_ld + m0 + r] = v;
        }
      }
      break;
    }
    case EPI_ARGMAX: {
      for (int r = warp; r < rows; r += nwarps) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = lane + 32 * k, n = n0 + c;
          if (n < e.N) {
            const unsigned long long key = argmax_key(t0[r * ldt + c], n);
            best = key > best ? key : best;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
          best = other > best ? other : best;
        }
        if (lane == 0 && best) atomicMax(e.argmax_keys + m0 + r, best);
      }
      break;
    }
    case EPI_TOPK: {
      // per row: the tile's topk best keys by topk rounds of a warp max over
      // the 128 features (four per lane, sorted first); a row whose best key in
      // this tile is below its running bound contributes nothing, which after
      // the first tiles is almost every row.  Keys are unique (the id is part
      // of the key), so one lane wins each round.
      const int K = e.topk;
      const int tile = n0 >> 7;
      unsigned long long *base = e.topk_keys + (size_t)tile * e.topk_ld * K;
      // A row's running lower bound of its K-th best key over the whole
      // vocabulary: K slots per row, slot s the best key of the tiles t with
      // t % K == s seen so far; the smallest slot is reached by K distinct
      // keys, so it bounds the K-th best (0 while a slot is empty).  The
      // slots of this warp's rows are read at once (lane i: the warp's i-th
      // row; rows <= 32 per call).
      const int r_l = warp + nwarps * lane;
      unsigned long long my_bound = 0ull;
      if (r_l < rows) {
        my_bound = ~0ull;
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
          if (sl < K) {
            const unsigned long long v =
                *(volatile const unsigned long long *)(e.topk_bound + (size_t)sl * e.topk_ld + m0 + r_l);
            my_bound = v < my_bound ? v : my_bound;
          }
        }
      }
      for (int r = warp, i_row = 0; r < rows; r += nwarps, ++i_row) {
        unsigned long long k0, k1, k2, k3;
        {
          const int n = n0 + lane;
          k0 = n < e.N ? argmax_key(t0[r * ldt + lane], n) : 0ull;
          k1 = n + 32 < e.N ? argmax_key(t0[r * ldt + lane + 32], n + 32) : 0ull;
          k2 = n + 64 < e.N ? argmax_key(t0[r * ldt + lane + 64], n + 64) : 0ull;
          k3 = n + 96 < e.N ? argmax_key(t0[r * ldt + lane + 96], n + 96) : 0ull;
        }
        auto order = [](unsigned long long &a, unsigned long long &b) {
          if (a < b) {
            const unsigned long long t = a;
            a = b;
            b = t;
          }
        };
        order(k0, k1);
        order(k2, k3);
        order(k0, k2);
        order(k1, k3);
        order(k1, k2);
        const int m = m0 + r;
        const unsigned long long bound = __shfl_sync(0xffffffffu, my_bound, i_row & 31);
        unsigned long long mine_out = 0ull, top1 = 0ull;
        int head = 0;
        for (int j = 0; j < K; ++j) {
          const unsigned long long mine = head == 0 ? k0 : head == 1 ? k1 : head == 2 ? k2
                                          : head == 3 ? k3 : 0ull;
          unsigned long long best = mine;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
          }
          if (j == 0 && best < bound) break;   // uniform across the warp
          if (best != 0ull && mine == best) ++head;
          if (lane == j) mine_out = best;
          if (j == 0) top1 = best;
        }
        // lanes below topk write the row's list (zeros past a short list or a skipped row)
        if (lane < K) base[(size_t)m * K + lane] = mine_out;
        if (lane == 0 && top1 != 0ull) atomicMax(e.topk_bound + (size_t)(tile % K) * e.topk_ld + m, top1);
      }
      break;
    }
    case EPI_QKV:
    case EPI_KV_CACHE: {
      int *s_pos = s_int, *s_slot = s_int + kEpiMaxRows;   // after s_rstd was consumed
      for (int r = tid; r < rows; r += nthreads) {
        s_pos[r] = e.row_pos[m0 + r];
        s_slot[r] = e.op == EPI_KV_CACHE ? e.row_slot[m0 + r] : 0;
      }
      sync();
      if (heads_wide)
        head_ops_d128<T>(e, t0, ldt, m0, rows, n0, lane, warp, nwarps, s_pos, s_slot, rs);
      else if (e.head_dim == 128)
        head_ops<T, 2>(e, t0, ldt, m0, rows, n0, lane, warp, nwarps, s_pos, s_slot, sync);
      else
        head_ops<T, 1>(e, t0, ldt, m0, rows, n0, lane, warp, nwarps, s_pos, s_slot, sync);
      sync();
      break;
    }
    default:
      break;
  }
}

}  // namespace dflash
