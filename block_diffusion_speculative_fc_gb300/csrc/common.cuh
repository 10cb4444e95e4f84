// Shared device helpers of the DFlash CUDA library (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/dflash.h"

namespace dflash {

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ void raise_error(unsigned int *err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// Argmax key: the order-preserving image of the fp32 logit in the high word
// and the bitwise complement of the index in the low word, so that an
// unsigned 64-bit max picks the largest logit and, among equal logits, the
// lowest index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  unsigned int u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned int)(~(unsigned int)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(~(unsigned int)(k & 0xffffffffull));
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

// Two OCP FP8 E4M3 codes of lo / scale and hi / scale (IEEE float32 division)
// packed little-endian (lo in the low byte): nearest code, ties to the even
// code, magnitudes beyond 448 saturate to +-448 (the hardware conversion's
// round-to-nearest-even with .satfinite).
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi, float scale) {
  const float a = __fdiv_rn(lo, scale), b = __fdiv_rn(hi, scale);
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Programmatic dependent launch.  Every kernel is launched so that it may be
// scheduled before its predecessor in the stream has exited.  A kernel waits
// for its predecessor (griddepcontrol.wait) right before it first reads what
// the predecessor wrote; only writes a CTA made before it signals its
// dependents (griddepcontrol.launch_dependents) are covered by that wait, so
// each kernel signals only after its last global write (or not at all, which
// signals at exit).  Work that does not depend on the predecessor -- above
// all the GEMM weight stream -- runs before the wait.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace dflash
