// Device-side helpers shared by the kernels: status word, bounded waits, bf16 packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gqa_attn.h"

namespace gqa {

constexpr int kHeadDim = 256;
// log2(e) / 16: folds the 1/sqrt(256) score scale into the base-2 exponent.
constexpr float kScaleLog2 = 1.4426950408889634f / 16.0f;
constexpr float kLn2 = 0.6931471805599453f;

// Per-launch settings every kernel receives by value.
struct LaunchCtl {
  int* status;                   // device status word (first error wins)
  unsigned long long timeout_ns; // bound on each spin wait
};

__device__ __forceinline__ void record_status(int* status, int code) {
  atomicCAS(status, GQA_OK, code);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_half2(uint32_t u) {
  __half2 v = *reinterpret_cast<__half2*>(&u);
  return __half22float2(v);
}

// Two 16-bit elements of the kernels' element type (fp16 or bf16) <-> float2.
template <bool kF16>
__device__ __forceinline__ uint32_t pack_elem2(float lo, float hi) {
  if constexpr (kF16) return pack_half2(lo, hi); else return pack_bf16x2(lo, hi);
}
template <bool kF16>
__device__ __forceinline__ float2 unpack_elem2(uint32_t u) {
  if constexpr (kF16) return unpack_half2(u); else return unpack_bf16x2(u);
}

// Logistic function for the output gate, fp32.  The approximate divide has no
// branch to an IEEE slow path, so a thread's 128 gates interleave; its error (a few
// fp32 ulp, like __expf's) is far below the one rounding of the output to bf16/fp16.
// g = -inf or < -88 gives exactly 0 (1/inf), g = +inf gives 1, NaN stays NaN.
__device__ __forceinline__ float gate_sigmoid(float g) {
  return __fdividef(1.0f, 1.0f + __expf(-g));
}

}  // namespace gqa
