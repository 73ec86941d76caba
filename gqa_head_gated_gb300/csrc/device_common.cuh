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

// Non-finite V values at keys masked for some rows (both kernels).
// A 16-bit element (bf16 or fp16 bits) that is NaN or +-Inf: exponent all ones.
template <bool kF16>
__device__ __forceinline__ bool elem_nonfinite(uint32_t e) {
  return kF16 ? (e & 0x7C00u) == 0x7C00u : (e & 0x7F80u) == 0x7F80u;
}
template <bool kF16>
__device__ __forceinline__ float elem_to_float(uint32_t e) {
  if constexpr (kF16) return __half2float(__ushort_as_half(static_cast<unsigned short>(e)));
  else return __uint_as_float(e << 16);
}
// Sets the NaN / Inf elements of a 16-byte chunk to +0; returns whether there was one.
template <bool kF16>
__device__ __forceinline__ bool clear_nonfinite(uint4& u) {
  uint32_t w[4] = {u.x, u.y, u.z, u.w};
  bool any = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (elem_nonfinite<kF16>(w[i] & 0xFFFFu)) { w[i] &= 0xFFFF0000u; any = true; }
    if (elem_nonfinite<kF16>(w[i] >> 16)) { w[i] &= 0x0000FFFFu; any = true; }
  }
  u = make_uint4(w[0], w[1], w[2], w[3]);
  return any;
}

// acc + x * 0 on a packed pair (acc starts at +0): stays +0 while every x is finite and
// becomes NaN for good once some x is NaN or +-Inf (Inf * 0 is NaN).
template <bool kF16>
__device__ __forceinline__ uint32_t nonfinite_acc(uint32_t acc, uint32_t x) {
  uint32_t r;
  if constexpr (kF16)
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0u), "r"(acc));
  else
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0u), "r"(acc));
  return r;
}
// The same for one fp32 value.
__device__ __forceinline__ float nonfinite_acc_f32(float acc, float x) {
  float r;
  asm("fma.rn.f32 %0, %1, 0f00000000, %2;" : "=f"(r) : "f"(x), "f"(acc));
  return r;
}

// Logistic function for the output gate, fp32.  The approximate divide has no
// branch to an IEEE slow path, so a thread's 128 gates interleave; its error (a few
// fp32 ulp, like __expf's) is far below the one rounding of the output to bf16/fp16.
// g = -inf or < -88 gives exactly 0 (1/inf), g = +inf gives 1, NaN stays NaN.
__device__ __forceinline__ float gate_sigmoid(float g) {
  return __fdividef(1.0f, 1.0f + __expf(-g));
}

}  // namespace gqa
