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

// Logistic function for the output gate, fp32: 1 / (1 + 2^(-g log2 e)), from the
// approximate flush-to-zero ex2 and rcp instructions directly (one multiply, one
// add, two multi-function-unit operations, no range fix-ups), so a thread's 128
// gates interleave and the gate epilogue issues few instructions.  Its error (a few
// fp32 ulp, from the two approximations) is far below the one rounding of the output
// to bf16 / fp16.  g = +inf gives 1 (2^-inf = 0); g = -inf, or g below about -87.3,
// gives 0 (1 + 2^x >= 2^126, whose reciprocal is below fp32's smallest normal and is
// flushed); a NaN gate stays NaN.
__device__ __forceinline__ float gate_sigmoid(float g) {
  float e, s;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(g * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(s) : "f"(1.0f + e));
  return s;
}

// Two gates at once, with the multiplies and adds as packed fp32 pairs (the same
// per-element operations as gate_sigmoid).
__device__ __forceinline__ float2 gate_sigmoid2(float g0, float g1) {
  float s0, s1;
  asm("{\n\t"
      ".reg .b64 x, c, d;\n\t"
      ".reg .f32 x0, x1, e0, e1;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 c, {%4, %4};\n\t"
      "mul.rn.f32x2 x, x, c;\n\t"
      "mov.b64 {x0, x1}, x;\n\t"
      "ex2.approx.ftz.f32 e0, x0;\n\t"
      "ex2.approx.ftz.f32 e1, x1;\n\t"
      "mov.b64 x, {e0, e1};\n\t"
      "mov.b64 c, {%5, %5};\n\t"
      "add.rn.f32x2 d, x, c;\n\t"
      "mov.b64 {x0, x1}, d;\n\t"
      "rcp.approx.ftz.f32 %0, x0;\n\t"
      "rcp.approx.ftz.f32 %1, x1;\n\t"
      "}" : "=f"(s0), "=f"(s1) : "f"(g0), "f"(g1), "f"(-1.4426950408889634f), "f"(1.0f));
  return make_float2(s0, s1);
}

// (a.x * b.x + c.x, a.y * b.y + c.y) as one packed fp32 fma.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float x, y;
  asm("{\n\t"
      ".reg .b64 pa, pb, pc;\n\t"
      "mov.b64 pa, {%2, %3};\n\t"
      "mov.b64 pb, {%4, %5};\n\t"
      "mov.b64 pc, {%6, %7};\n\t"
      "fma.rn.f32x2 pa, pa, pb, pc;\n\t"
      "mov.b64 {%0, %1}, pa;\n\t"
      "}" : "=f"(x), "=f"(y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return make_float2(x, y);
}

// (a.x + b.x, a.y + b.y) as one packed fp32 add.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float x, y;
  asm("{\n\t"
      ".reg .b64 pa, pb;\n\t"
      "mov.b64 pa, {%2, %3};\n\t"
      "mov.b64 pb, {%4, %5};\n\t"
      "add.rn.f32x2 pa, pa, pb;\n\t"
      "mov.b64 {%0, %1}, pa;\n\t"
      "}" : "=f"(x), "=f"(y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return make_float2(x, y);
}

// (a.x * b.x, a.y * b.y) as one packed fp32 multiply.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float x, y;
  asm("{\n\t"
      ".reg .b64 p, q;\n\t"
      "mov.b64 p, {%2, %3};\n\t"
      "mov.b64 q, {%4, %5};\n\t"
      "mul.rn.f32x2 p, p, q;\n\t"
      "mov.b64 {%0, %1}, p;\n\t"
      "}" : "=f"(x), "=f"(y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return make_float2(x, y);
}

}  // namespace gqa
