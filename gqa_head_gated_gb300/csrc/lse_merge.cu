// attn_lse_merge: combine S partial attention results of the same rows computed
// over disjoint key sets, then apply the sigmoid output gate and round to bf16
// (or fp16: the gate and output element type is a template flag).
//
//   out[n,:] = sum_s exp(lse_s - M) O_s[n,:] / sum_s exp(lse_s - M) * sigmoid(G[n,:])
//   lse[n]   = M + ln sum_s exp(lse_s - M),   M = max_s lse_s
//
// This is the tail-chunk merge of the TensorFold PR #1009 attention contract
// ("Receipt": decode over cache chunks, then a merge; its control "a merge
// dropping later tail chunks" must fail).  Parts with lse = -inf carry weight 0
// and their O rows are never read.  A NaN lse (a part that saw a NaN score)
// makes the row NaN, as float64 arithmetic of the formula would.  One warp per
// row; each lane owns 8 of the 256 columns and reads them as two float4 per part,
// the loads of sixteen parts issued together (the kernel is latency-bound: a decode
// merge moves a few MB).  It is launched as a programmatic dependent of the split
// kernel, so its launch overlaps that kernel's last CTAs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace gqa {
namespace {

constexpr int kWarps = 8;

// Waits (hardware dependency, no spinning) until the kernel this launch depends on
// programmatically has completed and its writes are visible; returns at once when
// there is no such kernel.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int kBatch = 16;  // parts whose loads are issued together

template <bool kF16>
__global__ void __launch_bounds__(kWarps * 32)
lse_merge_kernel(const float* __restrict__ O_parts, const float* __restrict__ lse_parts, int S,
                 int N, const uint16_t* __restrict__ G, uint16_t* __restrict__ out,
                 float* __restrict__ lse_out, int gate_early) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (n >= N) return;
  const size_t stride = size_t(N);
  const int c0 = lane * 8;

  // After the library's own split kernel the gate, written before that kernel in
  // stream order, is read before waiting for it (gate_early); otherwise after.
  if (!gate_early) grid_dependency_wait();
  float gs[8];
  if (G != nullptr) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(G + size_t(n) * 256 + c0));
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack_elem2<kF16>(w4[e]);
      gs[2 * e] = gate_sigmoid(f.x);
      gs[2 * e + 1] = gate_sigmoid(f.y);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) gs[e] = 1.f;
  }
  if (gate_early) grid_dependency_wait();

  // Max over parts (lane s reads part s of each round of 32).  fmaxf drops NaN; a NaN
  // part still gets weight NaN below.  With S <= 32 the first round's values are kept.
  const float ls0 = lane < S ? __ldcg(lse_parts + size_t(lane) * stride + n) : -INFINITY;
  float M = ls0;
  for (int s = lane + 32; s < S; s += 32) M = fmaxf(M, __ldcg(lse_parts + size_t(s) * stride + n));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  const float Msub = M == -INFINITY ? 0.f : M;
  for (int s0 = 0; s0 < S; s0 += 32) {
    // lane s holds the weight of part s0 + s (0 for an empty or missing part)
    const int sl = s0 + lane;
    const float ls = s0 == 0 ? ls0 : sl < S ? __ldcg(lse_parts + size_t(sl) * stride + n)
                                            : -INFINITY;
    const float wl = ls == -INFINITY ? 0.f : __expf(ls - Msub);
    const int cnt = min(32, S - s0);
    for (int b = 0; b < cnt; b += kBatch) {
      float w[kBatch];
      float4 va[kBatch], vb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        w[u] = __shfl_sync(0xffffffffu, wl, min(b + u, 31));
        if (b + u >= cnt) w[u] = 0.f;
        va[u] = vb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (w[u] != 0.f) {
          const float4* src = reinterpret_cast<const float4*>(
              O_parts + (size_t(s0 + b + u) * stride + n) * 256 + c0);
          va[u] = __ldcg(src);
          vb[u] = __ldcg(src + 1);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        wsum += w[u];
        acc[0] += w[u] * va[u].x;
        acc[1] += w[u] * va[u].y;
        acc[2] += w[u] * va[u].z;
        acc[3] += w[u] * va[u].w;
        acc[4] += w[u] * vb[u].x;
        acc[5] += w[u] * vb[u].y;
        acc[6] += w[u] * vb[u].z;
        acc[7] += w[u] * vb[u].w;
      }
    }
  }
  const float inv = wsum == 0.f ? 0.f : 1.f / wsum;
  uint4 o;
  o.x = pack_elem2<kF16>(acc[0] * inv * gs[0], acc[1] * inv * gs[1]);
  o.y = pack_elem2<kF16>(acc[2] * inv * gs[2], acc[3] * inv * gs[3]);
  o.z = pack_elem2<kF16>(acc[4] * inv * gs[4], acc[5] * inv * gs[5]);
  o.w = pack_elem2<kF16>(acc[6] * inv * gs[6], acc[7] * inv * gs[7]);
  *reinterpret_cast<uint4*>(out + size_t(n) * 256 + c0) = o;
  if (lse_out != nullptr && lane == 0)
    lse_out[n] = wsum == 0.f ? -INFINITY : Msub + __logf(wsum);
}

template <bool kF16>
cudaError_t launch_merge_t(const MergeArgs& a, long long grid, cudaStream_t stream) {
  if (!a.after_split) {
    lse_merge_kernel<kF16><<<dim3(unsigned(grid)), dim3(kWarps * 32), 0, stream>>>(
        a.O_parts, a.lse_parts, a.S, a.N, static_cast<const uint16_t*>(a.G),
        static_cast<uint16_t*>(a.out), a.lse_out, 0);
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
      note_launch(kF16 ? "lse_merge_kernel<fp16>" : "lse_merge_kernel<bf16>", grid, kWarps * 32, 0);
    return e;
  }
  // Right after the library's split kernel: programmatic dependent launch, so the
  // merge may be scheduled while that kernel drains; it waits for it in
  // grid_dependency_wait before reading the parts.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, lse_merge_kernel<kF16>, a.O_parts, a.lse_parts, a.S, a.N,
                         static_cast<const uint16_t*>(a.G), static_cast<uint16_t*>(a.out),
                         a.lse_out, 1);
  if (e == cudaSuccess)
    note_launch(kF16 ? "lse_merge_kernel<fp16> dependent" : "lse_merge_kernel<bf16> dependent",
                grid, kWarps * 32, 0);
  return e;
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, const LaunchCtl& ctl, cudaStream_t stream) {
  (void)ctl;
  const long long grid = (a.N + kWarps - 1) / kWarps;
  return a.f16 ? launch_merge_t<true>(a, grid, stream) : launch_merge_t<false>(a, grid, stream);
}

}  // namespace gqa
