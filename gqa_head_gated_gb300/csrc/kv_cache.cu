// KV-cache maintenance around decode / verify: append new rows after the keys a
// sequence holds, and keep the accepted draft rows after verification (TensorFold
// PR #1009, "Receipt": packing, append and keep are compared bit for bit; control
// "an append one row late").  Both are plain 16-byte copies of 512-byte key rows by
// whole warps (append: four rows per warp; keep: one sequence and KV head per warp);
// sequence lengths live on the device and are range-checked there.
#include <cuda_runtime.h>

#include "gqa_attn.h"
#include "internal.h"

namespace gqa {
namespace {

constexpr int kWarps = 8;

// Sequence holding token t: the largest b with cu_rows[b] <= t (binary search).
__device__ __forceinline__ int seq_of(const int* cu_rows, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu_rows + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

constexpr int kRowsPerWarp = 4;   // (token, KV head) rows per warp: 8 loads in flight per lane

// One warp per kRowsPerWarp consecutive (new token, KV head) items: K and V rows of
// 512 bytes, 16 bytes per lane; all loads are issued before the stores.
__global__ void __launch_bounds__(kWarps * 32)
kv_append_kernel(const uint4* __restrict__ Knew, const uint4* __restrict__ Vnew,
                 const int* __restrict__ cu_rows, const int* __restrict__ kv_lens,
                 uint4* __restrict__ Kc, uint4* __restrict__ Vc, int B, int T, int Hkv,
                 int Lcap, LaunchCtl ctl) {
  const long long w0 = ((long long)blockIdx.x * kWarps + (threadIdx.x >> 5)) * kRowsPerWarp;
  const int lane = threadIdx.x & 31;
  const long long n_items = (long long)T * Hkv;
  uint4 kv[kRowsPerWarp][2];
  size_t dst[kRowsPerWarp];
  bool live[kRowsPerWarp];
#pragma unroll
  for (int u = 0; u < kRowsPerWarp; ++u) {
    const long long w = w0 + u;
    live[u] = false;
    dst[u] = 0;
    if (w >= n_items) continue;
    const int t = int(w / Hkv);
    const int g = int(w - (long long)t * Hkv);
    const int b = cu_rows ? seq_of(cu_rows, B, t) : t;
    const int i = cu_rows ? t - __ldg(cu_rows + b) : 0;
    const int pos = __ldg(kv_lens + b) + i;
    if (pos < 0 || pos >= Lcap) {
      if (lane == 0) record_status(ctl.status, GQA_ERR_DEVICE_RANGE);
      continue;
    }
    const size_t src = (size_t(t) * Hkv + g) * 32 + lane;
    dst[u] = ((size_t(b) * Hkv + g) * size_t(Lcap) + pos) * 32 + lane;
    kv[u][0] = __ldg(Knew + src);
    kv[u][1] = __ldg(Vnew + src);
    live[u] = true;
  }
#pragma unroll
  for (int u = 0; u < kRowsPerWarp; ++u) {
    if (!live[u]) continue;
    Kc[dst[u]] = kv[u][0];
    Vc[dst[u]] = kv[u][1];
  }
}

// One warp per (sequence, KV head): kept draft rows move to the front of the draft
// region in increasing order.  Destinations never pass their sources (keep indices
// strictly increase), so copying the rows one after another in that order is safe
// in place.
__global__ void __launch_bounds__(kWarps * 32)
kv_keep_kernel(uint4* __restrict__ Kc, uint4* __restrict__ Vc, const int* __restrict__ kv_lens,
               const int* __restrict__ cu_rows, const int* __restrict__ keep_idx,
               const int* __restrict__ cu_keep, int* __restrict__ kv_lens_out, int B, int Hkv,
               int Lcap, LaunchCtl ctl) {
  const int w = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= B * Hkv) return;
  const int b = w / Hkv;
  const int g = w - b * Hkv;
  const int r = __ldg(cu_rows + b + 1) - __ldg(cu_rows + b);
  const int L = __ldg(kv_lens + b);
  const int k0 = __ldg(cu_keep + b);
  const int nk = __ldg(cu_keep + b + 1) - k0;
  const int base = L - r;
  bool ok = r >= 0 && base >= 0 && L <= Lcap && nk >= 0 && nk <= r;
  for (int k = 0; ok && k < nk; ++k) {
    const int idx = __ldg(keep_idx + k0 + k);
    ok = idx >= 0 && idx < r && (k == 0 || idx > __ldg(keep_idx + k0 + k - 1));
  }
  if (!ok) {
    if (lane == 0 && g == 0) record_status(ctl.status, GQA_ERR_DEVICE_RANGE);
    return;
  }
  const size_t row0 = (size_t(b) * Hkv + g) * size_t(Lcap);
  for (int k = 0; k < nk; ++k) {
    const int idx = __ldg(keep_idx + k0 + k);
    if (idx == k) continue;   // already in place
    const size_t s = (row0 + base + idx) * 32 + lane;
    const size_t d = (row0 + base + k) * 32 + lane;
    const uint4 kv = Kc[s];
    const uint4 vv = Vc[s];
    __syncwarp();
    Kc[d] = kv;
    Vc[d] = vv;
    __syncwarp();
  }
  if (kv_lens_out != nullptr && g == 0 && lane == 0) kv_lens_out[b] = base + nk;
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" {

int gqa_kv_append(const void* Knew, const void* Vnew, const int* cu_rows, const int* kv_lens,
                  void* Kcache, void* Vcache, int B, int T, int Hkv, int Lcap,
                  gqa_stream_t stream) {
  if (B < 1 || T < 0 || Hkv < 1 || Lcap < 1 || (cu_rows == nullptr && T != B))
    return GQA_ERR_INVALID_ARG;
  if ((long long)T * Hkv >= (1LL << 31) || (long long)B * Hkv * Lcap >= (1LL << 40))
    return GQA_ERR_UNSUPPORTED;
  if (T == 0) return GQA_OK;
  const auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (Knew == nullptr || Vnew == nullptr || kv_lens == nullptr || Kcache == nullptr ||
      Vcache == nullptr || !al(Knew, 16) || !al(Vnew, 16) || !al(Kcache, 16) || !al(Vcache, 16) ||
      !al(kv_lens, 4) || (cu_rows != nullptr && !al(cu_rows, 4)))
    return GQA_ERR_INVALID_ARG;
  LaunchCtl ctl;
  if (!make_launch_ctl(&ctl)) return GQA_ERR_CUDA;
  const long long per_cta = (long long)kWarps * kRowsPerWarp;
  const long long grid = ((long long)T * Hkv + per_cta - 1) / per_cta;
  kv_append_kernel<<<dim3(unsigned(grid)), kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(Knew), static_cast<const uint4*>(Vnew), cu_rows, kv_lens,
      static_cast<uint4*>(Kcache), static_cast<uint4*>(Vcache), B, T, Hkv, Lcap, ctl);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  note_launch("kv_append_kernel", grid, kWarps * 32, 0);
  return GQA_OK;
}

int gqa_kv_keep(void* Kcache, void* Vcache, const int* kv_lens, const int* cu_rows,
                const int* keep_idx, const int* cu_keep, int* kv_lens_out, int B, int Hkv,
                int Lcap, gqa_stream_t stream) {
  if (B < 1 || Hkv < 1 || Lcap < 1) return GQA_ERR_INVALID_ARG;
  if ((long long)B * Hkv >= (1LL << 31) || (long long)B * Hkv * Lcap >= (1LL << 40))
    return GQA_ERR_UNSUPPORTED;
  const auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (Kcache == nullptr || Vcache == nullptr || kv_lens == nullptr || cu_rows == nullptr ||
      keep_idx == nullptr || cu_keep == nullptr || !al(Kcache, 16) || !al(Vcache, 16) ||
      !al(kv_lens, 4) || !al(cu_rows, 4) || !al(keep_idx, 4) || !al(cu_keep, 4) ||
      (kv_lens_out != nullptr && (!al(kv_lens_out, 4) || kv_lens_out == kv_lens)))
    return GQA_ERR_INVALID_ARG;
  LaunchCtl ctl;
  if (!make_launch_ctl(&ctl)) return GQA_ERR_CUDA;
  const long long grid = ((long long)B * Hkv + kWarps - 1) / kWarps;
  kv_keep_kernel<<<dim3(unsigned(grid)), kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(Kcache), static_cast<uint4*>(Vcache), kv_lens, cu_rows, keep_idx,
      cu_keep, kv_lens_out, B, Hkv, Lcap, ctl);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  note_launch("kv_keep_kernel", grid, kWarps * 32, 0);
  return GQA_OK;
}

}  // extern "C"
