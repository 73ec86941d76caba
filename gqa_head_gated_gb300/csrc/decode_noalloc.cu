// gqa_attn_decode_noalloc: decode / chain verify for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at decode time: a
// serving loop that must not touch a device allocator between steps (an allocation
// can stall on device-wide synchronisation or fail under memory pressure in the
// middle of a request), or a plug-in whose host application hands it only fixed
// input and output buffers and owns all other device memory.
// This entry point takes the same inputs and outputs as gqa_attn_decode but keeps
// the split partial results in a fixed area of device memory that belongs to the
// library, so the caller passes no workspace.
//
// The area is a file-scope __device__ array of kStaticScratchBytes (16 MiB).  Every
// GPU that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current, on the
// first call made on that device; that first call should therefore come before
// any stream capture.  All calls on a device share the one area and it keeps the
// previous call's contents: nothing in it needs to start at zero (the split kernel
// writes every partial row the merge reads), but two calls whose kernels overlap on
// the GPU (different streams, no ordering between them) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "gqa_attn.h"
#include "internal.h"

namespace gqa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch on the current device; nullptr on failure.
void* scratch_on_current_device() {
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" {

int gqa_attn_decode_noalloc(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                            const int* kv_lens, const int* cu_rows, void* out, float* lse_out,
                            int B, int T, int Hq, int Hkv, int Lcap, int max_rows,
                            int max_kv_len, gqa_stream_t stream) {
  const int st = decode_check_args(B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, cu_rows != nullptr);
  if (st != GQA_OK) return st;
  if (T == 0) return GQA_OK;
  if (Q == nullptr || Kcache == nullptr || Vcache == nullptr || kv_lens == nullptr ||
      out == nullptr)
    return GQA_ERR_INVALID_ARG;
  const auto al = [](const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; };
  if (!al(Q, 16) || !al(Kcache, 16) || !al(Vcache, 16) || !al(out, 16) ||
      (G != nullptr && !al(G, 16)) || (lse_out != nullptr && !al(lse_out, 4)) ||
      !al(kv_lens, 4) || (cu_rows != nullptr && !al(cu_rows, 4)))
    return GQA_ERR_INVALID_ARG;
  int S = 0, C = 0;
  decode_plan_current_device(B, Hq, Hkv, max_rows, max_kv_len, &S, &C);
  if (decode_workspace_bytes(T, Hq, S) > kStaticScratchBytes) return GQA_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  LaunchCtl ctl;
  if (scratch == nullptr || !make_launch_ctl(&ctl)) return GQA_ERR_CUDA;
  float* O_parts = static_cast<float*>(scratch);
  float* lse_parts = O_parts + size_t(S) * size_t(T) * Hq * 256;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DecodeSplitArgs a{Q, Kcache, Vcache, kv_lens, cu_rows, O_parts, lse_parts, B, T, Hq, Hkv,
                    Lcap, max_rows, max_kv_len, S, C};
  if (launch_decode_split(a, ctl, s) != cudaSuccess) return GQA_ERR_CUDA;
  MergeArgs m{O_parts, lse_parts, S, T * Hq, G, out, lse_out};
  m.after_split = true;
  return launch_lse_merge(m, ctl, s) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // extern "C"
