// gqa_attn_decode_noalloc: decode / chain verify for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at decode time: a
// serving loop that must not touch a device allocator between steps (an allocation
// can stall on device-wide synchronisation or fail under memory pressure in the
// middle of a request), or a plug-in whose host application hands it only fixed
// input and output buffers and owns all other device memory.
// This entry point is gqa_attn_decode with a workspace that belongs to the library:
// the same argument checks, plan, kernels and results, bit for bit, and the same
// workspace rule (gqa_attn_decode_workspace_size() for the call must fit the area,
// else GQA_ERR_WORKSPACE before any launch).
//
// The area is a file-scope __device__ array of kStaticScratchBytes (16 MiB).  Every
// GPU that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, with that device current, on the
// first call made on that device; that first call should therefore come before
// any stream capture.  All calls on a device share the one area and it keeps the
// previous call's contents: nothing in it needs to start at zero (the split kernels
// write every partial row the merge reads), but two calls whose kernels overlap on
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
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return GQA_ERR_CUDA;
  return decode_bf16_with_workspace(Q, Kcache, Vcache, G, kv_lens, cu_rows, out, lse_out, B, T,
                                    Hq, Hkv, Lcap, max_rows, max_kv_len, scratch,
                                    kStaticScratchBytes, stream);
}

}  // extern "C"
