// gqa_selftest_wait_timeout: exercises the kernels' bounded wait on the device.
//
// Every spin wait in the library's kernels is ptx::mbar_wait with a deadline; on
// expiry the kernel records GQA_ERR_TIMEOUT and unwinds instead of hanging.  This
// entry point runs that same wait on an mbarrier that nothing will ever complete,
// so a caller (or a test) can watch the bound fire and the context stay usable,
// without faulting or hanging the GPU.
#include <cuda_runtime.h>

#include "gqa_attn.h"
#include "internal.h"
#include "ptx_sm100.cuh"

namespace gqa {
namespace {

__global__ void wait_timeout_probe(LaunchCtl ctl, unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  __shared__ int zero;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);   // one arrival would complete phase 0; none comes
    zero = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    if (!ptx::mbar_wait(&bar, 0, ctl.timeout_ns, &zero)) record_status(ctl.status, GQA_ERR_TIMEOUT);
    if (elapsed_ns != nullptr) *elapsed_ns = global_timer_ns() - t0;
  }
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" int gqa_selftest_wait_timeout(unsigned long long* elapsed_ns, gqa_stream_t stream) {
  if (elapsed_ns != nullptr && reinterpret_cast<uintptr_t>(elapsed_ns) % 8 != 0)
    return GQA_ERR_INVALID_ARG;
  LaunchCtl ctl;
  if (!make_launch_ctl(&ctl)) return GQA_ERR_CUDA;
  wait_timeout_probe<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctl, elapsed_ns);
  if (cudaGetLastError() != cudaSuccess) return GQA_ERR_CUDA;
  note_launch("wait_timeout_probe", 1, 32, 0);
  return GQA_OK;
}
