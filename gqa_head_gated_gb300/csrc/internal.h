// Host-side launchers shared between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "device_common.cuh"

namespace gqa {

struct PrefillArgs {
  const void* Q;
  const void* K;
  const void* V;
  const void* G;
  void* out;
  float* lse;
  int B, Hq, Hkv, Lq, Lkv, kv_offset;
  bool f16 = false;   // fp16 instead of bf16 elements
  // General-mask form (gqa_attn_masked).  `masked` selects the kernel that reads a
  // mask and honours `causal`; the plain prefill is always causal and unmasked.
  bool masked = false;
  bool causal = true;
  const void* mask = nullptr;
  int mask_kind = 0;        // gqa_mask_kind
  int mask_hmode = 0;       // 0: one mask head; 1: mask head = query head; 2: chunk-local
  int mask_chunk = 1;       // chunk size for mode 2
  long long mask_strides[4] = {0, 0, 0, 0};   // elements; [batch, head, row, key]
};

// Rows of one prefill tile: floor(128 / GQA) query rows of every head in the group.
inline int prefill_rows_per_tile(int gqa) { return 128 / gqa; }

// Returns cudaSuccess, or the error of encoding the tensor maps / launching.
// Sets *encode_failed when a TMA descriptor could not be built.
cudaError_t launch_prefill(const PrefillArgs& a, const LaunchCtl& ctl, cudaStream_t stream,
                           bool* encode_failed);
// The plain (causal, unmasked) prefill on CTA pairs (gqa_attn_prefill_pair; and
// gqa_attn_prefill when the last row sees at least kPairMinKeys keys).
constexpr int kPairMinKeys = 2048;
cudaError_t launch_prefill_pair(const PrefillArgs& a, const LaunchCtl& ctl, cudaStream_t stream,
                                bool* encode_failed);

struct DecodeSplitArgs {
  const void* Q;
  const void* K;
  const void* V;
  const int* kv_lens;
  const int* cu_rows;
  float* O_parts;
  float* lse_parts;
  int B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, num_splits, split_keys;
  // Tree verify: per new row, a mask over its sequence's new rows (bit k = new row
  // k visible); null for chain verify / decode.
  const unsigned long long* tree_mask = nullptr;
  bool f16 = false;   // fp16 instead of bf16 elements
  // mma.sync kernel only: equal shares of all sequences' key tiles per CTA instead
  // of one (b, g, split, row block) unit per CTA; num_splits is then the part
  // capacity per row (>= 3) and split_keys is unused.  B <= kBalancedMaxSeqs.
  bool balanced = false;
};

constexpr int kBalancedMaxSeqs = 256;
constexpr int kBalancedParts = 16;

// Packed query rows (heads x rows of one KV group) per decode CTA: 16, 32 or 64.
int decode_rows_per_cta(int packed_rows);

cudaError_t launch_decode_split(const DecodeSplitArgs& a, const LaunchCtl& ctl,
                                cudaStream_t stream);

// The same split on the tcgen05 kernel (split mode of the prefill kernel); split_keys
// must be a multiple of tc_split_keys_multiple().  Sets *encode_failed when a TMA
// descriptor could not be built.
int tc_split_keys_multiple();
cudaError_t launch_decode_split_tc(const DecodeSplitArgs& a, const LaunchCtl& ctl,
                                   cudaStream_t stream, bool* encode_failed);

struct MergeArgs {
  const float* O_parts;
  const float* lse_parts;
  int S, N;
  const void* G;
  void* out;
  float* lse_out;
  bool f16 = false;   // fp16 instead of bf16 G / out
  // Launched right after the library's split kernel on the same stream: programmatic
  // dependent launch (the merge is scheduled while the split kernel drains).
  bool after_split = false;
};

cudaError_t launch_lse_merge(const MergeArgs& a, const LaunchCtl& ctl, cudaStream_t stream);

// Notes a kernel launch in the library's launch log (gqa_launch_log); `kernel` is
// copied (at most 63 characters).  Call it after the launch call succeeded.
void note_launch(const char* kernel, long long grid, int block, size_t dynamic_smem);

// gqa_attn_decode's host side, shared with the no-allocation entry point: its argument
// checks, and the whole call (checks, plan, kernels) with a given workspace.
int decode_check_args(int B, int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                      bool has_cu_rows);
// The launch control block (status word, wait bound) for the current device.
bool make_launch_ctl(LaunchCtl* ctl);
int decode_bf16_with_workspace(const void* Q, const void* Kcache, const void* Vcache,
                               const void* G, const int* kv_lens, const int* cu_rows, void* out,
                               float* lse_out, int B, int T, int Hq, int Hkv, int Lcap,
                               int max_rows, int max_kv_len, void* workspace,
                               size_t workspace_bytes, gqa_stream_t stream);

}  // namespace gqa
