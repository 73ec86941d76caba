// C ABI of libgqa_attn.so: argument validation, split planning, the device
// status word, and the launches.  The operation and conventions are stated in
// include/gqa_attn.h.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "gqa_attn.h"
#include "internal.h"

namespace gqa {
namespace {

__device__ int g_status_word;

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};

constexpr int kMaxDevices = 64;
constexpr int kDefaultSMs = 152;   // GB300

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device address of the status word on the current device (looked up once per device).
int* status_ptr() {
  static std::mutex mu;
  static int* ptrs[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

int sm_count() {
  static std::mutex mu;
  static int counts[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kDefaultSMs;
  std::lock_guard<std::mutex> lock(mu);
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kDefaultSMs;
    counts[dev] = n;
  }
  return counts[dev];
}

bool make_ctl(LaunchCtl* ctl) {
  ctl->status = status_ptr();
  ctl->timeout_ns = g_timeout_ns.load();
  return ctl->status != nullptr;
}

int ceil_div(long long a, long long b) { return int((a + b - 1) / b); }

// Decode / verify groups with more than 16 packed rows (new rows x query heads per KV
// group) run on the tcgen05 kernel; up to 16 on the mma.sync split kernel, in its
// 16-row form with two CTAs per SM.  Measured on GB300 (one-call decode, L2 flushed):
// from 18 packed rows on the tcgen05 split is 1.15-1.8x faster (the mma.sync kernel's
// 32- and 64-row forms run one CTA per SM); from 6 to 16 the two are within ~10 %,
// the mma.sync kernel ahead on the 27B decode.
constexpr long long kTcMinPackedRows = 17;
constexpr int kTcMinSplitKeys = 1024;   // at least 8 key tiles per tcgen05 CTA

bool tc_path(int Hq, int Hkv, int max_rows) {
  return (long long)max_rows * (Hq / Hkv) >= kTcMinPackedRows && Hq / Hkv <= 128;
}

// Fixed-split decode plan (gqa_attn_decode_plan, and the one-call decode when it does
// not run balanced shares): aim for about three waves of resident CTAs over the
// (sequence, group, row block) units (two CTAs fit per SM up to 32 packed rows, one
// above), so that ragged kv lengths still leave enough CTAs to balance the SMs;
// splits are whole 64-key steps (128-key tiles on the tcgen05 path).
int plan_decode(int B, int Hq, int Hkv, int max_rows, int max_kv_len, int num_sms, int* S,
                int* C) {
  const int gqa = Hq / Hkv;
  if (tc_path(Hq, Hkv, max_rows)) {
    // tcgen05 path: one CTA per SM; aim for ~3 CTAs per SM on the longest sequence's
    // basis (ragged lengths leave fewer live), splits of whole 128-key tiles and at
    // least kTcMinSplitKeys keys so the prologue, the epilogue and the merge stay small.
    const int kt = tc_split_keys_multiple();
    const long long R = 128 / gqa;
    const long long units = (long long)B * Hkv * ((max_rows + R - 1) / R);
    const long long want = 3LL * num_sms;
    long long s = (want + units - 1) / units;
    const long long tiles = (max_kv_len + kt - 1) / kt;
    if (s > tiles) s = tiles;
    if (s < 1) s = 1;
    long long c = ((max_kv_len + s - 1) / s + kt - 1) / kt * kt;
    if (c < kTcMinSplitKeys) c = kTcMinSplitKeys;
    s = (max_kv_len + c - 1) / c;
    *S = int(s);
    *C = int(c);
    return GQA_OK;
  }
  const long long packed = (long long)max_rows * gqa;
  const int MB = decode_rows_per_cta(int(packed > (1 << 30) ? (1 << 30) : packed));
  const long long n_rb = (packed + MB - 1) / MB;
  const long long units = (long long)B * Hkv * n_rb;
  const long long want = (MB <= 32 ? 6LL : 4LL) * num_sms;
  long long s = (want + units - 1) / units;
  const long long steps = (max_kv_len + 63) / 64;
  if (s > steps) s = steps;
  if (s < 1) s = 1;
  long long c = ((max_kv_len + s - 1) / s + 63) / 64 * 64;
  s = (max_kv_len + c - 1) / c;
  *S = int(s);
  *C = int(c);
  return GQA_OK;
}

int check_decode_args(int B, int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                      bool has_cu_rows) {
  if (B < 1 || T < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lcap < 1) return GQA_ERR_INVALID_ARG;
  if (max_rows < 1 || max_kv_len < 1 || max_kv_len > Lcap || max_rows > max_kv_len)
    return GQA_ERR_INVALID_ARG;
  if (!has_cu_rows && (T != B || max_rows != 1)) return GQA_ERR_INVALID_ARG;
  if ((long long)T > (long long)B * max_rows) return GQA_ERR_INVALID_ARG;
  if ((long long)T * Hq >= (1LL << 31)) return GQA_ERR_UNSUPPORTED;
  if ((long long)B * Hkv * Lcap >= (1LL << 40)) return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

size_t workspace_bytes_for(int T, int Hq, int S) {
  const size_t rows = size_t(T) * size_t(Hq);
  return size_t(S) * rows * 256 * sizeof(float) + size_t(S) * rows * sizeof(float);
}

// The one-call decode's choice: the mma.sync kernel (at most 16 packed rows per KV
// group) runs balanced shares when the batch fits the kernel's table.
bool use_balanced(int B, int Hq, int Hkv, int max_rows) {
  return !tc_path(Hq, Hkv, max_rows) && B <= kBalancedMaxSeqs;
}

// Parts per row the one-call decode writes (its workspace holds this many).
int call_parts(int B, int Hq, int Hkv, int max_rows, int S) {
  return use_balanced(B, Hq, Hkv, max_rows) ? kBalancedParts : S;
}

int run_split(const void* Q, const void* Kc, const void* Vc, const int* kv_lens,
              const int* cu_rows, float* O_parts, float* lse_parts, int B, int T, int Hq, int Hkv,
              int Lcap, int max_rows, int max_kv_len, int S, int C, cudaStream_t stream,
              const unsigned long long* tree_mask, bool f16, bool balanced = false) {
  LaunchCtl ctl;
  if (!make_ctl(&ctl)) return GQA_ERR_CUDA;
  DecodeSplitArgs a{Q, Kc, Vc, kv_lens, cu_rows, O_parts, lse_parts, B, T, Hq, Hkv, Lcap,
                    max_rows, max_kv_len, S, C};
  a.tree_mask = tree_mask;
  a.f16 = f16;
  if (balanced) {
    a.balanced = true;
    return launch_decode_split(a, ctl, stream) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
  }
  if (tc_path(Hq, Hkv, max_rows) && C % tc_split_keys_multiple() == 0) {
    bool encode_failed = false;
    const cudaError_t e = launch_decode_split_tc(a, ctl, stream, &encode_failed);
    if (encode_failed) return GQA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
  }
  return launch_decode_split(a, ctl, stream) == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

}  // namespace

int decode_check_args(int B, int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                      bool has_cu_rows) {
  return check_decode_args(B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, has_cu_rows);
}
bool make_launch_ctl(LaunchCtl* ctl) { return make_ctl(ctl); }

namespace {

// Entry points for both element types; the extern "C" functions below pick one.
int gqa_attn_prefill_impl(bool f16, const void* Q, const void* K, const void* V, const void* G,
                          void* out, float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv,
                          int kv_offset, gqa_stream_t stream, bool pair = false) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lq < 0 || Lkv < 1 || kv_offset < 0 ||
      (long long)kv_offset + Lq > Lkv)
    return GQA_ERR_INVALID_ARG;
  if (Lq == 0) return GQA_OK;   // nothing to do (an empty tensor may have a null pointer)
  if (Q == nullptr || K == nullptr || V == nullptr || out == nullptr) return GQA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(out, 16) ||
      (G != nullptr && !aligned(G, 16)) || (lse_out != nullptr && !aligned(lse_out, 4)))
    return GQA_ERR_INVALID_ARG;
  if (Hq / Hkv > 128) return GQA_ERR_UNSUPPORTED;
  if ((long long)Hq * Lq >= (1LL << 31) || (long long)B * Hkv >= (1LL << 31))
    return GQA_ERR_UNSUPPORTED;
  // (the CTA-pair form rounds the row tiles up to pairs)
  const long long grid = (long long)(ceil_div(Lq, prefill_rows_per_tile(Hq / Hkv)) + 1) * B * Hkv;
  if (grid >= (1LL << 31)) return GQA_ERR_UNSUPPORTED;
  LaunchCtl ctl;
  if (!make_ctl(&ctl)) return GQA_ERR_CUDA;
  PrefillArgs a{Q, K, V, G, out, lse_out, B, Hq, Hkv, Lq, Lkv, kv_offset};
  a.f16 = f16;
  bool encode_failed = false;
  const cudaError_t e =
      pair ? launch_prefill_pair(a, ctl, static_cast<cudaStream_t>(stream), &encode_failed)
           : launch_prefill(a, ctl, static_cast<cudaStream_t>(stream), &encode_failed);
  if (encode_failed) return GQA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

int gqa_attn_decode_split_impl(bool f16, const void* Q, const void* Kcache, const void* Vcache,
                               const int* kv_lens, const int* cu_rows, float* O_parts,
                               float* lse_parts, int B, int T, int Hq, int Hkv, int Lcap,
                               int max_rows, int max_kv_len, int num_splits, int split_keys,
                               gqa_stream_t stream) {
  const int st = check_decode_args(B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, cu_rows != nullptr);
  if (st != GQA_OK) return st;
  const bool bal = split_keys == 0;   // balanced shares, num_splits part slots per row
  if (bal) {
    if (num_splits < 3) return GQA_ERR_INVALID_ARG;
    if (!use_balanced(B, Hq, Hkv, max_rows)) return GQA_ERR_UNSUPPORTED;
  } else if (num_splits < 1 || split_keys < 64 || split_keys % 64 != 0 ||
             (long long)num_splits * split_keys < max_kv_len) {
    return GQA_ERR_INVALID_ARG;
  }
  if (T == 0) return GQA_OK;
  if (Q == nullptr || Kcache == nullptr || Vcache == nullptr || kv_lens == nullptr ||
      O_parts == nullptr || lse_parts == nullptr)
    return GQA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(Kcache, 16) || !aligned(Vcache, 16) || !aligned(O_parts, 16) ||
      !aligned(lse_parts, 4) || !aligned(kv_lens, 4) || (cu_rows && !aligned(cu_rows, 4)))
    return GQA_ERR_INVALID_ARG;
  const int gqa = Hq / Hkv;
  const long long packed = (long long)max_rows * gqa;
  const int MB = decode_rows_per_cta(int(packed > (1 << 30) ? (1 << 30) : packed));
  const long long grid = (long long)B * Hkv * num_splits * ((packed + MB - 1) / MB);
  if (grid >= (1LL << 31)) return GQA_ERR_UNSUPPORTED;
  return run_split(Q, Kcache, Vcache, kv_lens, cu_rows, O_parts, lse_parts, B, T, Hq, Hkv, Lcap,
                   max_rows, max_kv_len, num_splits, split_keys,
                   static_cast<cudaStream_t>(stream), nullptr, f16, bal);
}

int attn_lse_merge_impl(bool f16, const float* O_parts, const float* lse_parts, int S, int N,
                        const void* G, void* out, float* lse_out, gqa_stream_t stream,
                        bool after_split = false) {
  if (S < 1 || N < 0) return GQA_ERR_INVALID_ARG;
  if (N == 0) return GQA_OK;
  if (O_parts == nullptr || lse_parts == nullptr || out == nullptr) return GQA_ERR_INVALID_ARG;
  if (!aligned(O_parts, 16) || !aligned(lse_parts, 4) || !aligned(out, 16) ||
      (G != nullptr && !aligned(G, 16)) || (lse_out != nullptr && !aligned(lse_out, 4)))
    return GQA_ERR_INVALID_ARG;
  LaunchCtl ctl;
  if (!make_ctl(&ctl)) return GQA_ERR_CUDA;
  MergeArgs a{O_parts, lse_parts, S, N, G, out, lse_out};
  a.f16 = f16;
  a.after_split = after_split;
  return launch_lse_merge(a, ctl, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

int gqa_attn_decode_impl(bool f16, const void* Q, const void* Kcache, const void* Vcache,
                         const void* G, const int* kv_lens, const int* cu_rows, void* out,
                         float* lse_out, int B, int T, int Hq, int Hkv, int Lcap, int max_rows,
                         int max_kv_len, void* workspace, size_t workspace_bytes,
                         gqa_stream_t stream) {
  const int st = check_decode_args(B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, cu_rows != nullptr);
  if (st != GQA_OK) return st;
  if (T == 0) return GQA_OK;
  if (Q == nullptr || Kcache == nullptr || Vcache == nullptr || kv_lens == nullptr ||
      out == nullptr)
    return GQA_ERR_INVALID_ARG;
  if (!aligned(out, 16) || (G != nullptr && !aligned(G, 16)) ||
      (lse_out != nullptr && !aligned(lse_out, 4)))
    return GQA_ERR_INVALID_ARG;
  int S = 0, C = 0;
  plan_decode(B, Hq, Hkv, max_rows, max_kv_len, sm_count(), &S, &C);
  const bool bal = use_balanced(B, Hq, Hkv, max_rows);
  if (bal) S = kBalancedParts;
  const size_t need = workspace_bytes_for(T, Hq, S);
  if (workspace == nullptr || workspace_bytes < need) return GQA_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return GQA_ERR_INVALID_ARG;
  float* O_parts = static_cast<float*>(workspace);
  float* lse_parts = O_parts + size_t(S) * size_t(T) * Hq * 256;
  const int r = gqa_attn_decode_split_impl(f16, Q, Kcache, Vcache, kv_lens, cu_rows, O_parts,
                                           lse_parts, B, T, Hq, Hkv, Lcap, max_rows, max_kv_len,
                                           S, bal ? 0 : C, stream);
  if (r != GQA_OK) return r;
  return attn_lse_merge_impl(f16, O_parts, lse_parts, S, T * Hq, G, out, lse_out, stream,
                             true);
}

int gqa_attn_verify_tree_impl(bool f16, const void* Q, const void* Kcache, const void* Vcache,
                              const void* G, const int* kv_lens, const int* cu_rows,
                              const unsigned long long* tree_mask, void* out, float* lse_out,
                              int B, int T, int Hq, int Hkv, int Lcap, int max_rows,
                              int max_kv_len, void* workspace, size_t workspace_bytes,
                              gqa_stream_t stream) {
  const int st = check_decode_args(B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, cu_rows != nullptr);
  if (st != GQA_OK) return st;
  if (max_rows > 64) return GQA_ERR_UNSUPPORTED;   // one 64-bit mask per row
  if (T == 0) return GQA_OK;
  if (Q == nullptr || Kcache == nullptr || Vcache == nullptr || kv_lens == nullptr ||
      cu_rows == nullptr || tree_mask == nullptr || out == nullptr)
    return GQA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(Kcache, 16) || !aligned(Vcache, 16) || !aligned(out, 16) ||
      (G != nullptr && !aligned(G, 16)) || (lse_out != nullptr && !aligned(lse_out, 4)) ||
      !aligned(kv_lens, 4) || !aligned(cu_rows, 4) || !aligned(tree_mask, 8))
    return GQA_ERR_INVALID_ARG;
  int S = 0, C = 0;
  plan_decode(B, Hq, Hkv, max_rows, max_kv_len, sm_count(), &S, &C);
  const bool bal = use_balanced(B, Hq, Hkv, max_rows);
  if (bal) S = kBalancedParts;
  const size_t need = workspace_bytes_for(T, Hq, S);
  if (workspace == nullptr || workspace_bytes < need) return GQA_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return GQA_ERR_INVALID_ARG;
  float* O_parts = static_cast<float*>(workspace);
  float* lse_parts = O_parts + size_t(S) * size_t(T) * Hq * 256;
  int r = run_split(Q, Kcache, Vcache, kv_lens, cu_rows, O_parts, lse_parts, B, T, Hq, Hkv, Lcap,
                    max_rows, max_kv_len, S, C, static_cast<cudaStream_t>(stream), tree_mask, f16,
                    bal);
  if (r != GQA_OK) return r;
  return attn_lse_merge_impl(f16, O_parts, lse_parts, S, T * Hq, G, out, lse_out, stream,
                             true);
}

// Which mask head a query head reads (DS4Server issue113 README, "Exact scope found
// during review": with head chunking the mask goes unchanged to every chunk's call).
// Chunked when enabled, rows <= 32 and rows * GQA > 32: chunks of min(GQA, 32/rows)
// heads plus a remainder, and the mask's head count must be 1 or every chunk's size.
// Otherwise one call over all Hq heads: 1 or Hq.  Returns false for a mask that does
// not broadcast.
bool mask_head_mode(int rows, int gqa, int Hq, long long mask_heads, bool chunking, int* mode,
                    int* chunk) {
  *chunk = 1;
  const bool chunked = chunking && rows <= 32 && (long long)rows * gqa > 32;
  if (mask_heads == 1) {
    *mode = 0;
    return true;
  }
  if (!chunked) {
    *mode = 1;
    return mask_heads == Hq;
  }
  const int c = gqa < 32 / rows ? gqa : 32 / rows;
  if (gqa % c == 0 && mask_heads == c) {
    *mode = 2;
    *chunk = c;
    return true;
  }
  return false;
}

// Host check of a mask description; fills the kernel's head mode and chunk size.
int check_mask(int B, int Hq, int Hkv, int Lq, int Lkv, int mask_kind,
               const long long* mask_shape, const long long* mask_strides, int head_chunking,
               int* hmode, int* chunk) {
  *hmode = 0;
  *chunk = 1;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lq < 0 || Lkv < 1)
    return GQA_ERR_INVALID_ARG;
  if (mask_kind < GQA_MASK_NONE || mask_kind > GQA_MASK_ADD_F16) return GQA_ERR_INVALID_ARG;
  if (mask_kind == GQA_MASK_NONE) return GQA_OK;
  if (mask_shape == nullptr || mask_strides == nullptr) return GQA_ERR_INVALID_ARG;
  const long long want[4] = {B, -1, Lq, Lkv};
  for (int d = 0; d < 4; ++d) {
    if (mask_shape[d] < 1 || mask_strides[d] < 0) return GQA_ERR_INVALID_ARG;
    if (d != 1 && mask_shape[d] != 1 && mask_shape[d] != want[d]) return GQA_ERR_INVALID_ARG;
  }
  if (Lq > 0 &&
      !mask_head_mode(Lq, Hq / Hkv, Hq, mask_shape[1], head_chunking != 0, hmode, chunk))
    return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

int gqa_attn_masked_impl(bool f16, const void* Q, const void* K, const void* V, const void* G,
                         const void* mask, int mask_kind, const long long* mask_shape,
                         const long long* mask_strides, void* out, float* lse_out, int B,
                         int Hq, int Hkv, int Lq, int Lkv, int causal, int kv_offset,
                         int head_chunking, gqa_stream_t stream) {
  PrefillArgs a{Q, K, V, G, out, lse_out, B, Hq, Hkv, Lq, Lkv, kv_offset};
  const int st = check_mask(B, Hq, Hkv, Lq, Lkv, mask_kind, mask_shape, mask_strides,
                            head_chunking, &a.mask_hmode, &a.mask_chunk);
  if (st != GQA_OK) return st;
  if (causal != 0 && (kv_offset < 0 || (long long)kv_offset + Lq > Lkv))
    return GQA_ERR_INVALID_ARG;
  a.kv_offset = causal != 0 ? kv_offset : 0;
  a.f16 = f16;
  a.masked = true;
  a.causal = causal != 0;
  a.mask_kind = mask_kind;
  if (mask_kind != GQA_MASK_NONE) {
    static const int kElem[5] = {0, 1, 4, 2, 2};
    if (mask == nullptr || !aligned(mask, size_t(kElem[mask_kind]))) return GQA_ERR_INVALID_ARG;
    a.mask = mask;
    for (int d = 0; d < 4; ++d) a.mask_strides[d] = mask_shape[d] == 1 ? 0 : mask_strides[d];
  }
  if (Lq == 0) return GQA_OK;
  if (Q == nullptr || K == nullptr || V == nullptr || out == nullptr) return GQA_ERR_INVALID_ARG;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(out, 16) ||
      (G != nullptr && !aligned(G, 16)) || (lse_out != nullptr && !aligned(lse_out, 4)))
    return GQA_ERR_INVALID_ARG;
  if (Hq / Hkv > 128) return GQA_ERR_UNSUPPORTED;
  if ((long long)Hq * Lq >= (1LL << 31) || (long long)B * Hkv >= (1LL << 31))
    return GQA_ERR_UNSUPPORTED;
  const long long grid = (long long)ceil_div(Lq, prefill_rows_per_tile(Hq / Hkv)) * B * Hkv;
  if (grid >= (1LL << 31)) return GQA_ERR_UNSUPPORTED;
  LaunchCtl ctl;
  if (!make_ctl(&ctl)) return GQA_ERR_CUDA;
  bool encode_failed = false;
  const cudaError_t e = launch_prefill(a, ctl, static_cast<cudaStream_t>(stream), &encode_failed);
  if (encode_failed) return GQA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

// The launch log: a ring of the last kLogSize launches, newest at (g_log_seq - 1).
constexpr int kLogSize = 64;
std::mutex g_log_mu;
gqa_launch_info g_log[kLogSize];
unsigned long long g_log_seq = 0;

}  // namespace

void note_launch(const char* kernel, long long grid, int block, size_t dynamic_smem) {
  gqa_launch_info r{};
  std::strncpy(r.kernel, kernel, sizeof(r.kernel) - 1);
  r.grid = static_cast<unsigned int>(grid);
  r.block = static_cast<unsigned int>(block);
  r.dynamic_smem = static_cast<unsigned int>(dynamic_smem);
  std::lock_guard<std::mutex> lock(g_log_mu);
  r.seq = ++g_log_seq;
  g_log[(r.seq - 1) % kLogSize] = r;
}

int decode_bf16_with_workspace(const void* Q, const void* Kcache, const void* Vcache,
                               const void* G, const int* kv_lens, const int* cu_rows, void* out,
                               float* lse_out, int B, int T, int Hq, int Hkv, int Lcap,
                               int max_rows, int max_kv_len, void* workspace,
                               size_t workspace_bytes, gqa_stream_t stream) {
  return gqa_attn_decode_impl(false, Q, Kcache, Vcache, G, kv_lens, cu_rows, out, lse_out, B, T,
                              Hq, Hkv, Lcap, max_rows, max_kv_len, workspace, workspace_bytes,
                              stream);
}

}  // namespace gqa

using namespace gqa;

extern "C" {

const char* gqa_status_string(int status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported configuration";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_TIMEOUT: return "device wait timed out";
    case GQA_ERR_WORKSPACE: return "workspace too small";
    case GQA_ERR_DEVICE_RANGE: return "device-side range error (kv_lens / cu_rows)";
    default: return "unknown status";
  }
}

const char* gqa_version(void) { return "0.1.0"; }

void gqa_set_wait_timeout_ns(unsigned long long ns) {
  g_timeout_ns.store(ns < 1000000ull ? 1000000ull : ns);
}

int gqa_attn_prefill(const void* Q, const void* K, const void* V, const void* G, void* out,
                     float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv, int kv_offset,
                     gqa_stream_t stream) {
  return gqa_attn_prefill_impl(false, Q, K, V, G, out, lse_out, B, Hq, Hkv, Lq, Lkv, kv_offset,
                               stream);
}
int gqa_attn_prefill_f16(const void* Q, const void* K, const void* V, const void* G, void* out,
                         float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv, int kv_offset,
                         gqa_stream_t stream) {
  return gqa_attn_prefill_impl(true, Q, K, V, G, out, lse_out, B, Hq, Hkv, Lq, Lkv, kv_offset,
                               stream);
}
int gqa_attn_prefill_pair(const void* Q, const void* K, const void* V, const void* G, void* out,
                          float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv, int kv_offset,
                          gqa_stream_t stream) {
  return gqa_attn_prefill_impl(false, Q, K, V, G, out, lse_out, B, Hq, Hkv, Lq, Lkv, kv_offset,
                               stream, true);
}

int gqa_attn_decode_plan(int B, int T, int Hq, int Hkv, int max_rows, int max_kv_len,
                         int* num_splits, int* split_keys) {
  if (num_splits == nullptr || split_keys == nullptr) return GQA_ERR_INVALID_ARG;
  const int st = check_decode_args(B, T, Hq, Hkv, max_kv_len, max_rows, max_kv_len, true);
  if (st != GQA_OK) return st;
  return plan_decode(B, Hq, Hkv, max_rows, max_kv_len, sm_count(), num_splits, split_keys);
}

size_t gqa_attn_decode_workspace_size(int B, int T, int Hq, int Hkv, int max_rows,
                                      int max_kv_len) {
  int S = 0, C = 0;
  if (gqa_attn_decode_plan(B, T, Hq, Hkv, max_rows, max_kv_len, &S, &C) != GQA_OK) return 0;
  return workspace_bytes_for(T, Hq, call_parts(B, Hq, Hkv, max_rows, S));
}

int gqa_attn_decode_split(const void* Q, const void* Kcache, const void* Vcache,
                          const int* kv_lens, const int* cu_rows, float* O_parts,
                          float* lse_parts, int B, int T, int Hq, int Hkv, int Lcap, int max_rows,
                          int max_kv_len, int num_splits, int split_keys, gqa_stream_t stream) {
  return gqa_attn_decode_split_impl(false, Q, Kcache, Vcache, kv_lens, cu_rows, O_parts,
                                    lse_parts, B, T, Hq, Hkv, Lcap, max_rows, max_kv_len,
                                    num_splits, split_keys, stream);
}
int gqa_attn_decode_split_f16(const void* Q, const void* Kcache, const void* Vcache,
                              const int* kv_lens, const int* cu_rows, float* O_parts,
                              float* lse_parts, int B, int T, int Hq, int Hkv, int Lcap,
                              int max_rows, int max_kv_len, int num_splits, int split_keys,
                              gqa_stream_t stream) {
  return gqa_attn_decode_split_impl(true, Q, Kcache, Vcache, kv_lens, cu_rows, O_parts,
                                    lse_parts, B, T, Hq, Hkv, Lcap, max_rows, max_kv_len,
                                    num_splits, split_keys, stream);
}

int attn_lse_merge(const float* O_parts, const float* lse_parts, int S, int N, const void* G,
                   void* out, float* lse_out, gqa_stream_t stream) {
  return attn_lse_merge_impl(false, O_parts, lse_parts, S, N, G, out, lse_out, stream);
}
int attn_lse_merge_f16(const float* O_parts, const float* lse_parts, int S, int N, const void* G,
                       void* out, float* lse_out, gqa_stream_t stream) {
  return attn_lse_merge_impl(true, O_parts, lse_parts, S, N, G, out, lse_out, stream);
}

int gqa_attn_decode(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                    const int* kv_lens, const int* cu_rows, void* out, float* lse_out, int B,
                    int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                    void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
  return gqa_attn_decode_impl(false, Q, Kcache, Vcache, G, kv_lens, cu_rows, out, lse_out, B, T,
                              Hq, Hkv, Lcap, max_rows, max_kv_len, workspace, workspace_bytes,
                              stream);
}
int gqa_attn_decode_f16(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                        const int* kv_lens, const int* cu_rows, void* out, float* lse_out, int B,
                        int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                        void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
  return gqa_attn_decode_impl(true, Q, Kcache, Vcache, G, kv_lens, cu_rows, out, lse_out, B, T,
                              Hq, Hkv, Lcap, max_rows, max_kv_len, workspace, workspace_bytes,
                              stream);
}

int gqa_attn_verify_tree(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                         const int* kv_lens, const int* cu_rows,
                         const unsigned long long* tree_mask, void* out, float* lse_out, int B,
                         int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                         void* workspace, size_t workspace_bytes, gqa_stream_t stream) {
  return gqa_attn_verify_tree_impl(false, Q, Kcache, Vcache, G, kv_lens, cu_rows, tree_mask, out,
                                   lse_out, B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, workspace,
                                   workspace_bytes, stream);
}
int gqa_attn_verify_tree_f16(const void* Q, const void* Kcache, const void* Vcache,
                             const void* G, const int* kv_lens, const int* cu_rows,
                             const unsigned long long* tree_mask, void* out, float* lse_out,
                             int B, int T, int Hq, int Hkv, int Lcap, int max_rows,
                             int max_kv_len, void* workspace, size_t workspace_bytes,
                             gqa_stream_t stream) {
  return gqa_attn_verify_tree_impl(true, Q, Kcache, Vcache, G, kv_lens, cu_rows, tree_mask, out,
                                   lse_out, B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, workspace,
                                   workspace_bytes, stream);
}

int gqa_attn_mask_check(int B, int Hq, int Hkv, int Lq, int Lkv, int mask_kind,
                        const long long* mask_shape, const long long* mask_strides,
                        int head_chunking) {
  int hmode = 0, chunk = 1;
  return check_mask(B, Hq, Hkv, Lq, Lkv, mask_kind, mask_shape, mask_strides, head_chunking,
                    &hmode, &chunk);
}

int gqa_attn_masked(const void* Q, const void* K, const void* V, const void* G, const void* mask,
                    int mask_kind, const long long* mask_shape, const long long* mask_strides,
                    void* out, float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv,
                    int causal, int kv_offset, int head_chunking, gqa_stream_t stream) {
  return gqa_attn_masked_impl(false, Q, K, V, G, mask, mask_kind, mask_shape, mask_strides, out,
                              lse_out, B, Hq, Hkv, Lq, Lkv, causal, kv_offset, head_chunking,
                              stream);
}
int gqa_attn_masked_f16(const void* Q, const void* K, const void* V, const void* G,
                        const void* mask, int mask_kind, const long long* mask_shape,
                        const long long* mask_strides, void* out, float* lse_out, int B, int Hq,
                        int Hkv, int Lq, int Lkv, int causal, int kv_offset, int head_chunking,
                        gqa_stream_t stream) {
  return gqa_attn_masked_impl(true, Q, K, V, G, mask, mask_kind, mask_shape, mask_strides, out,
                              lse_out, B, Hq, Hkv, Lq, Lkv, causal, kv_offset, head_chunking,
                              stream);
}

int gqa_launch_log(gqa_launch_info* out, int max_entries) {
  if (max_entries < 0 || (out == nullptr && max_entries > 0)) return -GQA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_log_mu);
  const unsigned long long have = g_log_seq < kLogSize ? g_log_seq : kLogSize;
  const int n = static_cast<int>(have < static_cast<unsigned long long>(max_entries) ? have
                                                                                     : max_entries);
  for (int i = 0; i < n; ++i) out[i] = g_log[(g_log_seq - 1 - i) % kLogSize];
  return n;
}

int gqa_last_device_status(gqa_stream_t stream) {
  int* p = status_ptr();
  if (p == nullptr) return GQA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return GQA_ERR_CUDA;
  if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return GQA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GQA_ERR_CUDA;
  return v;
}

}  // extern "C"
