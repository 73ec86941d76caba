/*
 * gqa_attn.h - C ABI of libgqa_attn.so: causal grouped-query attention at
 * head_dim 256 with sigmoid output gating, for NVIDIA GB300 (sm_103a).
 *
 *     out = softmax(Q K^T / 16 + causal/offset mask) V  (elementwise *)  sigmoid(G)
 *
 * Sources for the operation (page, section):
 *   - TensorFold PR #1009, "Receipt", attention contract paragraph: decode rows and
 *     prompt rows at 24 query heads over 4 KV heads and 16 over 2, checked against
 *     float64 gated attention; decode runs over cache chunks whose partial results
 *     are merged (its control "a merge dropping later tail chunks").
 *   - TensorFold PR #1009, "Design: one engine": gated full attention layers.
 *   - d-inference PR #640, "Summary": head_dim 256 attention, FP16 and BF16 symbols.
 *   - DS4Server issue113 README, opening rule: query heads inside each KV group
 *     share that group's K/V.
 *
 * Conventions shared by every entry point:
 *   - head_dim D is fixed at 256; every tensor is bf16, contiguous, row-major,
 *     and 16-byte aligned, unless stated otherwise.  Each attention entry point
 *     has an `_f16` twin (declared at the end) with the same arguments, rules and
 *     arithmetic whose Q, K, V, G and out are fp16 instead: the d-inference page
 *     ships FP16 and BF16 symbols of its head_dim-256 kernel.
 *   - Query head h reads KV head h / (Hq / Hkv) (consecutive groups).
 *   - Scores are scaled by 1/16 = 1/sqrt(256).  Softmax sums and all accumulation
 *     are fp32; the output is rounded once to bf16 (round to nearest even).
 *   - G may be NULL: no gate (the output is the plain attention).
 *   - lse outputs, when requested, are fp32 natural-log sum-exp of the scaled
 *     scores over the keys a row sees (-inf for a row that sees no key).
 *   - A row that sees no key outputs zeros.
 *   - Non-finite inputs: a key a row does not see is excluded from that row's
 *     sums, never weighted by probability 0.  So NaN or +-Inf anywhere in the K
 *     or V row of such a key (cache rows at or past kv_len, keys after the last
 *     prompt row, keys the causal rule, a tree mask or a general mask hides from
 *     the row while other rows of the call see them) never changes that row's
 *     output, bit for bit.  Non-finite Q, G, and K/V of keys a row sees propagate
 *     as IEEE float64 arithmetic of the formula would: a NaN score or value gives
 *     NaN, an Inf value under a positive probability gives +-Inf, a -Inf gate
 *     gives 0.  Finite inputs pay one check of each tile's outputs; a tile whose
 *     outputs hold a NaN / Inf is computed again with the non-finite V elements
 *     of keys some of its rows do not see (in fp16 on the tensor-memory kernels:
 *     of every key, as an fp16 P rounds to 0 25 log2 units below the row's
 *     maximum) taken out of the tensor-core product and added back for the rows
 *     that see them.  Limits: the general-mask calls and the fp16 calls on the
 *     tensor-memory kernels (prefill; decode / verify groups of 17 packed rows or
 *     more) handle up to 256 keys (384 on CTA pairs) with a non-finite V element
 *     per tile of query rows and KV head (every other call: any number); past
 *     that, rows that do not see the further keys may read NaN.  fp16 decode /
 *     verify groups of at most 16 packed rows (the cp.async kernel): a visible
 *     +-Inf V value at a key 25 or more log2 units below the row's maximum
 *     gives NaN, not +-Inf.  Probabilities and merge weights are fp32: a key
 *     more than 126 log2 units below the row's maximum has probability 0 (a
 *     +-Inf V value there gives NaN, except on the fp16 tensor-memory kernels),
 *     and a split part that far below has merge weight 0 (its values do not
 *     reach the output).
 *   - Ownership: the caller owns every buffer.  The library never allocates
 *     device memory; the decode workspace is caller-provided.
 *   - Streams: every call is asynchronous on `stream` (may be 0 = legacy default
 *     stream).  Pointers are device pointers unless a parameter says "host".
 *   - Errors: arguments are validated on the host before any launch; an invalid
 *     call returns GQA_ERR_INVALID_ARG (or GQA_ERR_UNSUPPORTED) and launches
 *     nothing.  A failed launch returns GQA_ERR_CUDA.  Conditions only the device
 *     can see (a kv length beyond the cache, a wait that timed out) are recorded
 *     in a device status word that gqa_last_device_status() reads; the kernel
 *     skips the offending work instead of faulting.
 *   - A call with no rows (Lq = 0, T = 0, N = 0) returns GQA_OK and launches
 *     nothing.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (a cudaStream_t). */
typedef void* gqa_stream_t;

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1, /* bad size, NULL or misaligned pointer, bad geometry   */
  GQA_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement         */
  GQA_ERR_CUDA = 3,        /* a CUDA call or launch failed                         */
  GQA_ERR_TIMEOUT = 4,     /* device: a bounded wait ran out (kernel returned)     */
  GQA_ERR_WORKSPACE = 5,   /* decode workspace too small                           */
  GQA_ERR_DEVICE_RANGE = 6 /* device: kv_lens / cu_rows out of range (work skipped) */
} gqa_status;

/* Static, NUL-terminated description of a status code. */
const char* gqa_status_string(int status);

/* Library version, "major.minor.patch". */
const char* gqa_version(void);

/*
 * Prompt rows (prefill), possibly a chunk of a longer prompt.
 *
 *   out[b,h,i,:] = sum_{j <= kv_offset+i} softmax_j(Q[b,h,i,:].K[b,g,j,:]/16) V[b,g,j,:]
 *                  * sigmoid(G[b,h,i,:]),   g = h / (Hq/Hkv)
 *
 * Q, G, out: [B, Hq, Lq, 256] bf16.  K, V: [B, Hkv, Lkv, 256] bf16.
 * lse_out: NULL, or fp32 [B, Hq, Lq].
 * Row i sits at absolute position kv_offset + i; keys at positions above
 * kv_offset + Lq - 1 are never read (they may hold anything, NaN included).
 * Requires B, Hq, Hkv >= 1, Hq % Hkv == 0, Hq/Hkv <= 128, Lq >= 0,
 * kv_offset >= 0, kv_offset + Lq <= Lkv, Lkv < 2^31.
 * Runs on tcgen05 tensor cores (TMEM accumulators, TMA-staged tiles); a prompt
 * whose last row sees 2048 keys or more (kv_offset + Lq >= 2048) runs on CTA pairs
 * (see gqa_attn_prefill_pair), a shorter one on single CTAs.
 */
int gqa_attn_prefill(const void* Q, const void* K, const void* V, const void* G,
                     void* out, float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv,
                     int kv_offset, gqa_stream_t stream);

/*
 * gqa_attn_prefill computed by CTA pairs whatever the prompt length: two CTAs of a
 * cluster take two row tiles of a KV group and share each 128-key K/V tile (each
 * copies half of it; the products, tcgen05 .cta_group::2 with M = 256, read both
 * halves).  Same arguments, rules, errors and results (within the parity bar; the
 * single-CTA form may differ in the last bit of an output) as gqa_attn_prefill,
 * which picks this form for long prompts by itself.
 */
int gqa_attn_prefill_pair(const void* Q, const void* K, const void* V, const void* G,
                          void* out, float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv,
                          int kv_offset, gqa_stream_t stream);

/*
 * Decode (one row per sequence) and chain verify (r_b rows per sequence, causal
 * within the rows) against a contiguous KV cache.
 *
 * Q, G, out: [T, Hq, 256] bf16, token-major; the rows of sequence b are tokens
 *   cu_rows[b] .. cu_rows[b+1]-1 (T = cu_rows[B]).
 * Kcache, Vcache: [B, Hkv, Lcap, 256] bf16.
 * kv_lens: int32 [B] (device): keys held for sequence b, counting its new rows;
 *   row i (0-based of r_b) sees keys j < kv_lens[b] - r_b + i + 1.  Cache rows at
 *   or beyond kv_lens[b] never affect the result (they may hold anything, NaN
 *   included): the mma.sync kernel does not read them, the tcgen05 kernel may copy
 *   some into shared memory and clears them there before use.
 * cu_rows: int32 [B+1] (device) exclusive prefix sum of rows, or NULL for one row
 *   per sequence (then T must equal B and max_rows must be 1).
 * lse_out: NULL, or fp32 [T, Hq].
 * T, max_rows, max_kv_len (host): total rows, an upper bound on r_b and on
 *   kv_lens[b]; they size the grid.  Sequences whose kv_lens/cu_rows break these
 *   bounds (or kv_lens[b] < r_b, or kv_lens[b] > Lcap) are skipped on the device
 *   and GQA_ERR_DEVICE_RANGE is recorded.
 * workspace: device buffer of at least gqa_attn_decode_workspace_size() bytes,
 *   16-byte aligned; holds the split partial results.
 * The call runs gqa_attn_decode_split() then attn_lse_merge() on `stream`.
 */
size_t gqa_attn_decode_workspace_size(int B, int T, int Hq, int Hkv, int max_rows,
                                      int max_kv_len);
int gqa_attn_decode(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                    const int* kv_lens, const int* cu_rows, void* out, float* lse_out,
                    int B, int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                    void* workspace, size_t workspace_bytes, gqa_stream_t stream);

/*
 * Draft verify over a token tree (TensorFold PR #1009, "Receipt": decode shapes
 * plan chains and trees).  As gqa_attn_decode, except that new row i of a sequence
 * sees every key before the sequence's new rows (positions < kv_lens[b] - r_b) and
 * the new key at position kv_lens[b] - r_b + k exactly when bit k of
 * tree_mask[t] is set (its ancestors and itself; a chain is bits 0..i).
 * tree_mask: uint64 [T] (device, 8-byte aligned), one mask per new row.
 * cu_rows is required; max_rows <= 64 (GQA_ERR_UNSUPPORTED above).  Same workspace
 * size and split plan as gqa_attn_decode.  A row whose mask selects no key and that
 * has no earlier key outputs zeros.
 */
int gqa_attn_verify_tree(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                         const int* kv_lens, const int* cu_rows,
                         const unsigned long long* tree_mask, void* out, float* lse_out, int B,
                         int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                         void* workspace, size_t workspace_bytes, gqa_stream_t stream);

/*
 * The fixed split plan: the number of key splits S and the keys per split (a
 * multiple of 64).  gqa_attn_decode uses it on the tcgen05 path and for B > 256;
 * on the mma.sync path with B <= 256 it runs balanced shares with 16 part slots
 * instead (see gqa_attn_decode_split).  Split s of sequence b covers keys
 * [s*split_keys, min((s+1)*split_keys, kv_lens[b])).  Host-only; returns
 * GQA_ERR_INVALID_ARG for bad sizes.
 */
int gqa_attn_decode_plan(int B, int T, int Hq, int Hkv, int max_rows, int max_kv_len,
                         int* num_splits, int* split_keys);

/*
 * First half of gqa_attn_decode: per (sequence, KV group, key split), the
 * attention of all of the group's query heads x rows over the split's keys,
 * written as normalised partial results for attn_lse_merge():
 *   O_parts  fp32 [num_splits, T*Hq, 256]: sum_j p_j V_j / l over the split's keys
 *   lse_parts fp32 [num_splits, T*Hq]: m + ln l, -inf when the row sees no key of
 *   the split (its O_parts row is then not written).
 * Row n of the parts is output row (t, h) with n = t*Hq + h.
 * num_splits >= 1 and split_keys (a positive multiple of 64) with
 * num_splits*split_keys >= max_kv_len; gqa_attn_decode_plan() gives the defaults.
 * split_keys = 0 selects balanced shares (the form gqa_attn_decode uses on the
 * mma.sync path, i.e. at most 16 packed rows per group, with B <= 256;
 * otherwise GQA_ERR_UNSUPPORTED): the keys of all (sequence, KV group, row block)
 * ranges are laid end to end in 32-key tiles and cut into equal shares, one per
 * resident CTA, so ragged lengths cost no tail; a range split among k CTAs gets
 * parts 0..k-1 and lse -inf in parts k..num_splits-1.  num_splits >= 3 is then the
 * part capacity per row (gqa_attn_decode uses 16); the shares are never cut so
 * finely that a range needs more.
 * Kernel: when a KV group packs more than 16 rows (max_rows x Hq/Hkv >= 17) and
 * split_keys is a multiple of 128, the split runs on tcgen05 tensor cores (TMEM
 * accumulators, TMA-staged tiles); otherwise on an mma.sync kernel with 16-byte
 * cp.async cache reads.  Both give the same partial results up to rounding.
 */
int gqa_attn_decode_split(const void* Q, const void* Kcache, const void* Vcache,
                          const int* kv_lens, const int* cu_rows, float* O_parts,
                          float* lse_parts, int B, int T, int Hq, int Hkv, int Lcap,
                          int max_rows, int max_kv_len, int num_splits, int split_keys,
                          gqa_stream_t stream);

/*
 * Merge S partial results of N rows computed over disjoint key sets:
 *   out[n,:] = (sum_s exp(lse_s) O_s[n,:]) / (sum_s exp(lse_s))  * sigmoid(G[n,:])
 * O_parts fp32 [S, N, 256], each part normalised (O_s / l_s); lse_parts fp32
 * [S, N] = m_s + ln l_s, -inf for an empty part (weight 0, its O row is never
 * read).  G: NULL (no gate) or bf16 [N, 256].  out: bf16 [N, 256].  lse_out:
 * NULL or fp32 [N].  A row whose parts are all empty gets zeros and lse -inf.
 * This is the tail-chunk merge of the TensorFold attention contract; it also lets
 * a caller compose results over longer contexts or key shards.
 * O_parts and lse_parts need 16- and 4-byte alignment.
 */
int attn_lse_merge(const float* O_parts, const float* lse_parts, int S, int N,
                   const void* G, void* out, float* lse_out, gqa_stream_t stream);

/*
 * Decode / chain verify for callers that cannot allocate device memory: serving
 * loops that must not touch a device allocator between steps (an allocation can
 * stall on device-wide synchronisation or fail under memory pressure mid-request),
 * plug-ins whose host application hands them only fixed input and output buffers.
 * The paper has
 * no counterpart: this is a library convenience.  It is gqa_attn_decode with a
 * workspace owned by the library: the same inputs, outputs, argument checks, plan,
 * kernels and results (bit for bit), but the split partial results live in a fixed
 * 16 MiB area of device memory (a file-scope __device__ array, held by every GPU
 * that loads the library until the process exits), so the caller passes no
 * workspace; the call itself allocates nothing.
 * Limit: gqa_attn_decode_workspace_size() for the same sizes must not exceed
 * 16 MiB (16,777,216 bytes); larger calls return GQA_ERR_WORKSPACE and launch
 * nothing.
 * The first call on a device looks up the area's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  All calls on a device share the area: calls whose kernels
 * may overlap on the GPU (unordered streams) race on it and must not be issued.
 */
int gqa_attn_decode_noalloc(const void* Q, const void* Kcache, const void* Vcache,
                            const void* G, const int* kv_lens, const int* cu_rows, void* out,
                            float* lse_out, int B, int T, int Hq, int Hkv, int Lcap,
                            int max_rows, int max_kv_len, gqa_stream_t stream);

/*
 * Launch log: the library notes, on the host, every kernel launch it makes - the
 * kernel and its instance, and the grid, block and dynamic shared memory the launch
 * used - in a ring holding the last 64 launches of the process.  gqa_launch_log
 * copies up to max_entries of them into `out` (host memory owned by the caller),
 * newest first, and returns how many it copied (0 before any launch).  A launch
 * the CUDA runtime refused is not logged.  Returns GQA_ERR_INVALID_ARG (as a
 * negative number, -1) for max_entries < 0, or for out == NULL with
 * max_entries > 0.  Thread-safe; makes no CUDA call.
 */
typedef struct gqa_launch_info {
  char kernel[64];              /* kernel and instance, NUL-terminated */
  unsigned long long seq;       /* 1 for the process's first launch, then 2, 3, ... */
  unsigned int grid;            /* CTAs (the grids are one-dimensional) */
  unsigned int block;           /* threads per CTA */
  unsigned int dynamic_smem;    /* bytes of dynamic shared memory per CTA */
} gqa_launch_info;

int gqa_launch_log(gqa_launch_info* out, int max_entries);

/*
 * Synchronises `stream`, then reads and clears the device status word that the
 * kernels set (GQA_ERR_TIMEOUT, GQA_ERR_DEVICE_RANGE); GQA_OK when clear.
 * Returns GQA_ERR_CUDA if the synchronisation fails.
 */
int gqa_last_device_status(gqa_stream_t stream);

/*
 * Bound (in nanoseconds) on every spin wait inside the kernels; after it runs
 * out the kernel records GQA_ERR_TIMEOUT and returns.  Default 2e9 (2 s).
 * Host-only setter, takes effect for later launches.  Values < 1e6 are clamped
 * to 1e6.
 */
void gqa_set_wait_timeout_ns(unsigned long long ns);

/*
 * KV-cache append (TensorFold PR #1009, "Receipt": packing, append and keep are
 * compared bit for bit).  Writes the new K and V rows of each sequence after the
 * keys it holds: Kcache[b, g, kv_lens[b] + i, :] = Knew[cu_rows[b] + i, g, :]
 * (likewise V), i < rows of b.  This is also the layout change ("pack") from the
 * token-major projection output to the head-major cache.
 * Knew, Vnew: bf16 [T, Hkv, 256] (device); Kcache, Vcache: [B, Hkv, Lcap, 256];
 * kv_lens: int32 [B] (device), keys held before the append (not updated here);
 * cu_rows: int32 [B+1] (device) or NULL for one row per sequence (T == B).
 * A row that would land at or past Lcap is skipped and GQA_ERR_DEVICE_RANGE is
 * recorded.  Bit-exact copies.
 */
int gqa_kv_append(const void* Knew, const void* Vnew, const int* cu_rows, const int* kv_lens,
                  void* Kcache, void* Vcache, int B, int T, int Hkv, int Lcap,
                  gqa_stream_t stream);

/*
 * KV-cache keep after draft verification.  Sequence b holds r_b = cu_rows[b+1] -
 * cu_rows[b] draft rows at positions kv_lens[b] - r_b .. kv_lens[b] - 1; the
 * accepted ones, keep_idx[cu_keep[b] .. cu_keep[b+1]) (draft-row indices, strictly
 * increasing), move in order to positions kv_lens[b] - r_b + k, in place.
 * kv_lens_out: NULL or int32 [B] (device, must not alias kv_lens) receiving
 * kv_lens[b] - r_b + (number kept).  A sequence with an invalid keep list is left
 * untouched and GQA_ERR_DEVICE_RANGE is recorded.  Bit-exact copies.
 */
int gqa_kv_keep(void* Kcache, void* Vcache, const int* kv_lens, const int* cu_rows,
                const int* keep_idx, const int* cu_keep, int* kv_lens_out, int B, int Hkv,
                int Lcap, gqa_stream_t stream);

/*
 * Failure-detection self test.  Launches one warp that runs the kernels' bounded
 * spin wait (the same code every mbarrier wait in the kernels uses) on a barrier
 * that nothing completes.  After the bound (gqa_set_wait_timeout_ns) it records
 * GQA_ERR_TIMEOUT in the device status word and returns; the context stays usable.
 * elapsed_ns: NULL, or a device pointer (8-byte aligned) that receives the time
 * the wait took, from the global timer.  Returns GQA_ERR_CUDA if the launch fails.
 * Read the outcome with gqa_last_device_status().
 */
int gqa_selftest_wait_timeout(unsigned long long* elapsed_ns, gqa_stream_t stream);

/*
 * Gated attention with a general mask: the dense SDPA consumer of the DS4Server
 * issue113 README ("Exact scope found during review"; its fixtures cover no,
 * bool, additive, two-dimensional, full-head and chunk-local masks, and mask
 * rejections), in the prefill layout:
 *   Q, G, out: [B, Hq, Lq, 256]; K, V: [B, Hkv, Lkv, 256]; bf16 (fp16: _f16).
 *   score(i, j) = Q_i . K_j / 16 + bias(i, j); a key is excluded when a bool mask
 *   holds 0 there, when an additive mask holds -inf, or (causal != 0) when
 *   j > kv_offset + i.  A row that keeps no key outputs zeros, lse -inf.
 * mask: NULL with mask_kind GQA_MASK_NONE (then only the causal rule, or none), or
 *   a device array read at  mask[b*s0 + hm*s1 + i*s2 + j*s3]  with mask_shape /
 *   mask_strides (host arrays of 4, elements, order [batch, head, row, key]); a
 *   dimension of size 1 broadcasts (its stride is ignored); otherwise batch must
 *   be B, row Lq, key Lkv.  Strides >= 0; the pointer aligned to its element.
 *   GQA_MASK_BOOL: uint8, nonzero = attend.  GQA_MASK_ADD_F32 / _BF16 / _F16: a
 *   value added to the scaled score (natural-log units).
 * Head rule (head_chunking != 0 is the page's default): when Lq <= 32 and
 *   Lq * GQA > 32, each KV group's heads run in chunks of min(GQA, 32 / Lq) heads
 *   (a smaller remainder last) and the mask is passed unchanged to every chunk,
 *   so its head count must be 1 or equal to every chunk's size, and query head
 *   k of a chunk reads mask head k (chunk-local).  Otherwise (or head_chunking
 *   == 0) the head count must be 1 or Hq and query head h reads mask head h.
 *   A mask that does not broadcast returns GQA_ERR_INVALID_ARG, launching
 *   nothing.  Head chunking changes no value: only which masks are accepted.
 * causal: 0 = every key of Lkv may be seen; 1 = also j <= kv_offset + i (then
 *   0 <= kv_offset, kv_offset + Lq <= Lkv).  Runs on the tcgen05 prefill kernel.
 */
typedef enum {
  GQA_MASK_NONE = 0,
  GQA_MASK_BOOL = 1,
  GQA_MASK_ADD_F32 = 2,
  GQA_MASK_ADD_BF16 = 3,
  GQA_MASK_ADD_F16 = 4
} gqa_mask_kind;

int gqa_attn_masked(const void* Q, const void* K, const void* V, const void* G, const void* mask,
                    int mask_kind, const long long* mask_shape, const long long* mask_strides,
                    void* out, float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv,
                    int causal, int kv_offset, int head_chunking, gqa_stream_t stream);

/*
 * Host-only check of a mask description against gqa_attn_masked's rules (sizes,
 * kind, broadcast of batch / row / key dimensions, strides >= 0, the head rule);
 * GQA_OK or GQA_ERR_INVALID_ARG.  Makes no CUDA call.  gqa_attn_masked runs the
 * same check first.
 */
int gqa_attn_mask_check(int B, int Hq, int Hkv, int Lq, int Lkv, int mask_kind,
                        const long long* mask_shape, const long long* mask_strides,
                        int head_chunking);

/*
 * FP16 twins (d-inference PR #640, "Summary": FP16 and BF16 symbols of the
 * head_dim-256 kernel).  Same arguments, rules, errors and arithmetic as the
 * bf16 entry point of the same name without `_f16`; Q, K/Kcache, V/Vcache, G and
 * out are fp16 (IEEE binary16) instead of bf16.  P enters the P.V product as
 * fp16; the tensor-core kernels rescale a row's running sum whenever its maximum
 * grows by more than 15 in log2 units, so every P stays at or below 2^15 = 32768,
 * inside fp16's range (bf16 uses 32).  Scores, softmax sums and accumulation stay fp32.
 * Partial results (O_parts, lse_parts) are fp32 in both types.  gqa_kv_append
 * and gqa_kv_keep copy 16-bit elements and serve both types unchanged.
 */
int gqa_attn_prefill_f16(const void* Q, const void* K, const void* V, const void* G, void* out,
                         float* lse_out, int B, int Hq, int Hkv, int Lq, int Lkv, int kv_offset,
                         gqa_stream_t stream);
int gqa_attn_decode_f16(const void* Q, const void* Kcache, const void* Vcache, const void* G,
                        const int* kv_lens, const int* cu_rows, void* out, float* lse_out, int B,
                        int T, int Hq, int Hkv, int Lcap, int max_rows, int max_kv_len,
                        void* workspace, size_t workspace_bytes, gqa_stream_t stream);
int gqa_attn_verify_tree_f16(const void* Q, const void* Kcache, const void* Vcache,
                             const void* G, const int* kv_lens, const int* cu_rows,
                             const unsigned long long* tree_mask, void* out, float* lse_out,
                             int B, int T, int Hq, int Hkv, int Lcap, int max_rows,
                             int max_kv_len, void* workspace, size_t workspace_bytes,
                             gqa_stream_t stream);
int gqa_attn_decode_split_f16(const void* Q, const void* Kcache, const void* Vcache,
                              const int* kv_lens, const int* cu_rows, float* O_parts,
                              float* lse_parts, int B, int T, int Hq, int Hkv, int Lcap,
                              int max_rows, int max_kv_len, int num_splits, int split_keys,
                              gqa_stream_t stream);
int attn_lse_merge_f16(const float* O_parts, const float* lse_parts, int S, int N,
                       const void* G, void* out, float* lse_out, gqa_stream_t stream);
int gqa_attn_masked_f16(const void* Q, const void* K, const void* V, const void* G,
                        const void* mask, int mask_kind, const long long* mask_shape,
                        const long long* mask_strides, void* out, float* lse_out, int B, int Hq,
                        int Hkv, int Lq, int Lkv, int causal, int kv_offset, int head_chunking,
                        gqa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_H */
