// Gated causal GQA attention on sm_103a tensor cores: prompt rows (prefill) and,
// in split mode, decode / verify rows against a KV cache over one key split.
//
// One CTA computes one tile of 128 packed rows: R = floor(128/GQA) consecutive
// query rows of every query head of one KV group (row m of the tile is head
// m / R, query row r0 + m % R), so each K/V tile staged in shared memory serves
// the whole group (DS4Server issue113 README, opening rule: the heads of a KV
// group share its K/V).  Rows past R*GQA are padding and are never stored.
//
// Roles (320 threads; 352 for the general-mask form):
//   warp 0      TMA producer: Q tile once, then K_0, K_1, V_0, K_2, V_1, ... as whole
//               tiles of kN keys x 256 dims (four 128-byte-swizzled column blocks of
//               64 dims), K tiles into a ring of kKS slots and V tiles into a ring of
//               kVS slots: K_{j+1} then waits only on S_{j+1-kKS}, never on a PV.
//   warp 1      TMEM allocator and MMA issuer (one thread):
//                 S_j = Q K_j^T          M=128, N=kN, K=256, A and B from smem
//                 O  += P_j V_j          M=128, N=256, K=kN, A (P) from TMEM
//               in the order S_0, S_1, PV_0, S_2, PV_1, ..., so the tensor pipe
//               works on S_{j+1} while the softmax runs on S_j.
//   warps 2..9  softmax and epilogue; TMEM lane = tile row, so a thread owns a row
//               and a pair of warps (w, w+4) shares its lanes: the first takes the
//               first kN/2 keys of the tile, the second the rest; the two exchange
//               row maxima and sums through shared memory.
//   warp 10     general-mask form only: stages the tile's mask rows in shared memory
//               when one mask head serves all query heads.
// TMEM (512 columns): O at 0..255 (fp32), S double buffer at 256 and 256 + kN;
// P_j is written as bf16 pairs over the first kN/4 columns of each half of S_j.
//
// Softmax: fp32, base 2 with the 1/16 scale folded in; a row's running max (and
// its O row in TMEM) is only moved when a tile raises it by more than 32, so
// p <= 2^32 and the fp32 sums stay far from overflow (l < 2^32 x keys) while
// rescales - a TMEM round trip of the whole O row - stay rare.  Masked keys get
// probability exactly 0 by selection, never exp(-inf)*0 arithmetic.
// Keys a row does not see are excluded from its sums, never weighted by 0, whatever
// their K and V hold (the TensorFold PR's second comment predicts NaN from a masked
// key's Inf value times probability 0).  K only enters masked scores, which are
// replaced.  V rows of such keys do enter the P.V product with probability 0, so a
// NaN / Inf there would make the row NaN: the epilogue checks the CTA's stored outputs
// and, only when one of them is NaN / Inf, the CTA runs its tile again in a cleaning
// pass - every V tile is checked from the first key some row may not see, its NaN /
// Inf elements are set to 0 before the product, and p * V of the original elements
// is added back in the epilogue of the rows that see those keys.  Inputs without such
// values take pass 0 alone (one check of the stored tile per CTA).
// Epilogue: out = O / l * sigmoid(G), rounded once to bf16; the gate tile arrives by
// TMA in Q's buffer and the output tile leaves by TMA stores from the K/V ring, half
// of its column blocks while the other half is still being computed.
//
// Split mode (decode / chain verify, TensorFold PR #1009 "Receipt": decode over cache
// chunks whose partial results are merged): one CTA takes R = floor(128/GQA) new
// tokens x all GQA heads of one (sequence, KV group) - row m is token m / GQA, head
// m % GQA, matching the token-major [T, Hq, 256] layout - against the keys of one
// split [k_lo, k_hi), k_lo a multiple of kN.  Sequence lengths live on the device,
// so the cache tensor map spans the whole capacity: K columns past kv_len are
// masked by selection, and the producer warp zeroes the V rows past kv_len of the
// CTA's last tile (its last copy) in shared memory before the last PV may start, so
// cache padding (any bits, NaN included) never meets a zero probability inside the
// MMA; keys of the split that some rows do not see are handled as above (the check
// covers the fp32 partial outputs).  The epilogue writes the normalised
// partial O / l (fp32) and lse = m + ln l for attn_lse_merge, or lse = -inf for a
// row that sees no key of the split.
#include <climits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include <mutex>

#include "internal.h"
#include "ptx_sm100.cuh"
#include "tc_common.cuh"

namespace gqa {
namespace {

constexpr int kKS = 1;                        // K ring slots (whole tiles)
constexpr int kVS = 1;                        // V ring slots
constexpr int kSlots = kKS + kVS;
static_assert(kSlots * kTileBytes >= kQBytes, "the output tile is staged in the K/V ring");
constexpr int kThreads = 320;
// Cleaning pass: keys whose V rows held a NaN / Inf element among the candidate keys
// (see cand_lo in the kernel); at most kMaxHits per CTA are handled exactly (rows past
// that are left as they are).  A causal prompt tile's candidates (its diagonal and the
// rest of its last key tile) and a verify tile's are fewer than 256; a general mask,
// and fp16, make every key a candidate.
constexpr int kMaxHits = 256;
// General masks with one mask head for all query heads: the tile's mask rows (R query
// rows x kN keys, each row padded by 16 bytes so that reads of different rows fall on
// different banks) are staged in two slots behind the Smem block.
constexpr int kMaskSlotBytes = 11264;
template <bool kF16>
constexpr uint32_t idesc_s() { return ptx::idesc_f32acc(kM, kN, 0, 0, kF16 ? 0u : 1u); }   // Q, K K-major
template <bool kF16>
constexpr uint32_t idesc_pv() { return ptx::idesc_f32acc(kM, 256, 0, 1, kF16 ? 0u : 1u); } // V MN-major

struct __align__(1024) Smem {
  uint8_t q[kQBytes];
  uint8_t kv[kSlots][kTileBytes];   // K ring: slots 0..kKS-1, V ring: the rest
  uint64_t q_full;
  uint64_t kv_full[kSlots];
  uint64_t kv_empty[kSlots];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done;
  uint64_t o_final;
  uint64_t drain;
  uint64_t v_clean;            // split mode: the last V tile's padding rows are zeroed
  uint64_t q_free;             // prefill: every S product has read Q (its buffer takes G)
  uint64_t g_full;             // prefill: the gate tile has landed in Q's buffer
  uint64_t mask_full[2];       // staged mask: slot holds tile j's mask rows
  uint64_t mask_empty[2];      // staged mask: every softmax warp is done with the slot
  uint32_t tmem_base;
  int abort;
  int zero;
  float red[2][2][kM];     // [tile parity][half][row]: row maxima, then row sums
  int ok[2][2][kM];        // [tile parity][half][row]: the thread's waits succeeded
  // Cleaning pass (see the kernel)
  uint64_t vs_ready[2];             // [j & 1]: V tile j is cleaned and its hits published
  uint32_t tile_hits[2][kN / 32];   // [j & 1]: bit c = key c of tile j is a hit
  int tile_base[2];                 // [j & 1]: hit-list index of tile j's first hit
  int n_hits;                       // hit-list length
  int need_clean;                   // a stored output of pass 0 is NaN / Inf
  int hit_key[kMaxHits];            // hit list: key indices, increasing
  uint32_t pz[kM][kMaxHits / 32];   // [row]: bit i = the row's probability for hit i is 0
};

struct Params {
  const uint16_t* G;        // bf16 or fp16 bits
  const uint16_t* V;        // V [B*Hkv, v_rows, 256]: re-read by the cleaning pass
  long long v_rows;         // rows per (batch, KV head): Lkv (prefill) or Lcap (split)
  uint16_t* out;
  float* lse;
  int B, Hq, Hkv, Lq, kv_offset, gqa, R, n_rtiles;
  // split mode
  const int* kv_lens;
  const int* cu_rows;
  const unsigned long long* tree_mask;   // split mode, tree verify; null: chain
  float* O_parts;
  float* lse_parts;
  int T, Lcap, max_rows, max_kv_len, split_keys, num_splits;
  // general-mask prefill (kMask)
  const void* mask;
  int mask_kind, mask_hmode, mask_chunk, causal, Lkv;
  long long ms_b, ms_h, ms_i, ms_j;
  int mask_stage;           // mask rows staged in shared memory (see kMaskSlotBytes)
  LaunchCtl ctl;
};

__device__ __forceinline__ void fail(Smem& sm, const Params& p) {
  sm.abort = 1;
  record_status(p.ctl.status, GQA_ERR_TIMEOUT);
}

// Applies the mask to one row's raw scores s[0..n) (keys key0 .. key0+n-1, keys at
// or past `lim` already -inf): an excluded key becomes -inf, a bias a moves the raw
// score by 16a, so that the scaled score moves by a.  Keys past lim are never read.
template <int kKind, typename E, int kN_>
__device__ __forceinline__ void apply_mask_row(uint32_t (&s)[kN_], const E* row, long long sj,
                                               int key0, int lim) {
  auto put = [&](int c, float a) {
    const float v = __uint_as_float(s[c]);
    s[c] = __float_as_uint(a == -INFINITY ? -INFINITY : fmaf(16.f, a, v));
  };
  constexpr int kVec = 16 / int(sizeof(E));
  const E* m = row + (long long)key0 * sj;
  if (sj == 1 && key0 + kN_ <= lim && (reinterpret_cast<uintptr_t>(m) & 15) == 0) {
#pragma unroll
    for (int c0 = 0; c0 < kN_; c0 += kVec) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(m + c0));
      const E* e = reinterpret_cast<const E*>(&u);
#pragma unroll
      for (int v = 0; v < kVec; ++v) put(c0 + v, mask_elem<kKind>(e[v]));
    }
  } else {
#pragma unroll
    for (int c = 0; c < kN_; ++c)
      if (key0 + c < lim) put(c, mask_elem<kKind>(__ldg(m + (long long)c * sj)));
  }
}

// The same for a row staged in shared memory (16-byte aligned, kN_ elements present,
// zeros past the mask's last key).
template <int kKind, typename E, int kN_>
__device__ __forceinline__ void apply_mask_row_smem(uint32_t (&s)[kN_], const E* row, int key0,
                                                    int lim) {
  constexpr int kVec = 16 / int(sizeof(E));
  static_assert(kVec % 2 == 0, "keys go in pairs");
  if (key0 + kN_ <= lim) {
    // Every key of the row's share is causally visible: no per-key check.  A bool
    // mask selects; an additive one moves pairs of scores by one packed fma.
#pragma unroll
    for (int c0 = 0; c0 < kN_; c0 += kVec) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + c0);
      const E* e = reinterpret_cast<const E*>(&u);
#pragma unroll
      for (int v = 0; v < kVec; v += 2) {
        if constexpr (kKind == 1) {
          if (!e[v]) s[c0 + v] = __float_as_uint(-INFINITY);
          if (!e[v + 1]) s[c0 + v + 1] = __float_as_uint(-INFINITY);
        } else {
          const float a0 = mask_elem<kKind>(e[v]);
          const float a1 = mask_elem<kKind>(e[v + 1]);
          const float2 x = fma2(make_float2(16.f, 16.f), make_float2(a0, a1),
                                make_float2(__uint_as_float(s[c0 + v]),
                                            __uint_as_float(s[c0 + v + 1])));
          s[c0 + v] = __float_as_uint(a0 == -INFINITY ? -INFINITY : x.x);
          s[c0 + v + 1] = __float_as_uint(a1 == -INFINITY ? -INFINITY : x.y);
        }
      }
    }
    return;
  }
#pragma unroll
  for (int c0 = 0; c0 < kN_; c0 += kVec) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + c0);
    const E* e = reinterpret_cast<const E*>(&u);
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      if (key0 + c0 + v < lim) {
        const float a = mask_elem<kKind>(e[v]);
        const float x = __uint_as_float(s[c0 + v]);
        s[c0 + v] = __float_as_uint(a == -INFINITY ? -INFINITY : fmaf(16.f, a, x));
      }
    }
  }
}

static_assert(sizeof(Smem) + 1024 + 16 + 2 * kMaskSlotBytes <= 227 * 1024,
              "the masked form's shared memory fits one CTA per SM");

// Threads of a CTA: the general-mask form adds a warp that stages mask rows.
template <bool kMask>
constexpr int cta_threads() { return kMask ? kThreads + 32 : kThreads; }


template <bool kSplit, bool kF16, bool kMask>
__global__ void __launch_bounds__(cta_threads<kMask>(), 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
               const __grid_constant__ CUtensorMap tmO, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.ctl.timeout_ns;
  // Split mode: the merge launched after this kernel (programmatic dependent launch)
  // may be scheduled once every CTA has started; it still waits for this grid to end.
  if constexpr (kSplit) asm volatile("griddepcontrol.launch_dependents;");

  int b, g, r0, rows_here, n_tiles, j0 = 0, bg;
  int key_end;   // keys the tile's last row sees (prefill) / of this split (split mode)
  // split mode only
  int s_idx = 0, t0 = 0, rows = 0, kv_len = 0, k_lo = 0, k_hi = 0, n_hi = 0;
  if constexpr (!kSplit) {
    const int BH = p.B * p.Hkv;
    const int rt = p.n_rtiles - 1 - static_cast<int>(blockIdx.x) / BH;   // longest first
    bg = static_cast<int>(blockIdx.x) % BH;
    b = bg / p.Hkv;
    g = bg % p.Hkv;
    r0 = rt * p.R;
    rows_here = min(p.R, p.Lq - r0);
    // keys the last row of the tile sees
    key_end = (kMask && !p.causal) ? p.Lkv : p.kv_offset + r0 + rows_here;
    n_tiles = (key_end + kN - 1) / kN;
  } else {
    int bid = static_cast<int>(blockIdx.x);
    const int rt = bid % p.n_rtiles;
    bid /= p.n_rtiles;
    s_idx = bid % p.num_splits;
    bid /= p.num_splits;
    g = bid % p.Hkv;
    b = bid / p.Hkv;
    bg = b * p.Hkv + g;
    kv_len = p.kv_lens[b];
    t0 = p.cu_rows ? p.cu_rows[b] : b;
    const int t1 = p.cu_rows ? p.cu_rows[b + 1] : b + 1;
    rows = t1 - t0;
    if (rows < 0 || rows > p.max_rows || t0 < 0 || t1 > p.T || kv_len > p.max_kv_len ||
        kv_len > p.Lcap || kv_len < rows) {
      if (threadIdx.x == 0 && rt == 0 && s_idx == 0 && g == 0)
        record_status(p.ctl.status, GQA_ERR_DEVICE_RANGE);
      return;
    }
    r0 = rt * p.R;                        // first new token of the tile (within the sequence)
    if (r0 >= rows) return;
    rows_here = min(p.R, rows - r0);
    k_lo = s_idx * p.split_keys;
    k_hi = min(k_lo + p.split_keys, kv_len);
    // keys the tile's last row sees (a tree row may see up to the last new key)
    n_hi = min(k_hi, p.tree_mask ? kv_len : kv_len - rows + r0 + rows_here);
    if (n_hi <= k_lo) {
      // No row of the tile sees a key of this split: empty parts.
      for (int m = threadIdx.x; m < rows_here * p.gqa; m += blockDim.x) {
        const size_t n = size_t(t0 + r0 + m / p.gqa) * p.Hq + size_t(g) * p.gqa + m % p.gqa;
        p.lse_parts[size_t(s_idx) * size_t(p.T) * p.Hq + n] = -INFINITY;
      }
      return;
    }
    j0 = k_lo / kN;
    n_tiles = (n_hi + kN - 1) / kN - j0;
    key_end = n_hi;
  }
  // First key that some row of the tile may not see: keys below it are seen by every
  // row; from it on (a causal prompt tile's diagonal, a verify tile's new keys past the
  // first row's, a tree's new keys, every key of a general mask, and every key of the
  // last tile past key_end) a V row can meet probability 0 in the P.V product.  The
  // cleaning pass checks the V rows of these keys.  In fp16 every key is a candidate:
  // an fp16 P rounds to 0 25 or more log2 units below the row maximum, where
  // float64's p (and so p * Inf) is not 0.
  int cand_lo;
  if constexpr (kMask || kF16)
    cand_lo = 0;
  else if constexpr (!kSplit)
    cand_lo = p.kv_offset + r0 + 1;
  else
    cand_lo = min(max(k_lo, p.tree_mask ? kv_len - rows : kv_len - rows + r0 + 1), key_end);

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      ptx::mbar_init(&sm.kv_full[s], 1);
      ptx::mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.s_full[s], 1);
      ptx::mbar_init(&sm.p_full[s], 8);
    }
    ptx::mbar_init(&sm.pv_done, 1);
    ptx::mbar_init(&sm.o_final, 1);
    ptx::mbar_init(&sm.drain, 1);
    ptx::mbar_init(&sm.v_clean, 1);
    ptx::mbar_init(&sm.q_free, 1);
    ptx::mbar_init(&sm.g_full, 1);
    for (int s2 = 0; s2 < 2; ++s2) {
      ptx::mbar_init(&sm.mask_full[s2], 32);   // the mask warp
      ptx::mbar_init(&sm.mask_empty[s2], 8);   // the softmax warps
      ptx::mbar_init(&sm.vs_ready[s2], 1);     // the producer warp (cleaning pass)
    }
    sm.abort = 0;
    sm.zero = 0;
    sm.need_clean = 0;
    sm.n_hits = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  // One pass over the CTA's tiles.  Pass 0 computes the outputs and checks them; the
  // cleaning pass (kClean) runs only when a stored output of pass 0 is NaN / Inf, and
  // recomputes the tile with the V rows of the candidate keys cleaned.  The barriers
  // carry on from pass 0 to the cleaning pass: a per-tile barrier counts the tiles of
  // both passes (global tile index J = J0 + j), a once-per-pass barrier is in phase pp.
  auto run_pass = [&](auto clean_tag) {
    constexpr bool kClean = decltype(clean_tag)::value;
    const int J0 = kClean ? n_tiles : 0;
    const uint32_t pp = kClean ? 1u : 0u;

    if (warp == 0) {
      // ---------------------------------------------------------- producer
      Ring rk = ring_after(J0, kKS, 0);
      Ring rv = ring_after(J0, kVS, kKS);
      bool issued_all = false;
      bool g_issued = false;
      const uint32_t q_bytes = 4u * 128u * uint32_t(p.R * p.gqa);
      if (lane == 0) {
        if constexpr (!kClean) {
          ptx::prefetch_tmap(&tmQ);
          ptx::prefetch_tmap(&tmK);
          ptx::prefetch_tmap(&tmV);
          if constexpr (!kSplit) {
            ptx::prefetch_tmap(&tmG);
            ptx::prefetch_tmap(&tmO);
          }
        }
        ptx::mbar_arrive_expect_tx(&sm.q_full, q_bytes);
        for (int dc = 0; dc < 4; ++dc) {
          if constexpr (!kSplit)
            ptx::tma_load_4d(sm.q + dc * kQChunk, &tmQ, &sm.q_full, dc * 64, r0, g * p.gqa, b);
          else
            ptx::tma_load_3d(sm.q + dc * kQChunk, &tmQ, &sm.q_full, dc * 64, g * p.gqa, t0 + r0);
        }
      }
      // Lane 0: the copy of K_j or V_j into its ring slot, once the slot's previous
      // use is done.
      auto issue_copy = [&](const Ring& r, bool is_v, int j) -> bool {
        const int slot = r.at();
        if (r.count >= r.n &&
            !ptx::mbar_wait(&sm.kv_empty[slot], r.phase ^ 1u, tmo, &sm.abort))
          return false;
        ptx::mbar_arrive_expect_tx(&sm.kv_full[slot], kTileBytes);
        const CUtensorMap* tm = is_v ? &tmV : &tmK;
        for (int dc = 0; dc < 4; ++dc)
          ptx::tma_load_3d(sm.kv[slot] + dc * kChunkBytes, tm, &sm.kv_full[slot], dc * 64,
                           (j0 + j) * kN, bg);
        return true;
      };
      if constexpr (!kClean) {
        if (lane == 0) {
          const int total = 2 * n_tiles;
          for (int it = 0; it < total; ++it) {
            bool is_v;
            int j;
            item_kind(it, n_tiles, is_v, j);
            Ring& r = is_v ? rv : rk;
            if (!issue_copy(r, is_v, j)) {
              fail(sm, p);
              break;
            }
            r.advance();
          }
        }
      } else {
        // The whole warp walks the copies (lane 0 issues them) and cleans each V tile
        // once it has landed, before its P.V product and the softmax's record of it:
        //   - split mode: cache rows at or past kv_len are zeroed (any bits, NaN
        //     included, past the sequence);
        //   - the V rows of candidate keys (from cand_lo on) are checked, a fast check
        //     of the whole run first; a row holding a NaN / Inf element has those
        //     elements set to 0 and its key appended to the hit list (kMaxHits at most;
        //     rows past that are left as they are).
        int n_hits = 0;
        const int total = 2 * n_tiles;
        for (int it = 0; it < total; ++it) {
          bool is_v;
          int j;
          item_kind(it, n_tiles, is_v, j);
          Ring& r = is_v ? rv : rk;
          const int slot = r.at();
          int go = 1;
          if (lane == 0) go = issue_copy(r, is_v, j) ? 1 : 0;
          if (__shfl_sync(0xffffffffu, go, 0) == 0) {
            if (lane == 0) fail(sm, p);
            break;
          }
          const uint32_t phase = r.phase;
          r.advance();
          if (!is_v) continue;
          if (!warp_all(ptx::mbar_wait(&sm.kv_full[slot], phase, tmo, &sm.abort))) {
            if (lane == 0) fail(sm, p);
            break;
          }
          uint8_t* const vt = sm.kv[slot];
          const int tile_key0 = (j0 + j) * kN;
          int pad = kN;   // first row past the sequence (split mode)
          if constexpr (kSplit) pad = min(max(kv_len - tile_key0, 0), kN);
          bool wrote = false;
          if (pad < kN) {
            const int per_blk = (kN - pad) * 8;   // 16-byte chunks per column block
            for (int c = lane; c < 4 * per_blk; c += 32) {
              const int blk = c / per_blk;
              const int rem = c - blk * per_blk;
              *reinterpret_cast<uint4*>(vt + blk * kChunkBytes + (pad + rem / 8) * 128 +
                                        (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            wrote = true;
          }
          const int c_lo = min(max(cand_lo - tile_key0, 0), pad);
          HitRows h{{0u, 0u, 0u, 0u}, n_hits, false};
          if (c_lo < pad) {
            // acc + x * 0 per packed pair stays 0 unless some x is NaN / Inf; 16-byte
            // chunk i of the run: column block i / (nr * 8), row c_lo + (i / 8) % nr
            const int nr = pad - c_lo;
            uint32_t a0 = 0u, a1 = 0u;
            for (int i = lane; i < 4 * nr * 8; i += 32) {
              const int blk4 = i / (nr * 8), rem = i - blk4 * nr * 8;
              const uint4 u = *reinterpret_cast<const uint4*>(vt + blk4 * kChunkBytes +
                                                              (c_lo + (rem >> 3)) * 128 +
                                                              (rem & 7) * 16);
              a0 = nonfinite_acc<kF16>(nonfinite_acc<kF16>(a0, u.x), u.y);
              a1 = nonfinite_acc<kF16>(nonfinite_acc<kF16>(a1, u.z), u.w);
            }
            if (__any_sync(0xffffffffu, (a0 | a1) != 0u)) {
              uint32_t w[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int lo = min(max(c_lo - 32 * q, 0), 32), hi = min(max(pad - 32 * q, 0), 32);
                w[q] = hi > lo ? ((hi - lo == 32 ? 0xffffffffu : ((1u << (hi - lo)) - 1u)) << lo) : 0u;
              }
              h = clean_rows<kF16>(sm, vt, make_uint4(w[0], w[1], w[2], w[3]), tile_key0, n_hits);
            }
          }
          if (__any_sync(0xffffffffu, wrote || h.wrote)) ptx::fence_proxy_async_smem();
          if (lane == 0) {
            for (int q = 0; q < kN / 32; ++q) sm.tile_hits[j & 1][q] = h.w[q];
            sm.tile_base[j & 1] = n_hits;
            sm.n_hits = h.n;
          }
          n_hits = h.n;
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.vs_ready[j & 1]);
        }
      }
      if (lane == 0) {
        issued_all = rv.count == J0 + n_tiles;
        if constexpr (!kSplit) {
          // Prefill: the gate tile (same box as Q) goes into Q's buffer once every S
          // product has read Q; it lands while the last P.V products run.
          if (p.G != nullptr && issued_all) {
            if (ptx::mbar_wait(&sm.q_free, pp, tmo, &sm.abort)) {
              ptx::mbar_arrive_expect_tx(&sm.g_full, q_bytes);
              for (int dc = 0; dc < 4; ++dc)
                ptx::tma_load_4d(sm.q + dc * kQChunk, &tmG, &sm.g_full, dc * 64, r0, g * p.gqa, b);
              g_issued = true;
            } else {
              fail(sm, p);
            }
          }
        }
      }
      if constexpr (kSplit && !kClean) {
        // Split mode: a tile holding cache rows at or past kv_len can only be the CTA's
        // last one, and its V copy is the last copy this warp issued.  That copy is use
        // u of its slot and use u-1 has landed (its slot was released before the copy
        // was issued), so the parity wait below is unambiguous.  Zero the padded rows,
        // make the writes visible to the tensor core, then release the last PV.
        const int jl = n_tiles - 1;
        const int tile_key0 = (j0 + jl) * kN;
        if (tile_key0 + kN > kv_len) {
          const int vslot = kKS + jl % kVS;
          const bool go = __shfl_sync(0xffffffffu, issued_all ? 1 : 0, 0) != 0;
          const bool landed =
              go && warp_all(ptx::mbar_wait(&sm.kv_full[vslot], uint32_t(jl / kVS) & 1u, tmo,
                                            &sm.abort));
          if (landed) {
            const int r_first = max(0, kv_len - tile_key0);
            const int per_blk = (kN - r_first) * 8;   // 16-byte chunks per column block
            uint4* base = reinterpret_cast<uint4*>(sm.kv[vslot]);
            for (int c = lane; c < 4 * per_blk; c += 32) {
              const int blk = c / per_blk;
              const int rem = c - blk * per_blk;
              base[(blk * kChunkBytes + (r_first + rem / 8) * 128) / 16 + rem % 8] =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            ptx::fence_proxy_async_smem();
          } else if (lane == 0) {
            fail(sm, p);
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&sm.v_clean);
        }
      }
      if (lane == 0) {
        // Let every copy this warp started land before the CTA can exit.
        for (Ring* r : {&rk, &rv})
          for (int c = max(J0, r->count - r->n); c < r->count; ++c)
            ptx::mbar_wait(&sm.kv_full[r->base + c % r->n], uint32_t(c / r->n) & 1u, tmo, &sm.zero);
        ptx::mbar_wait(&sm.q_full, pp, tmo, &sm.zero);
        if (g_issued) ptx::mbar_wait(&sm.g_full, pp, tmo, &sm.zero);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        bool ok = ptx::mbar_wait(&sm.q_full, pp, tmo, &sm.abort);
        ptx::tc_fence_after();
        const uint32_t qa = ptx::smem_addr(sm.q);
        Ring rk = ring_after(J0, kKS, 0);
        Ring rv = ring_after(J0, kVS, kKS);
        auto issue_s = [&](int j) -> bool {
          const int slot = rk.at();
          if (!ptx::mbar_wait(&sm.kv_full[slot], rk.phase, tmo, &sm.abort)) return false;
          ptx::tc_fence_after();
          const uint32_t ka = ptx::smem_addr(sm.kv[slot]);
          const uint32_t d = tmem + kTmS + uint32_t(kN) * uint32_t((J0 + j) & 1);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint32_t qo = uint32_t(kk >> 2) * kQChunk + uint32_t(kk & 3) * 32u;
            const uint32_t ko = uint32_t(kk >> 2) * kChunkBytes + uint32_t(kk & 3) * 32u;
            ptx::mma_ss(d, ptx::sdesc_sw128(qa + qo, 16, 1024), ptx::sdesc_sw128(ka + ko, 16, 1024),
                        idesc_s<kF16>(), kk > 0);
          }
          ptx::tc_commit(&sm.s_full[(J0 + j) & 1]);
          ptx::tc_commit(&sm.kv_empty[slot]);
          rk.advance();
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int J = J0 + j;
          if (!ptx::mbar_wait(&sm.p_full[J & 1], (J >> 1) & 1, tmo, &sm.abort)) return false;
          const int slot = rv.at();
          if (!ptx::mbar_wait(&sm.kv_full[slot], rv.phase, tmo, &sm.abort)) return false;
          if constexpr (kClean) {
            if (!ptx::mbar_wait(&sm.vs_ready[j & 1], (j >> 1) & 1, tmo, &sm.abort)) return false;
          } else if constexpr (kSplit) {
            if (j == n_tiles - 1 && (j0 + j) * kN + kN > kv_len &&
                !ptx::mbar_wait(&sm.v_clean, 0, tmo, &sm.abort))
              return false;
          }
          ptx::tc_fence_after();
          const uint32_t va = ptx::smem_addr(sm.kv[slot]);
          const uint32_t pa = tmem + kTmS + uint32_t(kN) * uint32_t(J & 1);
          constexpr int kStepsHalf = kHalf / 16;   // k16 steps per softmax half
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            // P of keys 16kk..16kk+15: half kk / kStepsHalf, 8 columns per k16 step
            const uint32_t acol = uint32_t(kk / kStepsHalf) * kHalf + uint32_t(kk % kStepsHalf) * 8u;
            ptx::mma_ts(tmem + kTmO, pa + acol,
                        ptx::sdesc_sw128(va + uint32_t(kk) * 2048u, kChunkBytes, 1024),
                        idesc_pv<kF16>(), (j > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::tc_commit(&sm.pv_done);
          ptx::tc_commit(&sm.kv_empty[slot]);
          rv.advance();
          return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 1; ok && j < n_tiles; ++j) {
          ok = issue_s(j);
          if (ok) ok = issue_pv(j - 1);
        }
        if constexpr (!kSplit) {
          if (ok) ptx::tc_commit(&sm.q_free);   // every S product issued: Q may be overwritten
        }
        if (ok) ok = issue_pv(n_tiles - 1);
        if (ok) {
          ptx::tc_commit(&sm.o_final);
        } else {
          fail(sm, p);
        }
        // Every MMA issued so far must finish before tensor memory is released (or
        // written again by the cleaning pass).
        ptx::tc_commit(&sm.drain);
        ptx::mbar_wait(&sm.drain, pp, tmo, &sm.zero);
      }
      __syncwarp();
    } else if (warp >= kThreads / 32) {
      // ---------------------------------------------------------- mask rows (kMask)
      // With one mask head, the R query rows of the tile share their mask rows across
      // the GQA heads: this warp copies tile j's rows into slot J % 2 (16-byte
      // cp.async, zero past the mask's last key) while the softmax warps use slot
      // (J - 1) % 2, and waits for the slot's release before reusing it.
      if constexpr (kMask) {
        if (p.mask_stage) {
          const int es = p.mask_kind == 1 ? 1 : p.mask_kind == 2 ? 4 : 2;
          const int pitch = kN * es + 16;
          const int cpr = kN * es / 16;   // 16-byte chunks per row
          const int kpc = 16 / es;        // keys per chunk
          const char* mbase = static_cast<const char*>(p.mask);
          uint8_t* const slots = reinterpret_cast<uint8_t*>(&sm) + ((sizeof(Smem) + 15) & ~size_t(15));
          for (int j = 0; j < n_tiles; ++j) {
            const int J = J0 + j;
            const int slot = J & 1;
            if (J >= 2 &&
                !warp_all(ptx::mbar_wait(&sm.mask_empty[slot], uint32_t((J - 2) >> 1) & 1u, tmo,
                                         &sm.abort))) {
              if (lane == 0) fail(sm, p);
              break;
            }
            const int key0 = (j0 + j) * kN;
            uint8_t* const dst = slots + slot * kMaskSlotBytes;
            for (int c = lane; c < rows_here * cpr; c += 32) {
              const int r = c / cpr, ch = c - r * cpr;
              const int kf = key0 + ch * kpc;
              const int nb = min(max((p.Lkv - kf) * es, 0), 16);
              const char* src =
                  nb > 0 ? mbase + ((long long)b * p.ms_b + (long long)(r0 + r) * p.ms_i + kf) * es
                         : mbase;
              ptx::cp_async16(ptx::smem_addr(dst + r * pitch + ch * 16), src, uint32_t(nb));
            }
            ptx::cp_async_mbar_arrive(&sm.mask_full[slot]);
          }
          ptx::cp_async_wait_all();   // no copy may land after the CTA exits
        }
      }
    } else {
      // ---------------------------------------------------------- softmax / epilogue
      const int sw = warp - 2;
      const int half = sw >> 2;
      const int lq = warp & 3;
      const int row = lq * 32 + lane;
      const uint32_t bar_id = 1 + lq;
      int hh, rr, lim;
      bool valid;
      if constexpr (!kSplit) {
        hh = row / p.R;                     // row m: head m / R, prompt row r0 + m % R
        rr = row - hh * p.R;
        valid = (row < p.R * p.gqa) && (r0 + rr < p.Lq);
        lim = valid ? p.kv_offset + r0 + rr + 1 : p.kv_offset + r0 + 1;
        if (kMask && !p.causal) lim = p.Lkv;
      } else {
        rr = row / p.gqa;                   // row m: token r0 + m / GQA, head m % GQA
        hh = row - rr * p.gqa;
        valid = (row < p.R * p.gqa) && (rr < rows_here);
        lim = valid ? min(p.tree_mask ? kv_len : kv_len - rows + r0 + rr + 1, k_hi) : n_hi;
      }
      // Tree verify: new key kv_len - rows + k is visible only when bit k is set.
      const unsigned long long tmask =
          (kSplit && p.tree_mask != nullptr && valid) ? p.tree_mask[t0 + r0 + rr] : ~0ull;
      const int tbase = kSplit && p.tree_mask != nullptr ? kv_len - rows : INT_MAX;
      const int q = r0 + rr;
      const uint32_t trow = tmem + (uint32_t(lq * 32) << 16);
      // General mask: offset (elements) of this row's mask entries.
      long long mrow = 0;
      if constexpr (kMask) {
        const int mh = p.mask_hmode == 0 ? 0 : p.mask_hmode == 1 ? g * p.gqa + hh
                                                                   : hh % p.mask_chunk;
        mrow = (long long)b * p.ms_b + (long long)mh * p.ms_h + (long long)q * p.ms_i;
      }

      float m_run = -INFINITY;
      float l_part = 0.f;
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const int J = J0 + j;
        const int buf = J & 1;
        bool mine = warp_all(ptx::mbar_wait(&sm.s_full[buf], (J >> 1) & 1, tmo, &sm.abort)) &&
                    !sm.abort;
        if constexpr (kMask) {
          if (p.mask_stage)
            mine = warp_all(ptx::mbar_wait(&sm.mask_full[buf], (J >> 1) & 1, tmo, &sm.abort)) &&
                   mine;
        }
        uint32_t s[kHalf];
        float mx = -INFINITY;
        if (mine) {
          ptx::tc_fence_after();
          const uint32_t sa = trow + kTmS + uint32_t(kN) * buf + uint32_t(kHalf) * half;
          if constexpr (kHalf == 64) {
            ptx::tmem_ld64_wait(sa, *reinterpret_cast<uint32_t(*)[64]>(&s[0]));
          } else {
            ptx::tmem_ld32_wait(sa, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
          }
          const int key0 = (j0 + j) * kN + half * kHalf;
          if (key0 + kHalf > lim) {
#pragma unroll
            for (int c = 0; c < kHalf; ++c)
              if (key0 + c >= lim) s[c] = __float_as_uint(-INFINITY);
          }
          if (key0 + kHalf > tbase) {
#pragma unroll
            for (int c = 0; c < kHalf; ++c) {
              const int k = key0 + c - tbase;
              if (k >= 0 && k < 64 && !((tmask >> k) & 1ull)) s[c] = __float_as_uint(-INFINITY);
            }
          }
          if constexpr (kMask) {
            if (p.mask_stage) {
              if (valid && key0 < lim) {
                const int es = p.mask_kind == 1 ? 1 : p.mask_kind == 2 ? 4 : 2;
                const uint8_t* srow = reinterpret_cast<const uint8_t*>(&sm) +
                                      ((sizeof(Smem) + 15) & ~size_t(15)) + buf * kMaskSlotBytes +
                                      rr * (kN * es + 16) + half * kHalf * es;
                switch (p.mask_kind) {
                  case 1:
                    apply_mask_row_smem<1>(s, srow, key0, lim);
                    break;
                  case 2:
                    apply_mask_row_smem<2>(s, reinterpret_cast<const float*>(srow), key0, lim);
                    break;
                  case 3:
                    apply_mask_row_smem<3>(s, reinterpret_cast<const uint16_t*>(srow), key0, lim);
                    break;
                  case 4:
                    apply_mask_row_smem<4>(s, reinterpret_cast<const uint16_t*>(srow), key0, lim);
                    break;
                  default:
                    break;
                }
              }
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(&sm.mask_empty[buf]);   // slot read by this warp
            } else if (valid && key0 < lim) {
              switch (p.mask_kind) {
                case 1:
                  apply_mask_row<1>(s, static_cast<const uint8_t*>(p.mask) + mrow, p.ms_j, key0, lim);
                  break;
                case 2:
                  apply_mask_row<2>(s, static_cast<const float*>(p.mask) + mrow, p.ms_j, key0, lim);
                  break;
                case 3:
                  apply_mask_row<3>(s, static_cast<const uint16_t*>(p.mask) + mrow, p.ms_j, key0, lim);
                  break;
                case 4:
                  apply_mask_row<4>(s, static_cast<const uint16_t*>(p.mask) + mrow, p.ms_j, key0, lim);
                  break;
                default:
                  break;
              }
            }
          }
          float m8[8];
#pragma unroll
          for (int c = 0; c < 8; ++c) m8[c] = __uint_as_float(s[c]);
#pragma unroll
          for (int c = 8; c < kHalf; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(s[c]));
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                     fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          mx *= kScaleLog2;
        }
        sm.red[buf][half][row] = mx;
        sm.ok[buf][half][row] = mine ? 1 : 0;
        ptx::named_bar_sync(bar_id, 64);
        ok = mine && sm.ok[buf][half ^ 1][row];
        if (!ok) break;
        const float tmax = fmaxf(mx, sm.red[buf][half ^ 1][row]);
        bool store_ok = true;
        bool late = false;        // fp16: O is rescaled by alpha_late after P_j is stored
        float alpha_late = 1.f;
        if (j == 0) {
          m_run = tmax;
        } else if (__any_sync(0xffffffffu, tmax > m_run + rescale_threshold<kF16>())) {
          // The branch is warp-uniform (tcgen05.ld/st are warp-collective; the partner
          // warp holds the same rows, so it takes it too), but only rows whose own max
          // rose past the threshold move it; the others multiply by exactly 1, so every
          // row's result depends on its own scores alone.
          const bool need = tmax > m_run + rescale_threshold<kF16>();
          const float alpha = need ? ex2(m_run - tmax) : 1.f;
          if (need) m_run = tmax;
          l_part *= alpha;
          if constexpr (kF16) {
            late = true;          // warp-uniform, as the branch is
            alpha_late = alpha;   // O is rescaled once P_j is stored (below)
          } else {
            // O must hold PV_{j-1} before it is rescaled.
            store_ok = warp_all(ptx::mbar_wait(&sm.pv_done, (J - 1) & 1, tmo, &sm.abort));
            if (store_ok) {
              ptx::tc_fence_after();
#pragma unroll 1
              for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                const uint32_t ta = trow + kTmO + 128u * half + 32u * cc;
                ptx::tmem_ld32_wait(ta, o);
#pragma unroll
                for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                ptx::tmem_st32_wait(ta, o);
              }
            }
          }
        }
        if (!store_ok) {
          fail(sm, p);
          continue;  // the next exchange stops both threads of the pair
        }
        const float msub = (m_run == -INFINITY) ? 0.f : m_run;
        float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[kHalf / 2];
        const float2 sc2 = make_float2(kScaleLog2, kScaleLog2);
        const float2 ms2 = make_float2(-msub, -msub);
        // fp16 cleaning pass: bit c of zk = key c's score is -inf, i.e. its probability
        // is exactly 0 (an fp16 P that rounds to 0 is not: see record_zero_scores)
        uint32_t zk[2] = {0u, 0u};
#pragma unroll
        for (int c = 0; c < kHalf / 2; ++c) {
          if constexpr (kClean && kF16) {
            zk[c >> 4] |= ((__uint_as_float(s[2 * c]) == -INFINITY ? 1u : 0u) |
                           (__uint_as_float(s[2 * c + 1]) == -INFINITY ? 2u : 0u))
                          << (2 * (c & 15));
          }
          const float2 x = fma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])),
                                sc2, ms2);
          const float p0 = ex2(x.x);
          const float p1 = ex2(x.y);
          ls2[c & 1] = add2(ls2[c & 1], make_float2(p0, p1));
          pk[c] = pack_elem2<kF16>(p0, p1);
        }
        l_part += (ls2[0].x + ls2[1].x) + (ls2[0].y + ls2[1].y);
        const uint32_t pdst = trow + kTmS + uint32_t(kN) * buf + uint32_t(kHalf) * half;
        if constexpr (kHalf == 64) {
          ptx::tmem_st32_wait(pdst, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        } else {
          ptx::tmem_st16_wait(pdst, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        }
        if constexpr (kF16) {
          // fp16's lower threshold makes rescales common where a row's maximum jumps
          // (key outliers): P_j was computed and stored while PV_{j-1} ran, and O is
          // rescaled now, before PV_j (out of line, so that the loop's registers are
          // not shaped by it).  The branch is warp-uniform, as above.
          if (late) {
            if (!warp_all(ptx::mbar_wait(&sm.pv_done, (J - 1) & 1, tmo, &sm.abort))) {
              fail(sm, p);
              continue;  // the next exchange stops both threads of the pair
            }
            ptx::tc_fence_after();
            rescale_o_cols(trow + kTmO + 128u * half, alpha_late);
          }
        }
        if constexpr (kClean) {
          // Once V_j is cleaned: for its hit keys among this thread's keys, record
          // whether the probability is 0 (bf16: read back from P; fp16: a -inf score).
          if (warp_all(ptx::mbar_wait(&sm.vs_ready[j & 1], (j >> 1) & 1, tmo, &sm.abort))) {
            const volatile uint32_t* th = sm.tile_hits[j & 1];
            const uint32_t w0 = th[2 * half], w1 = th[2 * half + 1];   // this half's keys
            if ((w0 | w1) != 0u) {
              const int idx = sm.tile_base[j & 1] + (half ? __popc(th[0]) + __popc(th[1]) : 0);
              if constexpr (kF16)
                record_zero_scores(sm, zk[0], zk[1], w0, w1, idx, row);
              else
                record_zero_probs(sm, pdst, w0, w1, idx, row);
            }
          } else if (lane == 0) {
            fail(sm, p);   // the next exchange stops both threads of the pair
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.p_full[buf]);
      }
      if (!ok) fail(sm, p);

      // -------------------------------------------------------------- epilogue
      bool fin = ok && warp_all(ptx::mbar_wait(&sm.o_final, pp, tmo, &sm.abort));
      const int pb = (J0 + n_tiles) & 1;   // parity slot not used by the last tile's exchange
      sm.red[pb][half][row] = l_part;
      sm.ok[pb][half][row] = fin ? 1 : 0;
      ptx::named_bar_sync(bar_id, 64);
      fin = fin && sm.ok[pb][half ^ 1][row];
      // Prefill: the gate tile arrives by TMA in Q's buffer (same swizzled layout as Q),
      // and the output tile is staged in the K/V ring (free once O is final) for one
      // TMA store: row m's 16-byte chunk c of column block dc sits at dc * kQChunk +
      // m * 128 + (c ^ (m & 7)) * 16 in both.
      if constexpr (!kSplit) {
        if (p.G != nullptr) fin = warp_all(ptx::mbar_wait(&sm.g_full, pp, tmo, &sm.abort)) && fin;
      }
      const float l_tot = l_part + sm.red[pb][half ^ 1][row];
      // l_tot is 0 exactly when the row saw no key, NaN when it saw a NaN score.
      const float inv_l = l_tot == 0.f ? 0.f : 1.f / l_tot;
      if constexpr (kClean) {
        // Hits: the P.V product took 0 for their NaN / Inf V elements.  A row that sees
        // the key adds p * V of each such element to its O (a NaN or an infinity, so the
        // scale of p does not matter; p = 0 gives NaN, as exact arithmetic would); a row
        // that does not see it adds nothing.
        const int n_hits = *reinterpret_cast<volatile int*>(&sm.n_hits);
        if (n_hits > 0 && __any_sync(0xffffffffu, fin))
          add_hit_terms<kF16, kMask>(sm, trow + kTmO + 128u * half, row, n_hits, fin && valid,
                                     p.V + (long long)bg * p.v_rows * kHeadDim + half * 128, lim,
                                     tbase, tmask, p.mask, p.mask_kind, mrow, p.ms_j);
      }
      if constexpr (!kSplit) {
        // Column blocks 0 and 2 are complete after the first two 32-column chunks of
        // both row halves, blocks 1 and 3 after the last two: each pair is stored while
        // the rest is computed (rows past Lq fall outside the tensor and are not
        // written).  Every softmax thread takes both barriers, failed or not.
        if (!fin) fail(sm, p);
        if (fin) ptx::tc_fence_after();
        uint8_t* const stage = &sm.kv[0][0];
        const size_t row_off =
            (size_t(b) * p.Hq + size_t(g * p.gqa + hh)) * size_t(p.Lq) + size_t(q);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (fin) {
            uint32_t o[32];
            ptx::tmem_ld32_wait(trow + kTmO + 128u * half + 32u * cc, o);
            const int dc = half * 2 + (cc >> 1);   // columns half*128 + cc*32 .. +31
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int c = (cc & 1) * 4 + v;
              const uint32_t off =
                  uint32_t(dc) * kQChunk + uint32_t(row) * 128u + (uint32_t(c ^ (row & 7)) << 4);
              uint32_t w[4] = {0u, 0u, 0u, 0u};
              if (p.G != nullptr) {
                const uint4 u = *reinterpret_cast<const uint4*>(sm.q + off);
                w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
              }
              uint32_t r[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float2 res = mul2(make_float2(__uint_as_float(o[v * 8 + 2 * e]),
                                              __uint_as_float(o[v * 8 + 2 * e + 1])),
                                  make_float2(inv_l, inv_l));
                if (p.G != nullptr) {
                  const float2 f = unpack_elem2<kF16>(w[e]);
                  res = mul2(res, gate_sigmoid2(f.x, f.y));
                }
                r[e] = pack_elem2<kF16>(res.x, res.y);
              }
              *reinterpret_cast<uint4*>(stage + off) = make_uint4(r[0], r[1], r[2], r[3]);
            }
          }
          if (cc & 1) {
            if (fin) ptx::fence_proxy_async_smem();   // the staged blocks are read by TMA
            ptx::named_bar_sync(5, 256);
            if (threadIdx.x == 64 && *reinterpret_cast<volatile int*>(&sm.abort) == 0) {
              const int d0 = cc >> 1, d1 = 2 + (cc >> 1);
              ptx::tma_store_4d(&tmO, stage + d0 * kQChunk, d0 * 64, r0, g * p.gqa, b);
              ptx::tma_store_4d(&tmO, stage + d1 * kQChunk, d1 * 64, r0, g * p.gqa, b);
              ptx::bulk_commit_group();
            }
          }
        }
        if constexpr (!kClean) {
          // Check of the row's stored values (read back while the stores drain): a NaN /
          // Inf output calls for the cleaning pass.
          if (fin && valid) {
            const uint8_t* const src = stage + (half * 2) * kQChunk + row * 128;
            uint32_t a0 = 0u, a1 = 0u;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const uint4 u = *reinterpret_cast<const uint4*>(
                  src + (k >> 3) * kQChunk + (((k & 7) ^ (row & 7)) << 4));
              a0 = nonfinite_acc<kF16>(nonfinite_acc<kF16>(a0, u.x), u.y);
              a1 = nonfinite_acc<kF16>(nonfinite_acc<kF16>(a1, u.z), u.w);
            }
            if ((a0 | a1) != 0u) sm.need_clean = 1;
          }
        }
        if (fin && valid && half == 0 && p.lse != nullptr)
          p.lse[row_off] = l_tot == 0.f ? -INFINITY : (m_run + __log2f(l_tot)) * kLn2;
        // Shared memory stays allocated until the stores have read it.
        if (threadIdx.x == 64) ptx::bulk_wait_group_read0();
      } else if (fin) {
        ptx::tc_fence_after();
        // Normalised partial O / l (fp32) and lse for the merge; -inf: no key seen.
        const size_t n = size_t(t0 + q) * p.Hq + size_t(g) * p.gqa + hh;
        const size_t part = size_t(s_idx) * size_t(p.T) * p.Hq + n;
        const bool live = valid && l_tot != 0.f;
        float d0 = 0.f, d1 = 0.f;   // pass 0: check of the written values (see above)
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          ptx::tmem_ld32_wait(trow + kTmO + 128u * half + 32u * cc, o);
          if (live) {
            float4* op =
                reinterpret_cast<float4*>(p.O_parts + part * kHeadDim + half * 128 + cc * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              const float4 f = make_float4(
                  __uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                  __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
              op[v] = f;
              if constexpr (!kClean) {
                d0 = nonfinite_acc_f32(nonfinite_acc_f32(d0, f.x), f.y);
                d1 = nonfinite_acc_f32(nonfinite_acc_f32(d1, f.z), f.w);
              }
            }
          }
        }
        if (valid && half == 0)
          p.lse_parts[part] = live ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
        if constexpr (!kClean) {
          if ((__float_as_uint(d0) | __float_as_uint(d1)) != 0u) sm.need_clean = 1;
        }
      } else {
        fail(sm, p);
      }
    }
  };

  run_pass(std::false_type{});
  ptx::tc_fence_before();
  __syncthreads();
  if (*reinterpret_cast<volatile int*>(&sm.need_clean) != 0 &&
      *reinterpret_cast<volatile int*>(&sm.abort) == 0) {
    // Cleaning pass: the stores of pass 0 must be complete before the same rows are
    // stored again, and the zero-probability record starts empty.
    if (threadIdx.x == 64) ptx::bulk_wait_group0();
    for (int i = threadIdx.x; i < kM * (kMaxHits / 32); i += blockDim.x) (&sm.pz[0][0])[i] = 0u;
    __syncthreads();
    ptx::tc_fence_after();
    run_pass(std::true_type{});
    ptx::tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
template <bool kSplit, bool kF16, bool kMask = false>
cudaError_t launch_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tg, const CUtensorMap& to, const Params& p,
                      long long grid, cudaStream_t stream) {
  // the Smem block (1024-aligned), then for kMask the two mask slots
  const size_t smem = sizeof(Smem) + 1024 + (kMask ? 16 + 2 * size_t(kMaskSlotBytes) : 0);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<kSplit, kF16, kMask>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  attn_tc_kernel<kSplit, kF16, kMask><<<dim3(unsigned(grid)), dim3(cta_threads<kMask>()), smem,
                                        stream>>>(tq, tk, tv, tg, to, p);
  e = cudaGetLastError();
  if (e == cudaSuccess)
    note_launch(kSplit  ? (kF16 ? "attn_tc_kernel<split,fp16>" : "attn_tc_kernel<split,bf16>")
                : kMask ? (kF16 ? "attn_tc_kernel<masked,fp16>" : "attn_tc_kernel<masked,bf16>")
                        : (kF16 ? "attn_tc_kernel<prefill,fp16>" : "attn_tc_kernel<prefill,bf16>"),
                grid, cta_threads<kMask>(), smem);
  return e;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const LaunchCtl& ctl, cudaStream_t stream,
                           bool* encode_failed) {
  // Long prompts run on CTA pairs, which copy and read half of every K/V tile per SM:
  // on GB300 that matches this kernel at 4K-8K keys and is faster when the rows see
  // many more keys than the row tiles hold (L2 traffic halves), while a short prompt
  // pays the pair's cluster set-up.
  if (!a.masked && a.kv_offset + a.Lq >= kPairMinKeys)
    return launch_prefill_pair(a, ctl, stream, encode_failed);
  *encode_failed = false;
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) {
    *encode_failed = true;
    return cudaErrorNotSupported;
  }
  const int gqa = a.Hq / a.Hkv;
  const int R = prefill_rows_per_tile(gqa);
  CUtensorMap tq, tk, tv, tg, to;
  {
    // Q, G and out [B, Hq, Lq, 256]: a box is R rows x the group's GQA heads x 64 dims.
    const cuuint64_t dims[4] = {256, cuuint64_t(a.Lq), cuuint64_t(a.Hq), cuuint64_t(a.B)};
    const cuuint64_t str[3] = {512, cuuint64_t(a.Lq) * 512, cuuint64_t(a.Hq) * a.Lq * 512};
    const cuuint32_t box[4] = {64, cuuint32_t(R), cuuint32_t(gqa), 1};
    if (!encode_16b(fn, &tq, a.Q, 4, dims, str, box, a.f16)) *encode_failed = true;
    if (!encode_16b(fn, &tg, a.G != nullptr ? a.G : a.Q, 4, dims, str, box, a.f16))
      *encode_failed = true;
    if (!encode_16b(fn, &to, a.out, 4, dims, str, box, a.f16)) *encode_failed = true;
  }
  {
    // Only keys a row of the call can see are addressable; TMA zero-fills the rest.
    const int kv_hi = a.causal ? a.kv_offset + a.Lq : a.Lkv;
    const cuuint64_t dims[3] = {256, cuuint64_t(kv_hi), cuuint64_t(a.B) * a.Hkv};
    const cuuint64_t str[2] = {512, cuuint64_t(a.Lkv) * 512};
    const cuuint32_t box[3] = {64, cuuint32_t(kN), 1};   // one column block of a tile
    if (!encode_16b(fn, &tk, a.K, 3, dims, str, box, a.f16)) *encode_failed = true;
    if (!encode_16b(fn, &tv, a.V, 3, dims, str, box, a.f16)) *encode_failed = true;
  }
  if (*encode_failed) return cudaErrorInvalidValue;

  Params p{};
  p.G = static_cast<const uint16_t*>(a.G);
  p.V = static_cast<const uint16_t*>(a.V);
  p.v_rows = a.Lkv;
  p.out = static_cast<uint16_t*>(a.out);
  p.lse = a.lse;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Lq = a.Lq;
  p.kv_offset = a.kv_offset;
  p.gqa = gqa;
  p.R = R;
  p.n_rtiles = (a.Lq + R - 1) / R;
  p.ctl = ctl;
  p.Lkv = a.Lkv;
  p.causal = a.causal ? 1 : 0;
  p.mask = a.mask;
  p.mask_kind = a.mask_kind;
  p.mask_hmode = a.mask_hmode;
  p.mask_chunk = a.mask_chunk;
  p.ms_b = a.mask_strides[0];
  p.ms_h = a.mask_strides[1];
  p.ms_i = a.mask_strides[2];
  p.ms_j = a.mask_strides[3];
  {
    // Stage the mask rows in shared memory when one mask head serves every query
    // head, keys are contiguous and every staged row starts on a 16-byte boundary.
    const int es = a.mask_kind == 1 ? 1 : a.mask_kind == 2 ? 4 : 2;
    const bool aligned16 = reinterpret_cast<uintptr_t>(a.mask) % 16 == 0 &&
                           (a.mask_strides[0] * es) % 16 == 0 && (a.mask_strides[2] * es) % 16 == 0;
    p.mask_stage = (a.masked && a.mask_kind >= 1 && a.mask_kind <= 4 && a.mask_hmode == 0 &&
                    a.mask_strides[3] == 1 && aligned16 && R * (kN * es + 16) <= kMaskSlotBytes)
                       ? 1 : 0;
  }

  const long long grid = (long long)p.n_rtiles * a.B * a.Hkv;
  if (a.masked)
    return a.f16 ? launch_tc<false, true, true>(tq, tk, tv, tg, to, p, grid, stream)
                 : launch_tc<false, false, true>(tq, tk, tv, tg, to, p, grid, stream);
  return a.f16 ? launch_tc<false, true>(tq, tk, tv, tg, to, p, grid, stream)
               : launch_tc<false, false>(tq, tk, tv, tg, to, p, grid, stream);
}

int tc_split_keys_multiple() { return kN; }

cudaError_t launch_decode_split_tc(const DecodeSplitArgs& a, const LaunchCtl& ctl,
                                   cudaStream_t stream, bool* encode_failed) {
  *encode_failed = false;
  EncodeTiledFn fn = get_encode_fn();
  if (fn == nullptr) {
    *encode_failed = true;
    return cudaErrorNotSupported;
  }
  const int gqa = a.Hq / a.Hkv;
  const int R = prefill_rows_per_tile(gqa);
  CUtensorMap tq, tk, tv;
  {
    // Q [T, Hq, 256]: a box is R tokens x the group's GQA heads x 64 dims.
    const cuuint64_t dims[3] = {256, cuuint64_t(a.Hq), cuuint64_t(a.T)};
    const cuuint64_t str[2] = {512, cuuint64_t(a.Hq) * 512};
    const cuuint32_t box[3] = {64, cuuint32_t(gqa), cuuint32_t(R)};
    if (!encode_16b(fn, &tq, a.Q, 3, dims, str, box, a.f16)) *encode_failed = true;
  }
  {
    const cuuint64_t dims[3] = {256, cuuint64_t(a.Lcap), cuuint64_t(a.B) * a.Hkv};
    const cuuint64_t str[2] = {512, cuuint64_t(a.Lcap) * 512};
    const cuuint32_t box[3] = {64, cuuint32_t(kN), 1};
    if (!encode_16b(fn, &tk, a.K, 3, dims, str, box, a.f16)) *encode_failed = true;
    if (!encode_16b(fn, &tv, a.V, 3, dims, str, box, a.f16)) *encode_failed = true;
  }
  if (*encode_failed) return cudaErrorInvalidValue;

  Params p{};
  p.V = static_cast<const uint16_t*>(a.V);
  p.v_rows = a.Lcap;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.gqa = gqa;
  p.R = R;
  p.n_rtiles = (a.max_rows + R - 1) / R;
  p.kv_lens = a.kv_lens;
  p.cu_rows = a.cu_rows;
  p.tree_mask = a.tree_mask;
  p.O_parts = a.O_parts;
  p.lse_parts = a.lse_parts;
  p.T = a.T;
  p.Lcap = a.Lcap;
  p.max_rows = a.max_rows;
  p.max_kv_len = a.max_kv_len;
  p.split_keys = a.split_keys;
  p.num_splits = a.num_splits;
  p.ctl = ctl;

  const long long grid = (long long)a.B * a.Hkv * a.num_splits * p.n_rtiles;
  // The gate and output maps are not used in split mode.
  return a.f16 ? launch_tc<true, true>(tq, tk, tv, tq, tq, p, grid, stream)
               : launch_tc<true, false>(tq, tk, tv, tq, tq, p, grid, stream);
}

}  // namespace gqa
