// Pieces shared by the tcgen05 attention kernels (the one-CTA kernel of
// prefill_tc.cu and the CTA-pair prefill of prefill_pair.cu): tile geometry,
// small device helpers, the out-of-line helpers of the cleaning pass, and the host's
// tensor-map encoder.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx_sm100.cuh"

namespace gqa {
namespace {

constexpr int kM = 128;                       // packed rows per CTA tile
constexpr int kN = 128;                       // keys per K/V tile
constexpr int kQChunk = 128 * 128;            // Q: 128 rows x 64 bf16 per column block
constexpr int kQBytes = 4 * kQChunk;
constexpr int kChunkBytes = kN * 128;         // K/V: kN rows x 64 bf16 per column block
constexpr int kTileBytes = 4 * kChunkBytes;   // kN keys x 256 bf16
constexpr int kHalf = kN / 2;                 // keys per softmax thread per tile
static_assert(kN == 128, "softmax threads take 64-key halves of a 128-key tile");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmO = 0;
constexpr uint32_t kTmS = 256;                // S buffer b at kTmS + kN*b
// Lazy-rescale threshold in log2 units: P <= 2^threshold must fit the element type
// (bf16: 2^32; fp16: 2^15 = 32768, below its 65504 maximum).  l and O are fp32.
template <bool kF16>
__device__ __forceinline__ float rescale_threshold() { return kF16 ? 15.0f : 32.0f; }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// O *= alpha over this thread's 128 columns of O from tensor-memory address ta0 (the
// fp16 kernels' lazy rescale, taken after P_j is stored).  Kept out of line so that
// the softmax loop's registers are not shaped by it.  Warp-collective (called from a
// warp-uniform branch).
__device__ __noinline__ void rescale_o_cols(uint32_t ta0, float alpha) {
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t o[32];
    const uint32_t ta = ta0 + 32u * cc;
    ptx::tmem_ld32_wait(ta, o);
#pragma unroll
    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
    ptx::tmem_st32_wait(ta, o);
  }
}

// Position in a ring of tile slots [base, base + n): slot, phase bit, tiles so far.
struct Ring {
  int slot;
  uint32_t phase;
  int count;
  int n;
  int base;
  __device__ __forceinline__ int at() const { return base + slot; }
  __device__ __forceinline__ void advance() {
    ++count;
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Item `it` of the load / consume sequence K_0, K_1, V_0, K_2, V_1, ..., V_{n-1}.
__device__ __forceinline__ void item_kind(int it, int n, bool& is_v, int& j) {
  if (it == 0) {
    is_v = false; j = 0;
  } else if (it == 2 * n - 1) {
    is_v = true; j = n - 1;
  } else {
    const int m = (it - 1) >> 1;
    is_v = ((it - 1) & 1) != 0;
    j = is_v ? m : m + 1;
  }
}

// Bias of one mask element in natural-log units: a bool mask gives 0 (attend) or
// -inf (excluded); an additive mask gives its value.
__device__ __forceinline__ float mask_bias(uint8_t v) { return v ? 0.f : -INFINITY; }
__device__ __forceinline__ float mask_bias(float v) { return v; }
__device__ __forceinline__ float mask_bias(uint16_t v, std::integral_constant<int, 3>) {
  return __uint_as_float(uint32_t(v) << 16);                       // bf16
}
__device__ __forceinline__ float mask_bias(uint16_t v, std::integral_constant<int, 4>) {
  return __half2float(__ushort_as_half(v));                         // fp16
}

template <int kKind, typename E>
__device__ __forceinline__ float mask_elem(E v) {
  if constexpr (kKind == 3 || kKind == 4)
    return mask_bias(v, std::integral_constant<int, kKind>{});
  else
    return mask_bias(v);
}


// ---------------------------------------------------------------- non-finite V values
// Out-of-line helpers of the cleaning pass (a NaN / Inf V element at a key that some
// rows of a tile see and others do not; see the kernel).

// Bits c of the result: key rows c of a landed V tile found holding a NaN / Inf
// element (which is set to +0 in shared memory), among the rows selected by `rows`;
// their keys (tile_key0 + c) are appended to the hit list from index `n`, up to
// kMaxHits (rows past that are left as they are).  One warp.
struct HitRows {
  uint32_t w[kN / 32];
  int n;          // hit-list length afterwards
  bool wrote;     // this lane wrote shared memory
};
template <bool kF16, typename Sm>
__device__ __noinline__ HitRows clean_rows(Sm& sm, uint8_t* vt, uint4 rows, int tile_key0,
                                           int n) {
  constexpr int kCap = int(sizeof(Sm::hit_key) / sizeof(int));
  const int lane = threadIdx.x & 31;
  const int blk = lane >> 3, ch = lane & 7;   // this lane's 16-byte chunk of a key row
  HitRows h{{0u, 0u, 0u, 0u}, n, false};
  const uint32_t rw[4] = {rows.x, rows.y, rows.z, rows.w};
  for (int w = 0; w < kN / 32; ++w) {
    uint32_t bits = rw[w];
    while (bits != 0u) {
      const int c = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1u;
      uint4* const a =
          reinterpret_cast<uint4*>(vt + blk * kChunkBytes + c * 128 + ((ch ^ (c & 7)) << 4));
      uint4 u = *a;
      const bool nf = clear_nonfinite<kF16>(u);
      if (__ballot_sync(0xffffffffu, nf) != 0u && h.n < kCap) {
        if (nf) {
          *a = u;
          h.wrote = true;
        }
        h.w[w] |= 1u << (c & 31);
        if (lane == 0) sm.hit_key[h.n] = tile_key0 + c;
        ++h.n;
      }
    }
  }
  return h;
}

// Records, for the hit keys among this thread's 64 keys of a cleaned tile (bits of
// w0, w1; hit-list indices from idx), whether the key's probability is 0, so that the
// epilogue's p * V term is then a NaN and otherwise the value's own infinity.  bf16:
// read back from P in tensor memory (a bf16 P is 0 exactly when the fp32 probability
// is: the score is -inf, or more than 126 log2 units below the row maximum, where ex2
// flushes to 0).  Whole warp.
template <typename Sm>
__device__ __noinline__ void record_zero_probs(Sm& sm, uint32_t p_taddr, uint32_t w0,
                                               uint32_t w1, int idx, int row) {
  uint32_t pw[32];
  ptx::tc_fence_after();
  ptx::tmem_ld32_wait(p_taddr, pw);
#pragma unroll 1
  for (int c = 0; c < kHalf; ++c) {
    if (((c < 32 ? w0 >> c : w1 >> (c - 32)) & 1u) != 0u) {
      if (((pw[c >> 1] >> ((c & 1) * 16)) & 0xFFFFu) == 0u)
        atomicOr(&sm.pz[row][idx >> 5], 1u << (idx & 31));
      ++idx;
    }
  }
}

// The same record for fp16, from the scores: an fp16 P rounds to 0 already 25 log2
// units below the row maximum, where float64's p (and so p * Inf) is not 0, so a
// probability counts as 0 only when the key's score is -inf (bits of z0, z1).
template <typename Sm>
__device__ __noinline__ void record_zero_scores(Sm& sm, uint32_t z0, uint32_t z1, uint32_t w0,
                                                uint32_t w1, int idx, int row) {
#pragma unroll 1
  for (int c = 0; c < kHalf; ++c) {
    if (((c < 32 ? w0 >> c : w1 >> (c - 32)) & 1u) != 0u) {
      if (((c < 32 ? z0 >> c : z1 >> (c - 32)) & 1u) != 0u)
        atomicOr(&sm.pz[row][idx >> 5], 1u << (idx & 31));
      ++idx;
    }
  }
}

// Epilogue of a CTA with hits: adds p * V of the original NaN / Inf elements of every
// hit key this row sees to its O row in tensor memory (o_taddr: the thread's 128
// columns).  The sum is then a NaN or an infinity, so the scale of p does not matter;
// a probability of 0 gives NaN, as float64 arithmetic would.  Whole warp; `act` says
// whether this lane's row takes part.  vrow0: V row 0 of the KV head, at the thread's
// first column.
template <bool kF16, bool kMask, typename Sm>
__device__ __noinline__ void add_hit_terms(const Sm& sm, uint32_t o_taddr, int row, int n_hits,
                                           bool act, const uint16_t* vrow0, int lim, int tbase,
                                           unsigned long long tmask, const void* mask,
                                           int mask_kind, long long mrow, long long ms_j) {
  ptx::tc_fence_after();
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t o[32];
    ptx::tmem_ld32_wait(o_taddr + 32u * cc, o);
    for (int i = 0; act && i < n_hits; ++i) {
      const int key = sm.hit_key[i];
      if (key >= lim) continue;
      if (key >= tbase && key - tbase < 64 && !((tmask >> (key - tbase)) & 1ull)) continue;
      if constexpr (kMask) {
        const long long at = mrow + (long long)key * ms_j;
        float a = 0.f;
        switch (mask_kind) {
          case 1: a = mask_elem<1>(static_cast<const uint8_t*>(mask)[at]); break;
          case 2: a = mask_elem<2>(static_cast<const float*>(mask)[at]); break;
          case 3: a = mask_elem<3>(static_cast<const uint16_t*>(mask)[at]); break;
          case 4: a = mask_elem<4>(static_cast<const uint16_t*>(mask)[at]); break;
          default: break;
        }
        if (a == -INFINITY) continue;
      }
      const float keep = ((sm.pz[row][i >> 5] >> (i & 31)) & 1u) ? 0.f : 1.f;
      const uint4* const v = reinterpret_cast<const uint4*>(vrow0 + (long long)key * kHeadDim + cc * 32);
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 u = __ldg(v + q4);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll 1
        for (int e = 0; e < 8; ++e) {
          const uint32_t x = (w[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu;
          if (elem_nonfinite<kF16>(x))
            o[q4 * 8 + e] =
                __float_as_uint(__uint_as_float(o[q4 * 8 + e]) + keep * elem_to_float<kF16>(x));
        }
      }
    }
    ptx::tmem_st32_wait(o_taddr + 32u * cc, o);
  }
}


// Ring position after `count` uses of a ring of n slots that starts at slot `base`.
__device__ __forceinline__ Ring ring_after(int count, int n, int base) {
  return Ring{count % n, uint32_t(count / n) & 1u, count, n, base};
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool encode_16b(EncodeTiledFn fn, CUtensorMap* map, const void* base, int rank,
                const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                bool f16) {
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cuuint32_t(rank), const_cast<void*>(base),
                  dims, strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace gqa
