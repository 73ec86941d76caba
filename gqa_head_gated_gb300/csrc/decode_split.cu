// Decode / chain-verify split kernel: for one (sequence b, KV group g, key split s,
// row block), the attention of the group's query heads x new rows over the split's
// keys, written as a normalised partial result (O/l, m + ln l) for the LSE merge.
//
// The method (TensorFold PR #1009, "Receipt", attention contract paragraph)
// runs decode over fixed-size cache chunks and merges their partial results; here
// a split is `split_keys` keys and the merge is attn_lse_merge.  All query heads
// of a KV group are packed with the rows into the MMA M dimension (packed row
// p = row * GQA + head), so every K/V byte is read once per split for the whole
// group (DS4Server issue113 README, opening rule).
//
// Memory-bound: K/V tiles of 32 keys (32 KB for K+V) stream through a 3-stage
// cp.async ring (two CTAs per SM for up to 32 packed rows) with 16-byte vector
// copies, coalesced along the 512-byte rows;
// rows at or past the split's end are zero-filled by the copy itself, so cache
// padding is never read.  Scores and P.V run on bf16 or fp16 mma.sync (m16n8k16,
// fp32 accumulate); the online softmax is fp32 with quad-shuffle row reductions
// and rescales at every tile, so P <= 1 in either element type.
//
// Work split: either one (b, g, split, row block) unit per CTA (fixed splits of
// `split_keys`), or balanced shares (the one-call decode): all units' key tiles laid
// end to end and cut into one equal contiguous share per resident CTA, a share that
// crosses units yielding one part per piece.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <type_traits>

#include "internal.h"

namespace gqa {
namespace {

constexpr int kTK = 32;          // keys per tile
constexpr int kStages = 3;
constexpr int kThreads = 128;
constexpr int kRowBytes = 512;   // 256 16-bit elements
constexpr int kTileBytes = kTK * kRowBytes;   // one of K or V

struct Params {
  const uint16_t* Q;   // bf16 or fp16 bits
  const uint16_t* K;
  const uint16_t* V;
  const int* kv_lens;
  const int* cu_rows;
  const unsigned long long* tree_mask;   // null: chain verify
  float* O_parts;
  float* lse_parts;
  int B, T, Hq, Hkv, Lcap, max_rows, max_kv_len, gqa, split_keys, num_splits, n_rb;
  // Balanced mode (balanced != 0): num_splits is the part capacity per row and
  // lmax_tiles = ceil(max_kv_len / kTK); see decode_split_kernel.
  int balanced, lmax_tiles;
  LaunchCtl ctl;
};

constexpr int kMaxBalancedSeqs = kBalancedMaxSeqs;   // sequences a balanced launch schedules

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy; src_bytes = 0 zero-fills without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk `c` (0..31) of row `r` in a 512-byte-row tile:
// chunks are XOR-swizzled by the row's low 3 bits so ldmatrix is conflict-free.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return uint32_t(r) * kRowBytes + uint32_t((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool kF16>
__device__ __forceinline__ void mma_16b(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- non-finite V values
// Keys that some rows of a block see and others do not ([pr_lo, pr_hi), fewer than 64)
// meet probability 0 in the P.V product for the rows that do not see them.  Their V
// rows' NaN / Inf elements are set to 0 in shared memory before the product and added
// back, as p * V, for the rows that see them when the part is written (keys a row does
// not see are excluded from its sums, never weighted by 0).  These helpers stay out of
// line so that the kernel's steady-state code is as it is without them.

// All threads: clears the NaN / Inf elements of V rows r_lo .. r_lo+nr-1 of a tile and
// sets bit (tile key0 + r - pr_lo) of *hit for each row that held one.
template <bool kF16>
__device__ __noinline__ void clean_tile_rows(uint8_t* vt, int r_lo, int nr, int bit0,
                                             unsigned long long* hit) {
  for (int c = threadIdx.x; c < nr * 32; c += blockDim.x) {
    const int r = r_lo + (c >> 5);
    uint4* const a = reinterpret_cast<uint4*>(vt + uint32_t(r) * 512u +
                                              uint32_t(((c & 31) ^ (r & 7)) << 4));
    uint4 u = *a;
    if (clear_nonfinite<kF16>(u)) {
      *a = u;
      atomicOr(hit, 1ull << (bit0 + r));
    }
  }
}

// Records bit off of *pz for each hit key this thread holds a zero probability for:
// z bit (2 * nt + e) = probability 0 for key key_w + 8 nt + 2 t4 + e.
__device__ __noinline__ void record_zero_probs(unsigned long long* pz, unsigned long long hits,
                                               int first_off, int t4, uint32_t z, int nt_count) {
  for (int nt = 0; nt < nt_count; ++nt)
    for (int e = 0; e < 2; ++e) {
      const int off = first_off + nt * 8 + 2 * t4 + e;
      if (((z >> (2 * nt + e)) & 1u) && off >= 0 && off < 64 && ((hits >> off) & 1ull))
        atomicOr(pz, 1ull << off);
    }
}

// p * V of the NaN / Inf elements taken out of P.V, for the hit keys a row sees, added
// to its normalised part (4 columns at Vg_c; a NaN or an infinity, so the scale of p
// does not matter; p = 0 gives NaN as float64 would).
template <bool kF16>
__device__ __noinline__ float4 add_hit_terms(float4 acc, unsigned long long hits,
                                             unsigned long long pz, int pr_lo, int lim,
                                             bool tree, int base, unsigned long long msk,
                                             const uint16_t* Vg_c) {
  while (hits != 0ull) {
    const int off = __ffsll(static_cast<long long>(hits)) - 1;
    hits &= hits - 1ull;
    const int key = pr_lo + off;
    if (key >= lim || (tree && key >= base && !((msk >> (key - base)) & 1ull))) continue;
    const float keep = ((pz >> off) & 1ull) ? 0.f : 1.f;
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(Vg_c + size_t(key) * 256));
    const uint32_t x[4] = {u.x & 0xFFFFu, u.x >> 16, u.y & 0xFFFFu, u.y >> 16};
    float* const a = &acc.x;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (elem_nonfinite<kF16>(x[e])) a[e] += keep * elem_to_float<kF16>(x[e]);
  }
  return acc;
}

// WR row groups of 16 packed rows; WK key groups per row group (WR * WK warps).
template <int WR, int WK, bool kF16>
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(const Params p) {
  constexpr int MB = 16 * WR;          // packed rows per CTA
  constexpr int NK = kTK / WK;         // keys per warp per tile
  constexpr int NT = NK / 8;           // score n-tiles per warp
  static_assert(WR * WK <= kThreads / 32, "too many warps");
  static_assert(NK % 16 == 0, "a warp needs whole k16 steps of P.V");

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;                                    // MB x 512 B
  uint8_t* sKV = smem + MB * kRowBytes;                  // kStages x (K tile, V tile)
  __shared__ float s_m[WK][MB];
  __shared__ float s_l[WK][MB];
  __shared__ int s_lim[MB];
  __shared__ unsigned long long s_mask[MB];
  // Keys some rows of the block see and others do not, [pr_lo, pr_hi) (fewer than 64):
  // bit k of s_hit = key pr_lo + k had a NaN / Inf V element (set to 0 in shared
  // memory before P.V); bit k of s_pz[row] = the row's probability for that key was 0.
  __shared__ unsigned long long s_hit;
  __shared__ unsigned long long s_pz[MB];

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // The merge launched after this kernel (programmatic dependent launch) may be
  // scheduled once every CTA has started; it still waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;");

  // One unit: the packed rows [rb*MB, rb*MB + MB) of (sequence b, KV group g) against
  // keys [k_lo, min(k_cap, kv_len)), written as part s.  CTA-uniform; returns early
  // (uniformly) when there is nothing to do.
  auto run_unit = [&](const int b, const int g, const int rb, const int s, const int k_lo,
                      const int k_cap) {
  const int kv_len = p.kv_lens[b];
  const int t0 = p.cu_rows ? p.cu_rows[b] : b;
  const int t1 = p.cu_rows ? p.cu_rows[b + 1] : b + 1;
  const int rows = t1 - t0;
  if (rows < 0 || rows > p.max_rows || t1 > p.T || t0 < 0 || kv_len > p.max_kv_len ||
      kv_len > p.Lcap || kv_len < rows) {
    if (tid == 0 && rb == 0 && s == 0 && g == 0) record_status(p.ctl.status, GQA_ERR_DEVICE_RANGE);
    return;
  }
  const int P = rows * p.gqa;                 // packed rows of this (b, g)
  const int p0 = rb * MB;
  if (p0 >= P) return;                        // row block past this sequence's rows
  if (s >= p.num_splits) {                    // cannot happen with a valid plan
    if (tid == 0) record_status(p.ctl.status, GQA_ERR_DEVICE_RANGE);
    return;
  }
  const int k_hi = min(k_cap, kv_len);

  // Visible keys of each packed row of the block (0 for padding rows).
  // Chain: row i sees keys < kv_len - rows + i + 1.  Tree: keys before the new rows,
  // and new key base + k when bit k of the row's mask is set.
  const bool tree = p.tree_mask != nullptr;
  const int base = kv_len - rows;
  if (tid < MB) {
    const int pp = p0 + tid;
    int lim = 0;
    unsigned long long m = 0;
    if (pp < P) {
      lim = tree ? kv_len : base + pp / p.gqa + 1;
      if (tree) m = p.tree_mask[t0 + pp / p.gqa];
    }
    s_lim[tid] = min(lim, k_hi);
    s_mask[tid] = m;
    s_pz[tid] = 0ull;
  }
  if (tid == 0) s_hit = 0ull;
  int n_hi = 0;   // keys any row of the block sees in this split
  {
    const int pl = min(P - 1, p0 + MB - 1);
    n_hi = min(tree ? kv_len : base + pl / p.gqa + 1, k_hi);
  }
  // Chain: the block's first row sees keys < base + p0/gqa + 1, so later new keys are
  // seen by some rows only; tree: any new key may be.
  const int pr_lo = max(k_lo, tree ? base : base + p0 / p.gqa + 1);
  const int pr_hi = n_hi;
  const int n_tiles = n_hi > k_lo ? (n_hi - k_lo + kTK - 1) / kTK : 0;
  const int scan_from = pr_hi > pr_lo ? (pr_lo - k_lo) / kTK : n_tiles;   // first tile to clean

  const size_t kv_base = (size_t(b) * p.Hkv + g) * size_t(p.Lcap) * 256;
  const uint16_t* Kg = p.K + kv_base;
  const uint16_t* Vg = p.V + kv_base;

  // Q block: packed row pp -> token t0 + pp / gqa, head g*gqa + pp % gqa.
  {
    const uint32_t q0 = saddr(sQ);
    for (int c = tid; c < MB * 32; c += kThreads) {
      const int r = c >> 5, ch = c & 31;
      const int pp = p0 + r;
      const bool ok = pp < P;
      const uint16_t* src =
          ok ? p.Q + ((size_t(t0 + pp / p.gqa) * p.Hq) + g * p.gqa + pp % p.gqa) * 256 + ch * 8
             : p.Q;
      cp_async16(q0 + swz(r, ch), src, ok ? 16u : 0u);
    }
    cp_async_commit();
  }
  auto load_tile = [&](int tile, int stage) {
    const int key0 = k_lo + tile * kTK;
    const uint32_t kd = saddr(sKV + stage * 2 * kTileBytes);
    const uint32_t vd = kd + kTileBytes;
#pragma unroll
    for (int i = 0; i < (kTK * 32) / kThreads; ++i) {
      const int c = tid + i * kThreads;
      const int r = c >> 5, ch = c & 31;
      const int key = key0 + r;
      const bool ok = key < n_hi;
      const size_t off = ok ? size_t(key) * 256 + ch * 8 : 0;
      cp_async16(kd + swz(r, ch), Kg + off, ok ? 16u : 0u);
      cp_async16(vd + swz(r, ch), Vg + off, ok ? 16u : 0u);
    }
  };
#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < n_tiles) load_tile(st, st);
    cp_async_commit();
  }

  const int wr = warp / WK;
  const int wk = warp % WK;
  const bool compute = warp < WR * WK;
  const int g4 = lane >> 2;       // row within the 8-row half of the fragment
  const int t4 = lane & 3;

  float o[32][4];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r[2] = {-INFINITY, -INFINITY};
  float l_r[2] = {0.f, 0.f};

  // One tile of keys; the tiles from scan_from on (keys some rows of the block do not
  // see) also get their V rows cleaned, in a second instance of the step so that the
  // steady-state loop carries none of that.
  auto step = [&](const int tile, auto with_hits) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nt = tile + kStages - 1;
      if (nt < n_tiles) load_tile(nt, nt % kStages);
      cp_async_commit();
    }
    const int stage = tile % kStages;
    // Keys of this tile that some rows do not see: their V rows' NaN / Inf elements are
    // set to 0 here, so a row that does not see the key multiplies 0 (not Inf or NaN)
    // by its probability 0; the rows that see it get p * V of the original element
    // added when the part is written (keys a row does not see are excluded from its
    // sums, never weighted by 0).
    bool hit_tile = false;
    if constexpr (decltype(with_hits)::value) {
      const int tkey0 = k_lo + tile * kTK;
      const int r_lo = max(pr_lo - tkey0, 0);
      clean_tile_rows<kF16>(sKV + stage * 2 * kTileBytes + kTileBytes, r_lo,
                            min(pr_hi - tkey0, kTK) - r_lo, tkey0 - pr_lo, &s_hit);
      __syncthreads();
      hit_tile = s_hit != 0ull;
    }
    if (!compute) return;
    const uint32_t kb = saddr(sKV + stage * 2 * kTileBytes);
    const uint32_t vb = kb + kTileBytes;
    const uint32_t qb = saddr(sQ);

    // S = Q K^T over this warp's NK keys.  With two n-tiles the 16-step k chain is
    // split over even and odd steps into independent accumulators (shorter latency).
    constexpr int KC = NT == 2 ? 2 : 1;
    float sc[NT][4];
    float sc2[KC][NT][4];
#pragma unroll
    for (int c = 0; c < KC; ++c)
#pragma unroll
      for (int i = 0; i < NT; ++i) sc2[c][i][0] = sc2[c][i][1] = sc2[c][i][2] = sc2[c][i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      {
        const int r = wr * 16 + (lane & 15);
        const int ch = 2 * kk + (lane >> 4);
        ldsm_x4(qb + swz(r, ch), a0, a1, a2, a3);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        const int r = wk * NK + np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = 2 * kk + ((lane >> 3) & 1);
        ldsm_x4(kb + swz(r, ch), b0, b1, b2, b3);
        mma_16b<kF16>(sc2[kk % KC][2 * np], a0, a1, a2, a3, b0, b1);
        mma_16b<kF16>(sc2[kk % KC][2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sc2[0][i][e];
#pragma unroll
        for (int c = 1; c < KC; ++c) v += sc2[c][i][e];
        sc[i][e] = v;
      }
    // Mask, online softmax (two rows per thread: g4 and g4 + 8).
    const int key_w = k_lo + tile * kTK + wk * NK;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int lim = s_lim[wr * 16 + g4 + 8 * hr];
      const unsigned long long msk = s_mask[wr * 16 + g4 + 8 * hr];
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key_w + nt * 8 + 2 * t4 + e;
          float v = sc[nt][2 * hr + e];
          const bool vis = key < lim && (!tree || key < base || ((msk >> (key - base)) & 1ull));
          v = vis ? v * kScaleLog2 : -INFINITY;
          sc[nt][2 * hr + e] = v;
          mx = fmaxf(mx, v);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_r[hr], mx);
      const float msub = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2(m_r[hr] - msub);   // 0 when nothing was seen before
      m_r[hr] = m_new;
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float pv = ex2(sc[nt][2 * hr + e] - msub);
          sc[nt][2 * hr + e] = pv;
          ls += pv;
        }
      }
      if (decltype(with_hits)::value && hit_tile) {
        // record the hit keys this row's probability is 0 for
        uint32_t z = 0u;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) z |= uint32_t(sc[nt][2 * hr + e] == 0.f) << (2 * nt + e);
        record_zero_probs(&s_pz[wr * 16 + g4 + 8 * hr], s_hit, key_w - pr_lo, t4, z, NT);
      }
      l_r[hr] = l_r[hr] * alpha + ls;
#pragma unroll
      for (int dn = 0; dn < 32; ++dn) {
        o[dn][2 * hr] *= alpha;
        o[dn][2 * hr + 1] *= alpha;
      }
    }
    // O += P V over this warp's keys.
#pragma unroll
    for (int ks = 0; ks < NK / 16; ++ks) {
      const uint32_t pa0 = pack_elem2<kF16>(sc[2 * ks][0], sc[2 * ks][1]);
      const uint32_t pa1 = pack_elem2<kF16>(sc[2 * ks][2], sc[2 * ks][3]);
      const uint32_t pa2 = pack_elem2<kF16>(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
      const uint32_t pa3 = pack_elem2<kF16>(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
      const int r = wk * NK + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int dp = 0; dp < 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        const int ch = 2 * dp + (lane >> 4);
        ldsm_x4_t(vb + swz(r, ch), b0, b1, b2, b3);
        mma_16b<kF16>(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
        mma_16b<kF16>(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
    }
  };
  for (int tile = 0; tile < min(scan_from, n_tiles); ++tile) step(tile, std::false_type{});
  for (int tile = scan_from; tile < n_tiles; ++tile) step(tile, std::true_type{});
  cp_async_wait<0>();
  __syncthreads();

  // Combine the key groups of each row block in shared memory, then write the
  // normalised part.  Reuses the K/V ring: WK x MB x 256 fp32 <= 64 KB.
  float* sO = reinterpret_cast<float*>(sKV);
  if (compute) {
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float l = l_r[hr];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const int r = wr * 16 + g4 + 8 * hr;
      if (t4 == 0) {
        s_m[wk][r] = m_r[hr];
        s_l[wk][r] = l;
      }
      float* dst = sO + (size_t(wk) * MB + r) * 256;
#pragma unroll
      for (int dn = 0; dn < 32; ++dn)
        *reinterpret_cast<float2*>(dst + dn * 8 + 2 * t4) = make_float2(o[dn][2 * hr], o[dn][2 * hr + 1]);
    }
  }
  __syncthreads();
  const int rows_blk = min(MB, P - p0);
  for (int idx = tid; idx < rows_blk * 64; idx += kThreads) {
    const int r = idx >> 6;
    const int c4 = (idx & 63) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < WK; ++k) M = fmaxf(M, s_m[k][r]);
    const int pp = p0 + r;
    const size_t n = size_t(t0 + pp / p.gqa) * p.Hq + g * p.gqa + pp % p.gqa;
    const size_t part = size_t(s) * size_t(p.T) * p.Hq + n;
    // fmaxf drops NaN scores, so a row that saw only NaN keeps M = -inf; it is
    // told apart from a row that saw no key by its sum (NaN, not 0).
    const float Msub = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < WK; ++k) {
      const float w = ex2(s_m[k][r] - Msub);
      L += w * s_l[k][r];
      const float4 v = *reinterpret_cast<const float4*>(sO + (size_t(k) * MB + r) * 256 + c4);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    if (L == 0.f) {   // no key of this split is visible to the row
      if (c4 == 0) p.lse_parts[part] = -INFINITY;
      continue;
    }
    const float inv = 1.f / L;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    if (s_hit != 0ull)
      acc = add_hit_terms<kF16>(acc, s_hit, s_pz[r], pr_lo, s_lim[r], tree, base, s_mask[r],
                                Vg + c4);
    *reinterpret_cast<float4*>(p.O_parts + part * 256 + c4) = acc;
    if (c4 == 0) p.lse_parts[part] = (Msub + __log2f(L)) * kLn2;
  }
  };   // run_unit

  if (!p.balanced) {
    // One unit per CTA: (b, g, split s, row block rb) from the block index.
    int bid = blockIdx.x;
    const int rb = bid % p.n_rb;
    bid /= p.n_rb;
    const int s = bid % p.num_splits;
    bid /= p.num_splits;
    const int g = bid % p.Hkv;
    const int b = bid / p.Hkv;
    run_unit(b, g, rb, s, s * p.split_keys, s * p.split_keys + p.split_keys);
    return;
  }

  // Balanced mode: the key ranges of all (sequence, KV group, row block) segments,
  // in tiles of kTK keys, are laid end to end (sequence-major) and cut into equal
  // contiguous shares, one per CTA, so every CTA streams the same number of tiles
  // whatever the sequence lengths.  A share that crosses segments yields one part per
  // piece; a piece's part index is its CTA's position among the CTAs sharing the
  // segment, and the CTA that ends a segment marks the unused part slots empty.
  __shared__ int s_base[kMaxBalancedSeqs + 1];
  for (int b = tid; b < p.B; b += kThreads) {
    const int kv = p.kv_lens[b];
    const int t0 = p.cu_rows ? p.cu_rows[b] : b;
    const int rows = (p.cu_rows ? p.cu_rows[b + 1] : b + 1) - t0;
    const bool ok = rows >= 0 && rows <= p.max_rows && kv >= rows && kv <= p.max_kv_len &&
                    kv <= p.Lcap && t0 >= 0 && t0 + rows <= p.T;
    const int nrb = (rows * p.gqa + MB - 1) / MB;
    s_base[b + 1] = ok ? p.Hkv * nrb * ((kv + kTK - 1) / kTK) : 0;
    if (!ok && rows != 0) record_status(p.ctl.status, GQA_ERR_DEVICE_RANGE);
  }
  __syncthreads();
  if (tid == 0) {
    s_base[0] = 0;
    for (int b = 0; b < p.B; ++b) s_base[b + 1] += s_base[b];
  }
  __syncthreads();
  const long long W = s_base[p.B];
  // Shares of at least lmax_tiles / (num_splits - 2) tiles keep every segment within
  // num_splits parts; every share holds at least one tile.
  long long n_cta = (W * (p.num_splits - 2)) / max(1, p.lmax_tiles);
  n_cta = min(min(n_cta, W), (long long)gridDim.x);
  n_cta = max(n_cta, 1LL);
  const long long i = blockIdx.x;
  if (i >= n_cta || W == 0) return;
  long long pos = W * i / n_cta;
  const long long r1 = W * (i + 1) / n_cta;
  while (pos < r1) {
    int b = 0;
    {
      int lo = 0, hi = p.B - 1;        // last b with s_base[b] <= pos
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_base[mid] <= pos) lo = mid; else hi = mid - 1;
      }
      b = lo;
    }
    const int kv = p.kv_lens[b];
    const int t0 = p.cu_rows ? p.cu_rows[b] : b;
    const int rows = (p.cu_rows ? p.cu_rows[b + 1] : b + 1) - t0;
    const int nrb = (rows * p.gqa + MB - 1) / MB;
    const long long seg_len = (kv + kTK - 1) / kTK;
    const long long off = pos - s_base[b];
    const long long seg = off / seg_len;
    const int g = int(seg / nrb);
    const int rb = int(seg % nrb);
    const long long seg_start = s_base[b] + seg * seg_len;
    const long long seg_end = seg_start + seg_len;
    const long long piece_end = min(r1, seg_end);
    const long long i0 = ((seg_start + 1) * n_cta + W - 1) / W - 1;   // CTA holding its first tile
    const int s = int(i - i0);
    run_unit(b, g, rb, s, int(pos - seg_start) * kTK, int(piece_end - seg_start) * kTK);
    if (piece_end == seg_end) {
      // Part slots s+1 .. num_splits-1 of this segment's rows are empty.
      const int P = rows * p.gqa;
      const int p0 = rb * MB;
      const int nr = min(MB, P - p0);
      const int nfill = p.num_splits - 1 - s;
      for (int idx = tid; idx < nfill * nr; idx += kThreads) {
        const int sp = s + 1 + idx / nr;
        const int pp = p0 + idx % nr;
        const size_t n = size_t(t0 + pp / p.gqa) * p.Hq + g * p.gqa + pp % p.gqa;
        p.lse_parts[size_t(sp) * size_t(p.T) * p.Hq + n] = -INFINITY;
      }
    }
    __syncthreads();                   // shared buffers are reused by the next piece
    pos = piece_end;
  }
}

template <int WR, int WK, bool kF16>
cudaError_t launch_t(const Params& p, cudaStream_t stream, long long grid) {
  constexpr int MB = 16 * WR;
  const size_t smem = size_t(MB) * kRowBytes + size_t(kStages) * 2 * kTileBytes;
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<WR, WK, kF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  if (p.balanced) {
    // One CTA per resident slot: the shares are cut on the device.
    int per_sm = 0, dev = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel<WR, WK, kF16>,
                                                      kThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    grid = (long long)(per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
  }
  decode_split_kernel<WR, WK, kF16><<<dim3(unsigned(grid)), dim3(kThreads), smem, stream>>>(p);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    char name[64];
    std::snprintf(name, sizeof(name), "decode_split_kernel<%d,%d,%s>%s", WR, WK,
                  kF16 ? "fp16" : "bf16", p.balanced ? " balanced" : "");
    note_launch(name, grid, kThreads, smem);
  }
  return e;
}

}  // namespace

int decode_rows_per_cta(int packed_rows) {
  if (packed_rows <= 16) return 16;
  if (packed_rows <= 32) return 32;
  return 64;
}

cudaError_t launch_decode_split(const DecodeSplitArgs& a, const LaunchCtl& ctl,
                                cudaStream_t stream) {
  Params p;
  p.Q = static_cast<const uint16_t*>(a.Q);
  p.K = static_cast<const uint16_t*>(a.K);
  p.V = static_cast<const uint16_t*>(a.V);
  p.kv_lens = a.kv_lens;
  p.cu_rows = a.cu_rows;
  p.tree_mask = a.tree_mask;
  p.O_parts = a.O_parts;
  p.lse_parts = a.lse_parts;
  p.B = a.B;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.Lcap = a.Lcap;
  p.max_rows = a.max_rows;
  p.max_kv_len = a.max_kv_len;
  p.gqa = a.Hq / a.Hkv;
  p.split_keys = a.split_keys;
  p.num_splits = a.num_splits;
  p.ctl = ctl;
  p.balanced = a.balanced ? 1 : 0;
  p.lmax_tiles = (a.max_kv_len + kTK - 1) / kTK;
  const int MB = decode_rows_per_cta(a.max_rows * p.gqa);
  p.n_rb = (a.max_rows * p.gqa + MB - 1) / MB;
  const long long grid = (long long)a.B * a.Hkv * a.num_splits * p.n_rb;
  if (a.f16) {
    if (MB == 16) return launch_t<1, 2, true>(p, stream, grid);
    if (MB == 32) return launch_t<2, 2, true>(p, stream, grid);
    return launch_t<4, 1, true>(p, stream, grid);
  }
  if (MB == 16) return launch_t<1, 2, false>(p, stream, grid);
  if (MB == 32) return launch_t<2, 2, false>(p, stream, grid);
  return launch_t<4, 1, false>(p, stream, grid);
}

}  // namespace gqa
