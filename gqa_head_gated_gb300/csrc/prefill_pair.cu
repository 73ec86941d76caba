// Gated causal GQA attention on prompt rows, computed by CTA pairs (tcgen05
// .cta_group::2) on sm_103a.
//
// The operation and the row layout are those of the one-CTA kernel (prefill_tc.cu):
// a CTA owns a tile of 128 packed rows, R = floor(128/GQA) consecutive query rows of
// every query head of one KV group (row m: head m / R, query row r0 + m % R), so that
// each K/V tile serves the whole group (DS4Server issue113 README, opening rule: the
// heads of a KV group share its K/V).  Here two CTAs of a cluster take two
// consecutive row tiles of the same KV group (CTA r of the pair owns tile 2t + r) and
// share every 128-key K/V tile: CTA r loads keys 64r .. 64r+63 of each K tile and
// dims 128r .. 128r+127 of each V tile, and the even CTA issues the products of both:
//   S = Q K^T      M = 256 (each CTA's 128 Q rows), N = 128 (64 keys from each CTA)
//   O += P V       M = 256 (each CTA's P in its own TMEM), N = 256 (128 dims from each)
// Each SM thus reads and copies half of every K/V tile where the one-CTA kernel's
// S products take both whole operands from shared memory; S, P and O of a CTA's
// rows live in its own tensor memory, and its softmax warps and epilogue work on
// them exactly as in the one-CTA kernel.  The pair covers the keys its later tile
// sees; the earlier tile's rows mask the extra keys by selection.
//
// Roles per CTA (320 threads): warp 0 TMA producer (its own Q, halves of K and V,
// then its gate tile), warp 1 TMEM allocation (both CTAs, together) and, in the even
// CTA, the MMA issuer, warps 2..9 softmax and epilogue.  Both CTAs' copies complete
// on the even CTA's full barriers, which count the pair's bytes; the even CTA's
// commits arrive on the barriers of both; the softmax warps of both arrive on the
// even CTA's P barrier.  Shared-memory layouts are identical in the two CTAs, as the
// pair products read both at the same offsets.
//
// Non-finite V values at keys some rows of the pair do not see: as in the one-CTA
// kernel, pass 0 checks its stored outputs and, when a CTA of the pair finds a NaN /
// Inf there, the pair runs its tiles again in a cleaning pass.  There each CTA loads
// whole V tiles (its own MMA half first), cleans the rows of the candidate keys
// (from the first key some row of the pair does not see) and keeps the hit list for
// its rows; the products wait until both CTAs have cleaned the tile.
#include <climits>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "internal.h"
#include "ptx_sm100.cuh"
#include "tc_common.cuh"

namespace gqa {
namespace {

constexpr int kThreadsP = 320;
constexpr int kHalfTileBytes = kTileBytes / 2;   // half of a K or V tile: 32 KB
constexpr int kKRingP = 2;                       // K ring: slots of 64 keys x 256 dims
constexpr int kVRingP = 2;                       // V ring: slots of 128 keys x 128 dims
constexpr int kKHalfChunk = 64 * 128;            // K half: 64 keys x 64 dims per column block
// Cleaning pass: a pair's candidate keys (the diagonal of its 2R rows and the rest of
// its last key tile) are fewer than 384 in bf16; in fp16 every key is a candidate, and
// hit keys past the first 384 are left as they are.
constexpr int kMaxHitsP = 384;

template <bool kF16>
constexpr uint32_t idesc_s_pair() { return ptx::idesc_f32acc(2 * kM, kN, 0, 0, kF16 ? 0u : 1u); }
template <bool kF16>
constexpr uint32_t idesc_pv_pair() { return ptx::idesc_f32acc(2 * kM, 256, 0, 1, kF16 ? 0u : 1u); }

struct __align__(1024) SmemP {
  uint8_t q[kQBytes];                               // Q tile, then the gate tile
  uint8_t kv[kKRingP + kVRingP][kHalfTileBytes];    // K ring: 0, 1; V ring: 2, 3
  uint64_t q_full;                     // even CTA: both Q tiles have landed
  uint64_t kv_full[kKRingP + kVRingP]; // even CTA: both halves of the slot's tile have landed
  uint64_t kv_empty[kKRingP + kVRingP];// the slot's last product has completed
  uint64_t s_full[2];
  uint64_t p_full[2];                  // even CTA: the 16 softmax warps of the pair wrote P
  uint64_t pv_done;
  uint64_t o_final;
  uint64_t drain;
  uint64_t q_free;                     // every S product has read Q (its buffer takes G)
  uint64_t g_full;                     // this CTA's gate tile has landed
  // cleaning pass
  uint64_t vl_full;                    // this CTA's whole V tile has landed
  uint64_t v_ready;                    // even CTA: both CTAs have cleaned the V tile
  uint64_t vs_ready;                   // this CTA has cleaned the V tile, hits published
  uint64_t v1_empty;                   // the V tile's product has completed
  uint32_t tmem_base;
  int abort;
  int zero;
  int need_clean;                      // a stored output of pass 0 is NaN / Inf
  int peer_flags;                      // from the other CTA: bit 0 need_clean, bit 1 abort
  float red[2][2][kM];                 // [tile parity][half][row]: row maxima, then sums
  int ok[2][2][kM];
  uint32_t tile_hits[2][kN / 32];      // [j & 1]: bit c = key c of tile j is a hit
  int tile_base[2];
  int n_hits;
  int hit_key[kMaxHitsP];
  uint32_t pz[kM][kMaxHitsP / 32];
};
static_assert(sizeof(SmemP) + 1024 <= 227 * 1024, "one CTA per SM");
static_assert(kKRingP * kHalfTileBytes >= kQBytes, "the output tile is staged in the K ring");
static_assert(kVRingP * kHalfTileBytes == kTileBytes, "a whole V tile fits the V ring");

struct ParamsP {
  const uint16_t* G;        // bf16 or fp16 bits
  const uint16_t* V;        // V [B*Hkv, Lkv, 256]: re-read by the cleaning pass
  long long v_rows;
  uint16_t* out;
  float* lse;
  int B, Hq, Hkv, Lq, kv_offset, gqa, R, n_rtiles, n_ptiles;
  LaunchCtl ctl;
};

__device__ __forceinline__ void fail(SmemP& sm, const ParamsP& p) {
  sm.abort = 1;
  record_status(p.ctl.status, GQA_ERR_TIMEOUT);
}

template <bool kF16>
__global__ void __launch_bounds__(kThreadsP, 1)
attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                 const __grid_constant__ CUtensorMap tmO, const ParamsP p) {
  extern __shared__ uint8_t smem_raw[];
  SmemP& sm = *reinterpret_cast<SmemP*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                        ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.ctl.timeout_ns;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool lead = rank == 0;

  // Cluster c -> (pair of row tiles, batch x KV group), the pairs with most keys first.
  const int BH = p.B * p.Hkv;
  const int cl = static_cast<int>(blockIdx.x) >> 1;
  const int pt = p.n_ptiles - 1 - cl / BH;
  const int bg = cl % BH;
  const int b = bg / p.Hkv;
  const int g = bg % p.Hkv;
  const int r0 = (2 * pt + static_cast<int>(rank)) * p.R;
  const int rows_here = min(p.R, p.Lq - r0);   // <= 0: the pair's second tile is past Lq
  const int rt_last = min(2 * pt + 1, p.n_rtiles - 1);
  const int key_end = p.kv_offset + min((rt_last + 1) * p.R, p.Lq);   // keys the pair's last row sees
  const int n_tiles = (key_end + kN - 1) / kN;
  // first key some row of the pair does not see (the cleaning pass's candidates); in
  // fp16 every key (an fp16 P rounds to 0 25 or more log2 units below the row
  // maximum, where float64's p is not 0)
  const int cand_lo = kF16 ? 0 : p.kv_offset + 2 * pt * p.R + 1;
  const uint32_t q_bytes = 4u * 128u * uint32_t(p.R * p.gqa);

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sm.q_full, 1);
    for (int s = 0; s < kKRingP + kVRingP; ++s) {
      ptx::mbar_init(&sm.kv_full[s], 1);
      ptx::mbar_init(&sm.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&sm.s_full[s], 1);
      ptx::mbar_init(&sm.p_full[s], 16);
    }
    ptx::mbar_init(&sm.pv_done, 1);
    ptx::mbar_init(&sm.o_final, 1);
    ptx::mbar_init(&sm.drain, 1);
    ptx::mbar_init(&sm.q_free, 1);
    ptx::mbar_init(&sm.g_full, 1);
    ptx::mbar_init(&sm.vl_full, 1);
    ptx::mbar_init(&sm.v_ready, 2);
    ptx::mbar_init(&sm.vs_ready, 1);
    ptx::mbar_init(&sm.v1_empty, 1);
    sm.abort = 0;
    sm.zero = 0;
    sm.need_clean = 0;
    sm.peer_flags = 0;
    sm.n_hits = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&sm.tmem_base, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // both CTAs' barriers exist before any copy or arrive reaches them
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // the even CTA's barriers, as cluster addresses
  auto lead_bar = [&](uint64_t* bar) { return ptx::mapa_shared(ptx::smem_addr(bar), 0); };

  // One pass over the pair's key tiles (see the one-CTA kernel: a per-tile barrier
  // counts the tiles of both passes, J = J0 + j; a once-per-pass barrier is in phase pp).
  auto run_pass = [&](auto clean_tag) {
    constexpr bool kClean = decltype(clean_tag)::value;
    const int J0 = kClean ? n_tiles : 0;
    const uint32_t pp = kClean ? 1u : 0u;

    if (warp == 0) {
      // ---------------------------------------------------------- producer
      Ring rk = ring_after(J0, kKRingP, 0);
      Ring rv = ring_after(J0, kVRingP, kKRingP);   // pass 0 only
      int v_uses = 0;                              // cleaning pass: V tiles copied
      bool g_issued = false;
      if (lane == 0) {
        if constexpr (!kClean) {
          ptx::prefetch_tmap(&tmQ);
          ptx::prefetch_tmap(&tmK);
          ptx::prefetch_tmap(&tmV);
          ptx::prefetch_tmap(&tmG);
          ptx::prefetch_tmap(&tmO);
        }
        if (lead) ptx::mbar_arrive_expect_tx(&sm.q_full, 2 * q_bytes);
        const uint32_t qf = lead_bar(&sm.q_full);
        for (int dc = 0; dc < 4; ++dc)
          ptx::tma_load_4d_pair(sm.q + dc * kQChunk, &tmQ, qf, dc * 64, r0, g * p.gqa, b);
      }
      int n_hits = 0;
      bool ok = true;
      for (int it = 0; ok && it < 2 * n_tiles; ++it) {
        bool is_v;
        int j;
        item_kind(it, n_tiles, is_v, j);
        const int tile_key0 = j * kN;
        if (!kClean || !is_v) {
          // half of K_j (keys 64r..) or of V_j (dims 128r..) into the ring
          if (!kClean && lane != 0) continue;
          Ring& r = is_v ? rv : rk;
          const int slot = r.at();
          int go = 1;
          if (lane == 0) {
            if (r.count >= r.n &&
                !ptx::mbar_wait(&sm.kv_empty[slot], r.phase ^ 1u, tmo, &sm.abort)) {
              go = 0;
            } else {
              if (lead) ptx::mbar_arrive_expect_tx(&sm.kv_full[slot], 2 * kHalfTileBytes);
              const uint32_t kf = lead_bar(&sm.kv_full[slot]);
              if (!is_v) {
                for (int dc = 0; dc < 4; ++dc)
                  ptx::tma_load_3d_pair(sm.kv[slot] + dc * kKHalfChunk, &tmK, kf, dc * 64,
                                        tile_key0 + 64 * static_cast<int>(rank), bg);
              } else {
                for (int dc = 0; dc < 2; ++dc)
                  ptx::tma_load_3d_pair(sm.kv[slot] + dc * kChunkBytes, &tmV, kf,
                                        128 * static_cast<int>(rank) + 64 * dc, tile_key0, bg);
              }
            }
          }
          if constexpr (kClean) go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) {
            if (lane == 0) fail(sm, p);
            ok = false;
            break;
          }
          r.advance();
          continue;
        }
        // Cleaning pass, V_j: the whole tile into the V ring (this CTA's product half,
        // dims 128r.., first), then its candidate rows cleaned (see the one-CTA kernel).
        int go = 1;
        if (lane == 0) {
          if (v_uses > 0 &&
              !ptx::mbar_wait(&sm.v1_empty, uint32_t(v_uses - 1) & 1u, tmo, &sm.abort)) {
            go = 0;
          } else {
            ptx::mbar_arrive_expect_tx(&sm.vl_full, kTileBytes);
            for (int dc = 0; dc < 4; ++dc)
              ptx::tma_load_3d(sm.kv[kKRingP] + dc * kChunkBytes, &tmV, &sm.vl_full,
                               64 * ((2 * static_cast<int>(rank) + dc) & 3), tile_key0, bg);
          }
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go || !warp_all(ptx::mbar_wait(&sm.vl_full, uint32_t(v_uses) & 1u, tmo, &sm.abort))) {
          if (lane == 0) fail(sm, p);
          ok = false;
          break;
        }
        ++v_uses;
        uint8_t* const vt = sm.kv[kKRingP];
        const int c_lo = min(max(cand_lo - tile_key0, 0), kN);
        HitRows h{{0u, 0u, 0u, 0u}, n_hits, false};
        if (c_lo < kN) {
          const int nr = kN - c_lo;
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
              const int lo = min(max(c_lo - 32 * q, 0), 32);
              w[q] = lo < 32 ? (0xffffffffu << lo) : 0u;
            }
            h = clean_rows<kF16>(sm, vt, make_uint4(w[0], w[1], w[2], w[3]), tile_key0, n_hits);
          }
        }
        if (__any_sync(0xffffffffu, h.wrote)) ptx::fence_proxy_async_smem();
        if (lane == 0) {
          for (int q = 0; q < kN / 32; ++q) sm.tile_hits[j & 1][q] = h.w[q];
          sm.tile_base[j & 1] = n_hits;
          sm.n_hits = h.n;
        }
        n_hits = h.n;
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&sm.vs_ready);
          ptx::mbar_arrive_cluster(lead_bar(&sm.v_ready));
        }
      }
      if (lane == 0) {
        const bool issued_all = kClean ? v_uses == n_tiles : rv.count == J0 + n_tiles;
        // The gate tile (same box as Q) goes into Q's buffer once every S product has
        // read Q; it lands while the last P.V products run.
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
        // Every copy of the pair completes on the even CTA's barriers: that CTA waits
        // for them all before the pair's closing cluster barrier.
        if (lead) {
          for (int c = max(J0, rk.count - rk.n); c < rk.count; ++c)
            ptx::mbar_wait(&sm.kv_full[rk.base + c % rk.n], uint32_t(c / rk.n) & 1u, tmo, &sm.zero);
          if constexpr (!kClean) {
            for (int c = max(J0, rv.count - rv.n); c < rv.count; ++c)
              ptx::mbar_wait(&sm.kv_full[rv.base + c % rv.n], uint32_t(c / rv.n) & 1u, tmo,
                             &sm.zero);
          }
          ptx::mbar_wait(&sm.q_full, pp, tmo, &sm.zero);
        }
        if (g_issued) ptx::mbar_wait(&sm.g_full, pp, tmo, &sm.zero);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      if (lead && lane == 0) {
        bool ok = ptx::mbar_wait(&sm.q_full, pp, tmo, &sm.abort);
        ptx::tc_fence_after();
        const uint32_t qa = ptx::smem_addr(sm.q);
        Ring rk = ring_after(J0, kKRingP, 0);
        Ring rv = ring_after(J0, kVRingP, kKRingP);
        auto issue_s = [&](int j) -> bool {
          const int slot = rk.at();
          if (!ptx::mbar_wait(&sm.kv_full[slot], rk.phase, tmo, &sm.abort)) return false;
          ptx::tc_fence_after();
          const uint32_t ka = ptx::smem_addr(sm.kv[slot]);
          const uint32_t d = tmem + kTmS + uint32_t(kN) * uint32_t((J0 + j) & 1);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint32_t qo = uint32_t(kk >> 2) * kQChunk + uint32_t(kk & 3) * 32u;
            const uint32_t ko = uint32_t(kk >> 2) * kKHalfChunk + uint32_t(kk & 3) * 32u;
            ptx::mma_ss_pair(d, ptx::sdesc_sw128(qa + qo, 16, 1024),
                             ptx::sdesc_sw128(ka + ko, 16, 1024), idesc_s_pair<kF16>(), kk > 0);
          }
          ptx::tc_commit_pair(&sm.s_full[(J0 + j) & 1], 3);
          ptx::tc_commit_pair(&sm.kv_empty[slot], 3);
          rk.advance();
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int J = J0 + j;
          if (!ptx::mbar_wait(&sm.p_full[J & 1], (J >> 1) & 1, tmo, &sm.abort)) return false;
          int slot = kKRingP;
          if constexpr (kClean) {
            if (!ptx::mbar_wait(&sm.v_ready, uint32_t(j) & 1u, tmo, &sm.abort)) return false;
          } else {
            slot = rv.at();
            if (!ptx::mbar_wait(&sm.kv_full[slot], rv.phase, tmo, &sm.abort)) return false;
          }
          ptx::tc_fence_after();
          const uint32_t va = ptx::smem_addr(sm.kv[slot]);
          const uint32_t pa = tmem + kTmS + uint32_t(kN) * uint32_t(J & 1);
          constexpr int kStepsHalf = kHalf / 16;   // k16 steps per softmax half
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            const uint32_t acol = uint32_t(kk / kStepsHalf) * kHalf + uint32_t(kk % kStepsHalf) * 8u;
            ptx::mma_ts_pair(tmem + kTmO, pa + acol,
                             ptx::sdesc_sw128(va + uint32_t(kk) * 2048u, kChunkBytes, 1024),
                             idesc_pv_pair<kF16>(), (j > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::tc_commit_pair(&sm.pv_done, 3);
          if constexpr (kClean) {
            ptx::tc_commit_pair(&sm.v1_empty, 3);
          } else {
            ptx::tc_commit_pair(&sm.kv_empty[slot], 3);
            rv.advance();
          }
          return true;
        };
        if (ok) ok = issue_s(0);
        for (int j = 1; ok && j < n_tiles; ++j) {
          ok = issue_s(j);
          if (ok) ok = issue_pv(j - 1);
        }
        if (ok) ptx::tc_commit_pair(&sm.q_free, 3);   // every S product issued: Q may be overwritten
        if (ok) ok = issue_pv(n_tiles - 1);
        if (ok) {
          ptx::tc_commit_pair(&sm.o_final, 3);
        } else {
          fail(sm, p);
        }
        // Every product issued so far completes before tensor memory is released (or
        // written again by the cleaning pass).
        ptx::tc_commit_pair(&sm.drain, 1);
        ptx::mbar_wait(&sm.drain, pp, tmo, &sm.zero);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- softmax / epilogue
      const int sw = warp - 2;
      const int half = sw >> 2;
      const int lq = warp & 3;
      const int row = lq * 32 + lane;
      const uint32_t bar_id = 1 + lq;
      const int hh = row / p.R;                     // row m: head m / R, prompt row r0 + m % R
      const int rr = row - hh * p.R;
      const bool valid = (row < p.R * p.gqa) && (r0 + rr < p.Lq);
      const int lim = valid ? p.kv_offset + r0 + rr + 1 : p.kv_offset + max(r0, 0) + 1;
      const int q = r0 + rr;
      const uint32_t trow = tmem + (uint32_t(lq * 32) << 16);

      float m_run = -INFINITY;
      float l_part = 0.f;
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const int J = J0 + j;
        const int buf = J & 1;
        const bool mine =
            warp_all(ptx::mbar_wait(&sm.s_full[buf], (J >> 1) & 1, tmo, &sm.abort)) && !sm.abort;
        uint32_t s[kHalf];
        float mx = -INFINITY;
        if (mine) {
          ptx::tc_fence_after();
          const uint32_t sa = trow + kTmS + uint32_t(kN) * buf + uint32_t(kHalf) * half;
          ptx::tmem_ld64_wait(sa, *reinterpret_cast<uint32_t(*)[64]>(&s[0]));
          const int key0 = j * kN + half * kHalf;
          if (key0 + kHalf > lim) {
#pragma unroll
            for (int c = 0; c < kHalf; ++c)
              if (key0 + c >= lim) s[c] = __float_as_uint(-INFINITY);
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
          // warp-uniform branch; only rows whose own max rose past the threshold move it
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
        ptx::tmem_st32_wait(pdst, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        if constexpr (kF16) {
          // fp16: O is rescaled after P_j is stored (see the one-CTA kernel)
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
          // once V_j is cleaned: record, for its hit keys among this thread's keys,
          // whether the probability is 0 (bf16: read back from P; fp16: a -inf score)
          if (warp_all(ptx::mbar_wait(&sm.vs_ready, uint32_t(j) & 1u, tmo, &sm.abort))) {
            const volatile uint32_t* th = sm.tile_hits[j & 1];
            const uint32_t w0 = th[2 * half], w1 = th[2 * half + 1];
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
        if (lane == 0) {
          if (lead)
            ptx::mbar_arrive(&sm.p_full[buf]);
          else
            ptx::mbar_arrive_remote(lead_bar(&sm.p_full[buf]));
        }
      }
      if (!ok) fail(sm, p);

      // -------------------------------------------------------------- epilogue
      bool fin = ok && warp_all(ptx::mbar_wait(&sm.o_final, pp, tmo, &sm.abort));
      const int pb = (J0 + n_tiles) & 1;   // parity slot not used by the last tile's exchange
      sm.red[pb][half][row] = l_part;
      sm.ok[pb][half][row] = fin ? 1 : 0;
      ptx::named_bar_sync(bar_id, 64);
      fin = fin && sm.ok[pb][half ^ 1][row];
      if (p.G != nullptr) fin = warp_all(ptx::mbar_wait(&sm.g_full, pp, tmo, &sm.abort)) && fin;
      const float l_tot = l_part + sm.red[pb][half ^ 1][row];
      // l_tot is 0 exactly when the row saw no key, NaN when it saw a NaN score.
      const float inv_l = l_tot == 0.f ? 0.f : 1.f / l_tot;
      if constexpr (kClean) {
        const int n_hits = *reinterpret_cast<volatile int*>(&sm.n_hits);
        if (n_hits > 0 && __any_sync(0xffffffffu, fin))
          add_hit_terms<kF16, false>(sm, trow + kTmO + 128u * half, row, n_hits, fin && valid,
                                     p.V + (long long)bg * p.v_rows * kHeadDim + half * 128, lim,
                                     INT_MAX, ~0ull, nullptr, 0, 0ll, 0ll);
      }
      // Output staged in the K ring (free once O is final) in Q's swizzled layout and
      // stored by TMA, column blocks 0 and 2 while 1 and 3 are computed (see the one-CTA
      // kernel).  Every softmax thread takes both barriers, failed or not.
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
          if (threadIdx.x == 64 && rows_here > 0 &&
              *reinterpret_cast<volatile int*>(&sm.abort) == 0) {
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
    }
  };

  run_pass(std::false_type{});
  ptx::tc_fence_before();
  __syncthreads();
  // The pair decides together: a cleaning pass when either CTA found a NaN / Inf
  // output and neither stopped on a timeout.
  if (threadIdx.x == 0)
    ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_addr(&sm.peer_flags), rank ^ 1u),
                        (sm.need_clean != 0 ? 1u : 0u) | (sm.abort != 0 ? 2u : 0u));
  ptx::cluster_sync();
  const int flags = *reinterpret_cast<volatile int*>(&sm.peer_flags) |
                    (*reinterpret_cast<volatile int*>(&sm.need_clean) != 0 ? 1 : 0) |
                    (*reinterpret_cast<volatile int*>(&sm.abort) != 0 ? 2 : 0);
  if (flags == 1) {
    // the stores of pass 0 complete before the same rows are stored again, and the
    // zero-probability record starts empty
    if (threadIdx.x == 64) ptx::bulk_wait_group0();
    for (int i = threadIdx.x; i < kM * (kMaxHitsP / 32); i += blockDim.x) (&sm.pz[0][0])[i] = 0u;
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    run_pass(std::true_type{});
    ptx::tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still reach its shared or tensor memory
    ptx::cluster_sync();
  }
  // (without a cleaning pass the exchange above is that barrier: every product, copy
  // and arrive of the pair is complete when a CTA reaches it)
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem, kTmemCols);
}

template <bool kF16>
cudaError_t launch_pair_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tg, const CUtensorMap& to, const ParamsP& p,
                          long long grid, cudaStream_t stream) {
  const size_t smem = sizeof(SmemP) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_pair_kernel<kF16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreadsP);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_pair_kernel<kF16>, tq, tk, tv, tg, to, p);
  if (e == cudaSuccess)
    note_launch(kF16 ? "attn_pair_kernel<prefill,fp16>" : "attn_pair_kernel<prefill,bf16>", grid,
                kThreadsP, smem);
  return e;
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillArgs& a, const LaunchCtl& ctl, cudaStream_t stream,
                                bool* encode_failed) {
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
    // K: a box is 64 keys x 64 dims (a CTA's half of a key tile, one column block);
    // V: 128 keys x 64 dims (one column block of a CTA's half of the dims).
    const int kv_hi = a.kv_offset + a.Lq;
    const cuuint64_t dims[3] = {256, cuuint64_t(kv_hi), cuuint64_t(a.B) * a.Hkv};
    const cuuint64_t str[2] = {512, cuuint64_t(a.Lkv) * 512};
    const cuuint32_t kbox[3] = {64, cuuint32_t(kN / 2), 1};
    const cuuint32_t vbox[3] = {64, cuuint32_t(kN), 1};
    if (!encode_16b(fn, &tk, a.K, 3, dims, str, kbox, a.f16)) *encode_failed = true;
    if (!encode_16b(fn, &tv, a.V, 3, dims, str, vbox, a.f16)) *encode_failed = true;
  }
  if (*encode_failed) return cudaErrorInvalidValue;

  ParamsP p{};
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
  p.n_ptiles = (p.n_rtiles + 1) / 2;
  p.ctl = ctl;
  const long long grid = 2LL * p.n_ptiles * a.B * a.Hkv;
  return a.f16 ? launch_pair_t<true>(tq, tk, tv, tg, to, p, grid, stream)
               : launch_pair_t<false>(tq, tk, tv, tg, to, p, grid, stream);
}

}  // namespace gqa
