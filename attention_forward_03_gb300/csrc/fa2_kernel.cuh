// FlashAttention-2 forward for GB300 (sm_103a): persistent, warp-specialised,
// TMA-fed, tcgen05 tensor cores accumulating in tensor memory (TMEM).
//
// What it computes is the FlashAttention-2 forward pass as the pages define it
// ("FlashAttention-2 MMA 代码学习", steps 0-1: O = softmax(QK^T*scale) V with
// the row-wise online (m, l) merge; yangyitao.com CUDA book ch. 15: outer loop
// over query tiles and inner loop over K/V tiles (15.1, change 1), sequence
// length as a grid axis (15.1, change 2), one thread of work per query row
// with no cross-warp reduction (15.1, change 3, the split-Q idea), deferred
// division by l and LSE = m + log l as the only statistic kept (15.1,
// change 4), causal tile skip, column and row masking for ragged N and the
// -inf guards (15.3)).
//
// Layout of one CTA (one per SM, persistent over work units):
//   work unit  = 256 query rows of one (batch, head): two 128-row sub-tiles.
//   warps 0-3  softmax warpgroup for sub-tile 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax warpgroup for sub-tile 1
//   warps 8-9  tcgen05 MMA issuers (one thread each): at head dim 96 and 128
//              warp 8 issues every S and warp 9 every P.V; at head dim 32
//              and 64 warp 8 + t issues both of sub-tile t. Warp 8 also owns the TMEM
//              allocation. The issuers and the producer sleep briefly between
//              barrier polls, leaving issue slots to the softmax warps that
//              share their SM sub-partitions.
//   warp  10   TMA producer (one thread); warp 11 idle. Warps 8-11 form the
//              third warpgroup, which gives registers to the softmax ones.
// Head dims 32 and 96 run in the layout of 64 and 128 (Dp below): their
// tiles are loaded 64 columns wide, the columns past D filled with zeros by
// the copy engine, and Q.K^T takes only the D/16 steps that cover real data.
// Tensor memory (512 columns x 128 lanes of 32 bits):
//   [128t, 128t+128)      S of sub-tile t (fp32 scores)
//   [256+tDp, 256+tDp+D)  O accumulator of sub-tile t (fp32)
//   [384+64t, 448+64t)    Dp = 64 only: P of sub-tile t (16-bit pairs)
// Shared memory: Q (2 sub-tiles, resident for the segment), at Dp = 128 P
// (2 sub-tiles, 16-bit), and a ring of K/V tiles; all 128-byte swizzled in
// 64-element-wide panels, the operand layout the MMAs read (TMA writes Q/K/V
// that way; the softmax threads write P that way). At Dp = 64 the O
// accumulators leave room for P in tensor memory, where the P.V MMA reads it
// as its A operand (the faster form of the instruction) and its shared
// memory goes to a deeper K/V ring.
//
// Per K/V tile j and sub-tile t the issuers issue:
//   S_t(j+1) = Q_t K_{j+1}^T   once softmax t has loaded S_t(j) into registers
//   O_t (+)= P_t(j) V_j        once softmax t has written P_t(j)
// P lives in shared memory, so the next scores are computed while the softmax
// of the current tile runs: each softmax warpgroup works tile after tile
// without waiting for a P.V product. Rescaling O (rare: the exponent base
// lags the row max by up to 2^8) waits for the previous P.V explicitly.
//
// Schedules. Work is a sequence of segments: K/V tiles [kv_begin, kv_end) of
// one unit. With the round schedule every segment is a whole unit. With the
// stream-K schedule each CTA takes an equal share of all K/V-tile steps, so a
// unit may be cut between consecutive CTAs: the CTA holding the unit's first
// tiles ("owner", the last segment of its share) merges the fp32 partial
// results the following CTAs wrote for the rest of the unit (each as the
// first segment of its share) before writing O and LSE. Partials carry their
// own exponent base and are combined with the usual (m, l) merge.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "fa2_fwd_common.cuh"

namespace fa2 {

template <int D>
struct Layout {
  static_assert(D <= 128 && fwd_head_dim_ok(D), "head dimension");
  // D = 32 and 96 use the tiles of 64 and 128 (their padded columns are zero)
  static constexpr int kPanels = (D + 63) / 64;
  static constexpr int kDp = kPanels * 64;                    // padded head dimension
  static constexpr int kTileBytes = kPanels * kPanelBytes;  // 128 rows x kDp (Q sub-tile, K or V tile)
  static constexpr bool kPInTmem = (kPanels == 1);
  static constexpr int kStages = (kPanels == 2) ? 3 : 12;
  // N of the P.V product = O columns accumulated. At D = 32 it stays 64: a
  // 32-wide B operand would cover half of a 128-byte swizzle row, a form the
  // operand layouts do not describe; the extra columns are P times zero.
  static constexpr int kNpv = (D == 32) ? 64 : D;
  static constexpr int kQBytes = kSubTiles * kTileBytes;
  static constexpr int kPOffset = kQBytes;
  static constexpr int kRingOffset = kPOffset + (kPInTmem ? 0 : kSubTiles * kPTileBytes);
  static constexpr int kBarOffset = kRingOffset + kStages * kTileBytes;
  // barriers: q_full, q_empty, ring full (K tile)[S], ring full (V tile)[S], ring empty[S], s_full[2],
  // s_free[2], p_full[2], p_free[2], o_full[2], drain[2], part_done[2], o_staged[2], o_buf_free[2]
  static constexpr int kNumBars = 2 + 3 * kStages + 2 * 9;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOffset + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kColO = 2 * kKeys;                 // O0 at 256, O1 at 256 + kDp
  static constexpr uint32_t kColP = kColO + 2 * kDp;            // kDp = 64: P0 at 384, P1 at 448
  static_assert(kColO + 2 * kDp + (kPInTmem ? 2 * kKeys / 2 : 0) <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// End of sub-tile 0's K/V range in a segment [b, e). Under the causal mask
// a unit of 256 query rows at q0 = 256 qt needs tiles [0, 2 qt + 2), but
// its first 128 rows see no key of tile 2 qt + 1: when the segment holds
// that tile and at least one other, sub-tile 0 stops one tile early (its S,
// softmax pass and P.V there would only add zeros).
template <bool kCausal>
__device__ __forceinline__ int sub0_end(const Segment& w) {
  if (!kCausal) return w.kv_end;
  const bool skip = w.kv_end == w.nkv && w.nkv == 2 * (w.q0 / (2 * kRows)) + 2 && w.kv_end - 1 > w.kv_begin;
  return skip ? w.kv_end - 1 : w.kv_end;
}

template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const Params p) {
  using L = Layout<D>;
  // MMA issuers split by instruction type (one thread for every S, one for
  // every P.V) or by sub-tile (each thread S and P.V of one sub-tile). Both
  // measured (with the issuers sleeping between polls): by type is 10-15 %
  // faster at head dim 128, by sub-tile 2-6 % faster at head dim 64.
  constexpr bool kTypeSplit = L::kPanels == 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base;
  const uint32_t sP = base + L::kPOffset;
  const uint32_t sRing = base + L::kRingOffset;
  const uint32_t bars = base + L::kBarOffset;
  const uint32_t bar_q_full = bars;
  const uint32_t bar_q_empty = bars + 8;
  // A ring slot holds K and V tiles in turn. Each type has its own "full"
  // barrier per slot, so that each issuer, which takes only one type, waits
  // on a barrier whose every phase it consumes (a barrier's phase is known
  // to a waiter only by its parity). The "empty" barrier is shared: the
  // producer walks every use of a slot in order.
  auto bar_full = [&](int s, uint32_t is_v) { return bars + 16 + 8u * (is_v * L::kStages + s); };
  auto bar_empty = [&](int s) { return bars + 16 + 8u * (2 * L::kStages + s); };
  const uint32_t bar_s_full0 = bars + 16 + 24u * L::kStages;  // [sub-tile]
  const uint32_t bar_s_free0 = bar_s_full0 + 16;              // [sub-tile]
  const uint32_t bar_p_full0 = bar_s_free0 + 16;              // [sub-tile]
  const uint32_t bar_p_free0 = bar_p_full0 + 16;              // [sub-tile]
  const uint32_t bar_o_full0 = bar_p_free0 + 16;              // [sub-tile]
  const uint32_t bar_drain = bar_o_full0 + 16;                // [issuer]
  const uint32_t bar_part0 = bar_drain + 16;                  // [sub-tile]
  // Epilogue at D >= 96: O of sub-tile t is staged in its (then idle) P
  // buffer and stored by TMA; o_staged counts the warpgroup's rows written,
  // o_buf_free tells it the store engine has read the buffer.
  const uint32_t bar_ostage0 = bar_part0 + 16;                // [sub-tile]
  const uint32_t bar_obuf0 = bar_ostage0 + 16;                // [sub-tile]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOffset + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    // released by the S issuer (K tile, Q) or the P.V issuer (V tile); with
    // per-sub-tile issuers by both issuers
    mbar_init(bar_q_empty, kTypeSplit ? 1 : 2);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_full(s, 0u), 1);
      mbar_init(bar_full(s, 1u), 1);
      mbar_init(bar_empty(s), kTypeSplit ? 1 : 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s_full0 + 8 * t, 1);
      mbar_init(bar_s_free0 + 8 * t, 4 * 32);
      mbar_init(bar_p_full0 + 8 * t, 4 * 32);
      mbar_init(bar_p_free0 + 8 * t, 1);
      mbar_init(bar_o_full0 + 8 * t, 1);
      mbar_init(bar_drain + 8 * t, 1);
      mbar_init(bar_part0 + 8 * t, 4 * 32);
      mbar_init(bar_ostage0 + 8 * t, 4 * 32);
      mbar_init(bar_obuf0 + 8 * t, 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
    // The first segment's Q and first K tile are requested here, before the
    // TMEM allocation, the CTA barrier and the register hand-off, so that
    // their load latency overlaps that set-up; the producer carries on after
    // them (ring slot 0).
    SegCursor c0 = first_cursor(p);
    Segment w0;
    if (next_segment<kCausal>(c0, w0, p)) {
      mbar_arrive_expect_tx(bar_q_full, L::kQBytes);
      for (int t = 0; t < kSubTiles; ++t)
        for (int pn = 0; pn < L::kPanels; ++pn)
          tma_load_3d_hint(sQ + t * L::kTileBytes + pn * kPanelBytes, &tmQ, bar_q_full, pn * 64, w0.q0 + t * kRows,
                           w0.bh, l2_policy_evict_first());
      if (!p.test_withhold) {  // test hook: the first tile never arrives
        mbar_arrive_expect_tx(bar_full(0, 0u), L::kTileBytes);
        for (int pn = 0; pn < L::kPanels; ++pn)
          tma_load_3d_hint(sRing + pn * kPanelBytes, &tmK, bar_full(0, 0u), pn * 64, w0.kv_begin * kKeys, w0.bh,
                           l2_policy_evict_last());
      }
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  Watchdog wd;
  wd.status = p.status;
  wd.abort_flag = abort_flag;
  wd.limit_ns = p.watchdog_ns;

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
    if (warp == kLoadWarp) {
      // ---------------------------------------------------------- producer
      // Ring order per segment [b, e): K_b, then for each j: K_{j+1}, V_j —
      // the order the MMA issuers consume and release them.
      if (lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        const uint64_t keep = l2_policy_evict_last();          // K/V: re-read by every query tile of the head
        const uint64_t stream_once = l2_policy_evict_first();  // Q: read once
        int slot = 0;
        uint32_t ring_ph = 0, issued = 0, q_round = 0;
        // per slot: type of its latest tile (bit set: V) and the parity of
        // the next use of its K / V full barrier
        uint32_t types = 0, kbits = 0, vbits = 0;
        bool ok = true;
        SegCursor cur = first_cursor(p);
        Segment w;
        auto load_tile = [&](const CUtensorMap* map, int j, uint32_t is_v) -> bool {
          if (!wait_bounded(bar_empty(slot), ring_ph ^ 1u, wd, kSiteLoadRingEmpty, true, kNapNs)) return false;
          const uint32_t full = bar_full(slot, is_v);
          if (!(p.test_withhold && issued == 0)) {  // test hook: the first tile never arrives
            mbar_arrive_expect_tx(full, L::kTileBytes);
            for (int pn = 0; pn < L::kPanels; ++pn)
              tma_load_3d_hint(sRing + slot * L::kTileBytes + pn * kPanelBytes, map, full, pn * 64, j * kKeys,
                               w.bh, keep);
          }
          types = (types & ~(1u << slot)) | (is_v << slot);
          if (is_v) vbits ^= 1u << slot; else kbits ^= 1u << slot;
          ++issued;
          if (++slot == L::kStages) {
            slot = 0;
            ring_ph ^= 1u;
          }
          return true;
        };
        while (ok && next_segment<kCausal>(cur, w, p)) {
          if (q_round == 0) {
            // Q and K_b of the first segment were requested at kernel entry
            // (into ring slot 0): account for them as loads of this thread.
            q_round = 1;
            kbits ^= 1u;
            ++issued;
            slot = 1;
          } else {
            if (!wait_bounded(bar_q_empty, (q_round - 1) & 1u, wd, kSiteLoadQEmpty, true, kNapNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar_q_full, L::kQBytes);
            for (int t = 0; t < kSubTiles; ++t)
              for (int pn = 0; pn < L::kPanels; ++pn)
                tma_load_3d_hint(sQ + t * L::kTileBytes + pn * kPanelBytes, &tmQ, bar_q_full, pn * 64,
                                 w.q0 + t * kRows, w.bh, stream_once);
            ++q_round;
            ok = load_tile(&tmK, w.kv_begin, 0u);
          }
          for (int j = w.kv_begin; j < w.kv_end && ok; ++j) {
            if (j + 1 < w.kv_end) ok = load_tile(&tmK, j + 1, 0u);
            if (ok) ok = load_tile(&tmV, j, 1u);
          }
        }
        // Drain: every copy issued must have landed before the CTA may exit.
        const uint32_t first = issued > (uint32_t)L::kStages ? issued - L::kStages : 0u;
        for (uint32_t i = first; i < issued; ++i) {  // the latest tile of each slot
          const int s = static_cast<int>(i % L::kStages);
          const uint32_t is_v = (types >> s) & 1u;
          const uint32_t par = (((is_v ? vbits : kbits) >> s) & 1u) ^ 1u;
          wait_bounded(bar_full(s, is_v), par, wd, kSiteDrain, false, kNapNs);
        }
        if (q_round > 0) wait_bounded(bar_q_full, (q_round - 1) & 1u, wd, kSiteDrain, false, kNapNs);
      }
      __syncwarp();
    } else if (warp < kMmaWarp + kIssuers) {
      // ------------------------------------------------------ MMA issuers
      if (lane == 0) {
        const int me = warp - kMmaWarp;  // split by type: 0 issues every S, 1 every P.V; else sub-tile me
        constexpr uint32_t idesc_s = make_idesc_f16(kBf16, kKeys, false);
        constexpr uint32_t idesc_o = make_idesc_f16(kBf16, L::kNpv, true);
        // Descriptor low words advance by compile-time offsets (the start
        // address field never carries: shared memory stays below 256 KB);
        // the high words are constants.
        constexpr uint32_t kHi = desc_hi_sw128(1024);  // 8-row (K-major) / 8-key (MN-major) groups 1 KB apart
        // S_t = Q_t K^T : D/16 steps of K=16 along the head dimension.
        auto issue_s = [&](int t, int slot) {
          const uint32_t q_lo = desc_lo_sw128(sQ, 16);
          const uint32_t ring_lo = desc_lo_sw128(sRing, 16);
          const uint32_t qa = q_lo + static_cast<uint32_t>((t * L::kTileBytes) >> 4);
          const uint32_t ka = ring_lo + static_cast<uint32_t>(slot * (L::kTileBytes >> 4));
          const uint32_t dt = tmem + static_cast<uint32_t>(t * kKeys);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
            mma_ss_w(dt, qa + off, kHi, ka + off, kHi, idesc_s, kk > 0 ? 1u : 0u);
          }
        };
        // O_t (+)= P_t V : P (K-major, shared memory; Dp = 64: tensor memory)
        // and V (MN-major, shared memory), 8 steps of 16 keys.
        auto issue_pv = [&](int t, int slot, bool acc) {
          const uint32_t p_lo = desc_lo_sw128(sP, 16);
          const uint32_t ring_lo_v = desc_lo_sw128(sRing, kPanelBytes);  // V: 64-column panels 16 KB apart
          const uint32_t pa = p_lo + static_cast<uint32_t>((t * kPTileBytes) >> 4);
          const uint32_t va = ring_lo_v + static_cast<uint32_t>(slot * (L::kTileBytes >> 4));
          const uint32_t dt = tmem + L::kColO + static_cast<uint32_t>(t * L::kDp);
          const uint32_t pt = tmem + L::kColP + static_cast<uint32_t>(t * (kKeys / 2));
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk) {
            const uint32_t vb = va + static_cast<uint32_t>((kk * 16 * 128) >> 4);
            const uint32_t acc_kk = (acc || kk > 0) ? 1u : 0u;
            if constexpr (L::kPInTmem) {
              mma_ts_w(dt, pt + 8u * kk, vb, kHi, idesc_o, acc_kk);
            } else {
              const uint32_t po = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
              mma_ss_w(dt, pa + po, kHi, vb, kHi, idesc_o, acc_kk);
            }
          }
        };

        // Position of a tile in the producer's load sequence of a segment
        // [b, e): K_b, then for each j: K_{j+1} (if any), V_j. Each issuer
        // walks the ring through the global load index of its own tiles.
        auto k_index = [](int j, int b) { return j == b ? 0 : 2 * (j - b) - 1; };
        auto v_index = [](int j, int b, int e) { return j == e - 1 ? 2 * (j - b) + 1 : 2 * (j - b) + 2; };
        // Each issuer takes every tile of the types it uses in load order;
        // bit s of bits[type] is the parity of the next use of slot s's full
        // barrier for that type.
        uint32_t bits[2] = {0u, 0u};
        auto take = [&](uint32_t idx, uint32_t is_v) -> int {
          const int s = static_cast<int>(idx % L::kStages);
          const uint32_t par = (bits[is_v] >> s) & 1u;
          bits[is_v] ^= 1u << s;
          return wait_bounded(bar_full(s, is_v), par, wd, kSiteMmaRingFull, true, kNapNs) ? s : -1;
        };
        uint32_t base_idx = 0;  // global load index of the current segment's first tile
        bool ok = true;
        SegCursor cur = first_cursor(p);
        Segment w;
        if constexpr (kTypeSplit) {
          if (me == 0) {
            // S issuer: S_t(j) for both sub-tiles, each as soon as K_j has landed
            // and the softmax has loaded the sub-tile's previous S (also across
            // segments) into registers.
            uint32_t q_round = 0, s_free_ph[2] = {0u, 0u};
            bool s_out[2] = {false, false};  // an S issued whose TMEM the softmax has not released yet
            while (ok && next_segment<kCausal>(cur, w, p)) {
              const int b = w.kv_begin, e = w.kv_end;
              if (!wait_bounded(bar_q_full, q_round & 1u, wd, kSiteMmaQFull, true, kNapNs)) { ok = false; break; }
              ++q_round;
              for (int j = b; j < e && ok; ++j) {
                const int slot_k = take(base_idx + k_index(j, b), 0u);
                if (slot_k < 0) { ok = false; break; }
                for (int t = 0; t < 2; ++t) {
                  if (s_out[t]) {
                    if (!wait_bounded(bar_s_free0 + 8 * t, s_free_ph[t], wd, kSiteMmaSFree, true, kNapNs)) { ok = false; break; }
                    s_free_ph[t] ^= 1u;
                  }
                  tc_fence_after_sync();
                  issue_s(t, slot_k);
                  mma_commit(bar_s_full0 + 8 * t);
                  s_out[t] = true;
                }
                if (!ok) break;
                mma_commit(bar_empty(slot_k));
                if (j == e - 1) mma_commit(bar_q_empty);
              }
              base_idx += 2u * static_cast<uint32_t>(e - b);
            }
          } else {
            // P.V issuer: O_t += P_t(j) V_j for both sub-tiles, each as soon as
            // V_j has landed and the softmax has published P_t(j).
            uint32_t p_full_ph[2] = {0u, 0u};
            while (ok && next_segment<kCausal>(cur, w, p)) {
              const int b = w.kv_begin, e = w.kv_end;
              for (int j = b; j < e && ok; ++j) {
                const int slot_v = take(base_idx + v_index(j, b, e), 1u);
                if (slot_v < 0) { ok = false; break; }
                for (int t = 0; t < 2; ++t) {
                  if (!wait_bounded(bar_p_full0 + 8 * t, p_full_ph[t], wd, kSiteMmaPFull, true, kNapNs)) { ok = false; break; }
                  p_full_ph[t] ^= 1u;
                  tc_fence_after_sync();
                  issue_pv(t, slot_v, j > b);
                  mma_commit(bar_p_free0 + 8 * t);
                  if (j == e - 1) mma_commit(bar_o_full0 + 8 * t);
                }
                if (!ok) break;
                mma_commit(bar_empty(slot_v));
              }
              base_idx += 2u * static_cast<uint32_t>(e - b);
            }
          }
        } else {
          // One issuer per sub-tile t = me: S_t one tile ahead of P.V_t, each
          // S as soon as its K tile has landed and the softmax has loaded the
          // previous S of the sub-tile, each P.V as soon as its V tile has
          // landed and the softmax has published P_t.
          const int t = me;
          uint32_t q_round = 0, s_free_ph = 0, p_full_ph = 0;
          bool s_out = false;
          bool skip_s = false;  // the S of the tile being taken is skipped (sub-tile 0, masked tile)
          auto next_s = [&](int slot_k) -> bool {
            if (skip_s) {  // a tile sub-tile 0 skips: release the K slot, no product
              mma_commit(bar_empty(slot_k));
              return true;
            }
            if (s_out) {
              if (!wait_bounded(bar_s_free0 + 8 * t, s_free_ph, wd, kSiteMmaSFree, true, kNapNs)) return false;
              s_free_ph ^= 1u;
            }
            tc_fence_after_sync();
            issue_s(t, slot_k);
            mma_commit(bar_s_full0 + 8 * t);
            mma_commit(bar_empty(slot_k));
            s_out = true;
            return true;
          };
          while (ok && next_segment<kCausal>(cur, w, p)) {
            const int b = w.kv_begin, e = w.kv_end;
            const int et = t == 0 ? sub0_end<kCausal>(w) : e;  // this sub-tile's end
            if (!wait_bounded(bar_q_full, q_round & 1u, wd, kSiteMmaQFull, true, kNapNs)) { ok = false; break; }
            ++q_round;
            int slot_k = take(base_idx + k_index(b, b), 0u);
            skip_s = false;
            if (slot_k < 0 || !next_s(slot_k)) { ok = false; break; }
            if (e - b == 1) mma_commit(bar_q_empty);
            for (int j = b; j < e && ok; ++j) {
              if (j + 1 < e) {
                slot_k = take(base_idx + k_index(j + 1, b), 0u);
                skip_s = j + 1 >= et;
                if (slot_k < 0 || !next_s(slot_k)) { ok = false; break; }
                if (j + 2 == e) mma_commit(bar_q_empty);
              }
              const int slot_v = take(base_idx + v_index(j, b, e), 1u);
              if (slot_v < 0) { ok = false; break; }
              if (j < et) {
                if (!wait_bounded(bar_p_full0 + 8 * t, p_full_ph, wd, kSiteMmaPFull, true, kNapNs)) { ok = false; break; }
                p_full_ph ^= 1u;
                tc_fence_after_sync();
                issue_pv(t, slot_v, j > b);
                mma_commit(bar_p_free0 + 8 * t);
                if (j == et - 1) mma_commit(bar_o_full0 + 8 * t);
              }
              mma_commit(bar_empty(slot_v));
            }
            base_idx += 2u * static_cast<uint32_t>(e - b);
          }
        }
        // Drain: all issued tensor-core work completes before TMEM is released.
        mma_commit(bar_drain + 8 * me);
        wait_bounded(bar_drain + 8 * me, 0u, wd, kSiteDrain, false, kNapNs);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------- softmax warpgroups
    const int t = warp >> 2;                 // sub-tile
    const int wr = warp & 3;                 // warp within the warpgroup: TMEM lanes 32*wr..
    const int rr = wr * 32 + lane;           // row within the sub-tile
    const uint32_t lane_off = static_cast<uint32_t>(wr * 32) << 16;
    const uint32_t tS = tmem + lane_off + static_cast<uint32_t>(t * kKeys);
    const uint32_t tO = tmem + lane_off + L::kColO + static_cast<uint32_t>(t * L::kDp);
    const uint32_t bar_s = bar_s_full0 + 8 * t;
    const uint32_t bar_sf = bar_s_free0 + 8 * t;
    const uint32_t bar_p = bar_p_full0 + 8 * t;
    const uint32_t bar_pf = bar_p_free0 + 8 * t;
    const uint32_t bar_o = bar_o_full0 + 8 * t;
    // this thread's P row in shared memory: 128 bytes per 64 keys, 16-byte
    // chunks placed by the 128-byte swizzle (chunk c of row r at c ^ (r % 8))
    const uint32_t p_row = sP + static_cast<uint32_t>(t * kPTileBytes + rr * 128);
    const uint32_t tP = tmem + lane_off + L::kColP + static_cast<uint32_t>(t * (kKeys / 2));
    const uint32_t p_xor = static_cast<uint32_t>(rr & 7);
    const float c = p.scale_log2;
    uint32_t s_phase = 0, o_phase = 0, part_phase = 0;
    // D >= 96, O staged in the P buffer (see the epilogue): bit 0 the parity
    // of the next o_staged phase, bit 1 that of o_buf_free, bit 2 set while
    // the buffer holds an O whose store may still be reading it
    uint32_t ost_state = 0;
    uint32_t p_count = 0;  // P tiles published so far (= P.V products issued or pending)
    bool ok = true;
    SegCursor cur = first_cursor(p);
    Segment w;
    while (ok && next_segment<kCausal>(cur, w, p)) {
      if constexpr (!L::kPInTmem) {
        // the previous segment's O was staged in this P buffer: the store
        // engine must have read it before this segment's first P overwrites it
        if (ost_state & 4u) {
          bool fb = wait_bounded(bar_obuf0 + 8 * t, (ost_state >> 1) & 1u, wd, kSiteOBufFree);
          fb = __all_sync(0xffffffffu, fb);
          if (!fb) break;
          ost_state = (ost_state ^ 2u) & ~4u;
        }
      }
      const int row = w.q0 + t * kRows + rr;
      const int limit = kCausal ? min(p.N, row + 1) : p.N;  // allowed keys: [0, limit)
      float m_raw = -CUDART_INF_F;  // running max of the raw scores seen so far
      float base = -CUDART_INF_F;   // exponent base (log2 units) that l and O are relative to
      float l = 0.f;    // sum of p (unrounded): LSE
      float l_o = 0.f;  // normaliser of O (see below)
      // sub-tile 0 skips its fully masked last tile where each sub-tile has
      // its own MMA issuer (D <= 64; with the issuers split by type the two
      // sub-tiles must stay in step)
      const int e_t = (t == 0 && L::kPInTmem) ? sub0_end<kCausal>(w) : w.kv_end;
      for (int j = w.kv_begin; j < e_t; ++j) {
        bool got = wait_bounded(bar_s, s_phase, wd, kSiteSoftmaxSFull);
        got = __all_sync(0xffffffffu, got);
        if (!got) { ok = false; break; }
        s_phase ^= 1u;
        tc_fence_after_sync();
        uint32_t sr[128];
        tmem_ld32x128_wait(tS, sr);
        // S is in registers: the issuer may compute the next scores into TMEM.
        tc_fence_before_sync();
        mbar_arrive(bar_sf);
        float s[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i]);
        const int kv0 = j * kKeys;
        if (kv0 + kKeys > limit) {  // ragged tail and/or causal diagonal: mask disallowed keys
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (kv0 + i >= limit) s[i] = -CUDART_INF_F;
        }
        // row max: four independent chains of 3-input maxima
        float mx[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mx[q] = fmax3(s[32 * q], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
          for (int i = 3; i < 31; i += 2) mx[q] = fmax3(mx[q], s[32 * q + i], s[32 * q + i + 1]);
          mx[q] = fmaxf(mx[q], s[32 * q + 31]);
        }
        const float m_tile = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]);
        m_raw = fmaxf(m_raw, m_tile);
        // Move the exponent base only when the max has grown by more than
        // kRescaleLog2 (or on the first tile); otherwise keep the old base, so
        // every p stays below 2^kRescaleLog2 and O, l need no rescale.
        // While a row has seen no allowed key its base stays -inf and every p
        // is 0 (exponent offset 0 instead of -inf, so no inf - inf).
        const float cand = m_raw * c;
        float alpha = 1.f;
        if (m_raw != -CUDART_INF_F && (base == -CUDART_INF_F || cand - base > kRescaleLog2)) {
          alpha = ex2_approx(base - cand);  // 0 on the first tile with an allowed key
          base = cand;
        }
        const float nb = (base == -CUDART_INF_F) ? 0.f : -base;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // p = 2^(s*c - base), packed to 16-bit pairs in registers while the
        // previous P.V may still be reading the P buffer.
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float x0, x1;
          ffma2_bcast(x0, x1, s[2 * i], s[2 * i + 1], c, nb);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          fadd2_acc(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], p0, p1);
          pk[i] = pack2(p0, p1, kBf16);
        }
        // The previous P.V must be complete before its P buffer is
        // overwritten and before O is rescaled.
        if (p_count > 0) {
          bool fr = wait_bounded(bar_pf, (p_count - 1) & 1u, wd, kSiteSoftmaxPFree);
          fr = __all_sync(0xffffffffu, fr);
          if (!fr) { ok = false; break; }
          tc_fence_after_sync();
        }
        if constexpr (L::kPInTmem) {
          // P: this row's 64 packed pairs into its lane of the P columns
          tmem_st32x32(tP, *reinterpret_cast<const uint32_t(*)[32]>(pk));
          tmem_st32x32(tP + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
        } else {
          // P: 16 chunks of 8 keys (4 packed pairs) into the swizzled row
#pragma unroll
          for (int ch = 0; ch < 16; ++ch) {
            const uint32_t addr = p_row + static_cast<uint32_t>((ch >> 3) * kPanelBytes) +
                                  ((static_cast<uint32_t>(ch & 7) ^ p_xor) << 4);
            st_shared_v4(addr, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
          }
        }
        // O holds P.V up to tile j-1 (complete, see above): rescale it now
        // that the scores are no longer held in registers.
        if (j > w.kv_begin && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tmem_ld32x32_wait(tO + cc, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32x32(tO + cc, o);
          }
        }
        tmem_wait_st();
        // the tensor core reads a shared-memory P through the async proxy
        if constexpr (!L::kPInTmem) fence_proxy_async_shared();
        tc_fence_before_sync();
        mbar_arrive(bar_p);
        ++p_count;
        const float lt = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        // P.V uses p rounded to 16 bits. With the base lagging the max, the
        // tile's largest p is not a power of two, so its rounding would leave
        // the dominant weight unnormalised; the O normaliser carries the
        // rounded value of that element (recomputed exactly as above) while
        // the LSE keeps the unrounded sum.
        float px, pxr;
        {
          float x0, x1;
          ffma2_bcast(x0, x1, m_tile, m_tile, c, nb);
          px = ex2_approx(x0);
          pxr = round16(px, kBf16);
        }
        l = l * alpha + lt;
        l_o = l_o * alpha + (lt + (pxr - px));
      }
      if (!ok) break;
      // -------------------------------------------------------- epilogue
      bool got = wait_bounded(bar_o, o_phase, wd, kSiteSoftmaxOFull);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      o_phase ^= 1u;
      tc_fence_after_sync();
      if (w.kv_begin > 0) {
        // Not the unit's first tiles: hand the unnormalised partial (O, base,
        // l, l_o) to the owner through this CTA's workspace slot.
        const size_t slot = static_cast<size_t>(blockIdx.x) * 2 + t;
        float* po = p.ws_o + slot * D * 128;
        float* ps = p.ws_stats + slot * 3 * 128;
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32x32_wait(tO + cc, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) __stcg(po + (cc + i) * 128 + rr, __uint_as_float(o[i]));
        }
        __stcg(ps + rr, base);
        __stcg(ps + 128 + rr, l);
        __stcg(ps + 256 + rr, l_o);
        __threadfence();
        mbar_arrive(bar_part0 + 8 * t);
        if (rr < 32) {  // the first warp waits as a whole, so that it stays converged
          bool done = wait_bounded(bar_part0 + 8 * t, part_phase, wd, kSitePartialWrite);
          done = __all_sync(0xffffffffu, done);
          if (!done) break;
          if (rr == 0) store_release(p.ws_flags + slot, p.epoch);
        }
        part_phase ^= 1u;
        tc_fence_before_sync();
        continue;
      }
      // Owner (or whole unit): fold in the partials of the CTAs that took the
      // rest of this unit, if any, then normalise and write O and LSE.
      float a_own = 1.f, nbase = base;
      int first_c = blockIdx.x + 1, last_c = blockIdx.x;  // partial holders [first_c, last_c]
      if (p.stream_k && w.kv_end < w.nkv) {
        while (last_c + 1 < static_cast<int>(gridDim.x) && stream_k_begin(p, last_c + 1) < w.unit_end) ++last_c;
        bool fine = true;
        for (int cb = first_c; cb <= last_c && fine; ++cb)
          fine = wait_flag(p.ws_flags + static_cast<size_t>(cb) * 2 + t, p.epoch, wd, kSitePartialFlag);
        fine = __all_sync(0xffffffffu, fine);
        if (!fine) break;
        for (int cb = first_c; cb <= last_c; ++cb)
          nbase = fmaxf(nbase, __ldcg(p.ws_stats + (static_cast<size_t>(cb) * 2 + t) * 3 * 128 + rr));
        a_own = ex2_approx(base - nbase);
        l *= a_own;
        l_o *= a_own;
        for (int cb = first_c; cb <= last_c; ++cb) {
          const float* ps = p.ws_stats + (static_cast<size_t>(cb) * 2 + t) * 3 * 128;
          const float a = ex2_approx(__ldcg(ps + rr) - nbase);  // 0 for a partial that saw no key
          l += a * __ldcg(ps + 128 + rr);
          l_o += a * __ldcg(ps + 256 + rr);
        }
        base = nbase;
      }
      const float inv = (l > 0.f) ? __frcp_rn(l_o) : 0.f;
      const bool live = row < p.N;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      (static_cast<size_t>(w.bh) * p.N + (live ? row : 0)) * (D * 2);
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t o[32];
        tmem_ld32x32_wait(tO + cc, o);
        float of[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) of[i] = __uint_as_float(o[i]) * a_own;
        for (int cb = first_c; cb <= last_c; ++cb) {
          const size_t slot = static_cast<size_t>(cb) * 2 + t;
          const float a = ex2_approx(__ldcg(p.ws_stats + slot * 3 * 128 + rr) - nbase);
          const float* po = p.ws_o + slot * D * 128;
#pragma unroll
          for (int i = 0; i < 32; ++i) of[i] = fmaf(a, __ldcg(po + (cc + i) * 128 + rr), of[i]);
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2(of[2 * i] * inv, of[2 * i + 1] * inv, kBf16);
        if constexpr (L::kPInTmem) {
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 2);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        } else {
          // into this row of the P buffer, in the 128-byte-swizzled layout
          // of the O map's boxes (8-element chunk c of the row at panel c/8,
          // chunk (c mod 8) xor (row mod 8))
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c8 = cc / 8 + q;
            const uint32_t addr = p_row + static_cast<uint32_t>((c8 >> 3) * kPanelBytes) +
                                  ((static_cast<uint32_t>(c8 & 7) ^ p_xor) << 4);
            st_shared_v4(addr, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
      }
      if constexpr (!L::kPInTmem) {
        // One thread stores the staged tile with TMA once every row is in
        // (rows past N are clipped by the map; a sub-tile wholly past N has
        // nothing to store). Coalesced, asynchronous writes instead of each
        // thread's 16-byte pieces of its own row, which serialised in the
        // load/store unit (about 6,000 cycles per epilogue).
        fence_proxy_async_shared();
        mbar_arrive(bar_ostage0 + 8 * t);
        if (rr == 0 && wait_bounded(bar_ostage0 + 8 * t, ost_state & 1u, wd, kSiteOStaged)) {
          if (w.q0 + t * kRows < p.N) {
            const uint32_t p_tile = sP + static_cast<uint32_t>(t * kPTileBytes);
            for (int pn = 0; pn < L::kPanels; ++pn)
              tma_store_3d(&tmO, p_tile + static_cast<uint32_t>(pn * kPanelBytes), pn * 64, w.q0 + t * kRows, w.bh);
            bulk_commit_group();
            bulk_wait_read_all();
          }
          mbar_arrive(bar_obuf0 + 8 * t);
        }
        ost_state = (ost_state ^ 1u) | 4u;
      }
      if (live) {
        p.lse[static_cast<size_t>(w.bh) * p.N + row] =
            (l > 0.f) ? (base + __log2f(l)) * 0.69314718055994530942f : CUDART_INF_F;
      }
      // O_t is read out; the next segment's first P.V may overwrite it once
      // this warpgroup publishes that segment's first P (ordered by bar_p).
      tc_fence_before_sync();
    }
    // the O stores this thread issued complete before the CTA exits
    if constexpr (!L::kPInTmem) {
      if (rr == 0) bulk_wait_all();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The stream-K schedule waits across CTAs, so it is launched cooperatively
// (the whole grid resident at once, or the launch fails).
template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                       const Params& p, int grid, cudaStream_t stream) {
  auto kern = fa2_fwd_kernel<D, kBf16, kCausal>;
  const int smem = Layout<D>::kSmemBytes;
  // Once per device: the register check and the shared-memory opt-in.
  static PerDeviceOnce prepared;
  const cudaError_t e = once_per_device(prepared, [&]() -> cudaError_t {
    cudaFuncAttributes fa;
    cudaError_t r = cudaFuncGetAttributes(&fa, kern);
    if (r != cudaSuccess) return r;
    // The in-kernel register split assumes exactly kLaunchRegs per thread at
    // launch; any other count could leave a warpgroup waiting for registers.
    if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = p.stream_k ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, p);
}

}  // namespace fa2
