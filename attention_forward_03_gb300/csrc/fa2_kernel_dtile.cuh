// FlashAttention-2 forward for GB300 (sm_103a) at head dimensions 512 and
// 1024: the output's head dimension is tiled.
//
// The operation is the one of fa2_kernel.cuh (the pages' FlashAttention-2
// forward: "FlashAttention-2 MMA 代码学习", steps 0-1; yangyitao.com CUDA
// book ch. 15, sections 15.1 and 15.3). The tiling_qk page of the GitHub
// mirror adds these head dims by tiling the head dimension of Q.K^T; here
// Q.K^T is tiled along d as well (its K-steps walk 128-column chunks of Q and
// K), and so is the output: a 128-row fp32 O accumulator would need D tensor-
// memory columns (all 512 at D = 512, twice that at 1024), so each work unit
// owns one 256-column chunk of O. A unit is (128 query rows of one (batch,
// head), output chunk oc); it computes the full scores S = Q K^T over all of
// D, the online softmax of the pages, and O[:, 256 oc : 256 oc + 256] += P V
// for its chunk only. The D / 256 units of one query tile each recompute the
// same S and the same row statistics (the arithmetic is identical, so they
// agree bit for bit); the unit with oc = 0 writes the LSE. The cost is the
// recomputed S: the tensor cores do 1.5x (D = 512) or 2.5x (D = 1024) the
// FLOPs of the definition.
//
// Layout of one CTA (one per SM, persistent over work units):
//   warps 0-3  softmax warpgroup (thread = query row = TMEM lane)
//   warps 4-7  idle (the launch's register split is the other kernels')
//   warp  8    S issuer: S(j) = sum over chunks c of Q_c K_{j,c}^T
//              (D / 16 K-steps); owns the TMEM allocation
//   warp  9    P.V issuer: O_oc (+)= P(j) V_j[:, oc] (8 K-steps of N = 256,
//              A = P from tensor memory)
//   warp 10    TMA producer; warp 11 idle
// Tensor memory: [0,128) S, [128,384) O (this unit's 256 columns), [384,448)
// P (16-bit pairs). One S buffer: the softmax copies S into registers and
// releases it at once, so S(j+1) is computed during the softmax of tile j.
// Shared memory at D = 512: the unit's Q (128 KB, resident for the segment)
// and a ring of three 32 KB slots; at D = 1024 (a resident Q would be 256 KB)
// a ring of seven slots and nothing else, Q streaming through the ring with
// K. Slot contents: a chunk of K (or, at D = 1024, of Q): 128 rows x 128
// head-dim columns, two 64-column panels; or half a V tile (64 keys x the
// unit's 256 columns, four panels of 64 rows); all 128-byte swizzled. Load
// order per segment [b, e): Q (D = 512), the S operands of tile b (K_{b,0},
// K_{b,1}, ...; at D = 1024 Q_0, K_{b,0}, Q_1, K_{b,1}, ...), then for each j:
// those of tile j+1 (if any), V_j's two halves.
// Only the round schedule runs here (whole units dealt to the CTAs); the
// host never asks for stream-K at these head dims.
#pragma once
#include "fa2_fwd_common.cuh"

namespace fa2 {

template <int D>
struct DtileLayout {
  static_assert(D == 512 || D == 1024, "the d-tiled kernel is built for head dimensions 512 and 1024");
  static constexpr int kChunks = D / 128;                   // S operand chunks (128 head-dim columns each)
  static constexpr int kOutChunks = D / kDtileOutCols;      // output chunks per query tile
  static constexpr int kSlotBytes = 2 * kPanelBytes;        // 32 KB
  static constexpr int kVPanelBytes = kSlotBytes / 4;       // V half: 64 rows x 64 columns per panel
  // Q resident in shared memory (D = 512: 128 rows x 512 = 128 KB) or
  // streamed through the ring with K (D = 1024)
  static constexpr bool kQRes = (D == 512);
  static constexpr int kQBytes = kQRes ? kRows * D * 2 : 0;
  static constexpr int kStages = kQRes ? 3 : 7;
  static constexpr int kItemsS = kQRes ? kChunks : 2 * kChunks;  // ring items of one S: K_c (and Q_c) per chunk
  static constexpr int kRingOffset = kQBytes;
  static constexpr int kBarOffset = kRingOffset + kStages * kSlotBytes;
  // barriers: ring full (S operand)[S], ring full (V half)[S], ring empty[S], s_full, s_free, p_full, p_free,
  // o_full, drain[2], q_full, q_empty
  static constexpr int kNumBars = 3 * kStages + 9;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOffset + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kColO = kKeys;                      // O at 128
  static constexpr uint32_t kColP = kColO + kDtileOutCols;      // P at 384
  static_assert(kColP + kKeys / 2 <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_fwd_dtile_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = DtileLayout<D>;
  constexpr int kR = 1;  // query sub-tiles per work unit
  constexpr int kNC = L::kChunks;
  constexpr int kNO = L::kOutChunks;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base;  // D = 512: the resident Q
  const uint32_t sRing = base + L::kRingOffset;
  const uint32_t bars = base + L::kBarOffset;
  // Per slot one "full" barrier per item type (0: S operand, 1: V half; each
  // issuer takes one type, so it consumes every phase of the barriers it
  // waits on) and a shared "empty" one.
  auto bar_full = [&](int s, uint32_t is_v) { return bars + 8u * (is_v * L::kStages + s); };
  auto bar_empty = [&](int s) { return bars + 8u * (2 * L::kStages + s); };
  const uint32_t bar_s_full = bars + 24u * L::kStages;
  const uint32_t bar_s_free = bar_s_full + 8;
  const uint32_t bar_p_full = bar_s_free + 8;
  const uint32_t bar_p_free = bar_p_full + 8;
  const uint32_t bar_o_full = bar_p_free + 8;
  const uint32_t bar_drain = bar_o_full + 8;  // [issuer]
  const uint32_t bar_q_full = bar_drain + 16;  // D = 512: the resident Q has landed
  const uint32_t bar_q_empty = bar_q_full + 8;  // D = 512: the segment's last S has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOffset + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_full(s, 0u), 1);
      mbar_init(bar_full(s, 1u), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, 4 * 32);
    mbar_init(bar_p_full, 4 * 32);
    mbar_init(bar_p_free, 1);
    mbar_init(bar_o_full, 1);
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain + 8, 1);
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_empty, 1);
    *abort_flag = 0;
    mbar_init_fence();
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

  // Ring positions within a segment [b, e): the S operands of tile b come
  // first, then per j those of tile j+1 (if any) and V_j's halves.
  auto s_pos = [](int j, int b) { return j == b ? 0 : L::kItemsS + (j - b - 1) * (L::kItemsS + 2); };
  auto v_pos = [](int j, int b, int e) {
    return L::kItemsS + (j - b) * (L::kItemsS + 2) + (j + 1 < e ? L::kItemsS : 0);
  };
  auto seg_items = [](int b, int e) { return (e - b) * (L::kItemsS + 2); };

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
    if (warp == kLoadWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        const uint64_t keep = l2_policy_evict_last();  // Q, K, V: each re-read by several units
        int slot = 0;
        uint32_t ring_ph = 0, issued = 0, q_round = 0;
        uint32_t types = 0, sbits = 0, vbits = 0;  // per slot: latest item's type; next S / V full parity
        bool ok = true;
        SegCursor cur = first_cursor(p);
        Segment w;
        // One ring item: `npanels` boxes of `map` at (x0 + 64 pn, y, bh), panels `pstride` bytes apart.
        auto load_item = [&](const CUtensorMap* map, int x0, int y, int bh, int npanels, uint32_t pstride,
                             uint32_t is_v) -> bool {
          if (!wait_bounded(bar_empty(slot), ring_ph ^ 1u, wd, kSiteLoadRingEmpty, true, kNapNs)) return false;
          const uint32_t full = bar_full(slot, is_v);
          const uint32_t dst = sRing + static_cast<uint32_t>(slot * L::kSlotBytes);
          if (!(p.test_withhold && issued == 0)) {  // test hook: the first item never arrives
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(npanels) * pstride);
            for (int pn = 0; pn < npanels; ++pn)
              tma_load_3d_hint(dst + pn * pstride, map, full, x0 + 64 * pn, y, bh, keep);
          }
          types = (types & ~(1u << slot)) | (is_v << slot);
          if (is_v) vbits ^= 1u << slot; else sbits ^= 1u << slot;
          ++issued;
          if (++slot == L::kStages) {
            slot = 0;
            ring_ph ^= 1u;
          }
          return true;
        };
        while (ok && next_segment<kCausal, kR>(cur, w, p)) {
          const int bh = w.bh / kNO, oc = w.bh % kNO;
          if constexpr (L::kQRes) {
            // the unit's Q, once the previous segment's last S has read it
            if (q_round > 0 && !wait_bounded(bar_q_empty, (q_round - 1) & 1u, wd, kSiteLoadQEmpty, true, kNapNs)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar_q_full, L::kQBytes);
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d_hint(sQ + pn * kPanelBytes, &tmQ, bar_q_full, 64 * pn, w.q0, bh, keep);
            ++q_round;
          }
          auto load_s = [&](int j) -> bool {
            for (int c = 0; c < kNC && ok; ++c) {
              if (!L::kQRes && !load_item(&tmQ, 128 * c, w.q0, bh, 2, kPanelBytes, 0u)) return false;
              if (!load_item(&tmK, 128 * c, j * kKeys, bh, 2, kPanelBytes, 0u)) return false;
            }
            return true;
          };
          auto load_v = [&](int j) -> bool {
            for (int h = 0; h < 2; ++h)
              if (!load_item(&tmV, kDtileOutCols * oc, j * kKeys + 64 * h, bh, 4, L::kVPanelBytes, 1u)) return false;
            return true;
          };
          ok = load_s(w.kv_begin);
          for (int j = w.kv_begin; j < w.kv_end && ok; ++j) {
            if (j + 1 < w.kv_end) ok = load_s(j + 1);
            if (ok) ok = load_v(j);
          }
        }
        // Drain: every copy issued must have landed before the CTA may exit.
        const uint32_t first = issued > (uint32_t)L::kStages ? issued - L::kStages : 0u;
        for (uint32_t i = first; i < issued; ++i) {  // the latest item of each slot
          const int s = static_cast<int>(i % L::kStages);
          const uint32_t is_v = (types >> s) & 1u;
          const uint32_t par = (((is_v ? vbits : sbits) >> s) & 1u) ^ 1u;
          wait_bounded(bar_full(s, is_v), par, wd, kSiteDrain, false, kNapNs);
        }
        if (L::kQRes && q_round > 0) wait_bounded(bar_q_full, (q_round - 1) & 1u, wd, kSiteDrain, false, kNapNs);
      }
      __syncwarp();
    } else if (warp < kMmaWarp + kIssuers) {
      // ------------------------------------------------------ MMA issuers
      if (lane == 0) {
        const int me = warp - kMmaWarp;  // 0 issues every S, 1 every P.V
        constexpr uint32_t idesc_s = make_idesc_f16(kBf16, kKeys, false);
        constexpr uint32_t idesc_o = make_idesc_f16(kBf16, kDtileOutCols, true);
        constexpr uint32_t kHi = desc_hi_sw128(1024);  // 8-row (K-major) / 8-key (MN-major) groups 1 KB apart
        uint32_t bits[2] = {0u, 0u};  // per type, bit s: parity of the next use of slot s's full barrier
        auto take = [&](uint32_t idx, uint32_t is_v) -> int {
          const int s = static_cast<int>(idx % L::kStages);
          const uint32_t par = (bits[is_v] >> s) & 1u;
          bits[is_v] ^= 1u << s;
          return wait_bounded(bar_full(s, is_v), par, wd, kSiteMmaRingFull, true, kNapNs) ? s : -1;
        };
        uint32_t base_idx = 0;  // ring index of the current segment's first item
        bool ok = true;
        SegCursor cur = first_cursor(p);
        Segment w;
        if (me == 0) {
          // S(j) = sum_c Q_c K_{j,c}^T: 8 K-steps per chunk, A = Q chunk and
          // B = K chunk (both K-major, two 64-column panels). The S buffer
          // is overwritten only once the softmax has copied the previous S.
          uint32_t s_free_ph = 0, q_round = 0;
          bool s_out = false;
          while (ok && next_segment<kCausal, kR>(cur, w, p)) {
            const int b = w.kv_begin, e = w.kv_end;
            if (L::kQRes) {
              if (!wait_bounded(bar_q_full, q_round & 1u, wd, kSiteMmaQFull, true, kNapNs)) { ok = false; break; }
              ++q_round;
            }
            for (int j = b; j < e && ok; ++j) {
              const uint32_t i0 = base_idx + static_cast<uint32_t>(s_pos(j, b));
              for (int c = 0; c < kNC; ++c) {
                // A: the Q chunk (resident at D = 512, else the ring item
                // before K's); B: the K chunk
                const int slot_q = L::kQRes ? 0 : take(i0 + 2 * c, 0u);
                const int slot_k = slot_q < 0 ? -1 : take(L::kQRes ? i0 + c : i0 + 2 * c + 1, 0u);
                if (slot_k < 0) { ok = false; break; }
                if (c == 0 && s_out) {
                  if (!wait_bounded(bar_s_free, s_free_ph, wd, kSiteMmaSFree, true, kNapNs)) { ok = false; break; }
                  s_free_ph ^= 1u;
                }
                tc_fence_after_sync();
                const uint32_t qa =
                    L::kQRes ? desc_lo_sw128(sQ, 16) + static_cast<uint32_t>(c * (L::kSlotBytes >> 4))
                             : desc_lo_sw128(sRing, 16) + static_cast<uint32_t>(slot_q * (L::kSlotBytes >> 4));
                const uint32_t ka = desc_lo_sw128(sRing, 16) + static_cast<uint32_t>(slot_k * (L::kSlotBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
                  mma_ss_w(tmem, qa + off, kHi, ka + off, kHi, idesc_s, (c > 0 || kk > 0) ? 1u : 0u);
                }
                if (!L::kQRes) mma_commit(bar_empty(slot_q));
                mma_commit(bar_empty(slot_k));
              }
              if (!ok) break;
              mma_commit(bar_s_full);
              s_out = true;
              if (L::kQRes && j == e - 1) mma_commit(bar_q_empty);
            }
            base_idx += static_cast<uint32_t>(seg_items(b, e));
          }
        } else {
          // O_oc (+)= P(j) V_j[:, oc]: per V half (64 keys), 4 K-steps of 16
          // keys with A = P (tensor memory, 8 columns per K-step) and B = the
          // half (MN-major, N = 256 across four panels 8 KB apart).
          uint32_t p_full_ph = 0;
          const uint32_t tP = tmem + L::kColP;
          while (ok && next_segment<kCausal, kR>(cur, w, p)) {
            const int b = w.kv_begin, e = w.kv_end;
            for (int j = b; j < e && ok; ++j) {
              const uint32_t i0 = base_idx + static_cast<uint32_t>(v_pos(j, b, e));
              for (int h = 0; h < 2; ++h) {
                const int slot_v = take(i0 + h, 1u);
                if (slot_v < 0) { ok = false; break; }
                if (h == 0) {
                  if (!wait_bounded(bar_p_full, p_full_ph, wd, kSiteMmaPFull, true, kNapNs)) { ok = false; break; }
                  p_full_ph ^= 1u;
                }
                tc_fence_after_sync();
                const uint32_t va =
                    desc_lo_sw128(sRing, L::kVPanelBytes) + static_cast<uint32_t>(slot_v * (L::kSlotBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint32_t vb = va + static_cast<uint32_t>((kk * 16 * 128) >> 4);
                  mma_ts_w(tmem + L::kColO, tP + 8u * (4 * h + kk), vb, kHi, idesc_o,
                           (j > b || h > 0 || kk > 0) ? 1u : 0u);
                }
                if (h == 1) {
                  mma_commit(bar_p_free);
                  if (j == e - 1) mma_commit(bar_o_full);
                }
                mma_commit(bar_empty(slot_v));
              }
            }
            base_idx += static_cast<uint32_t>(seg_items(b, e));
          }
        }
        // Drain: all issued tensor-core work completes before TMEM is released.
        mma_commit(bar_drain + 8 * me);
        wait_bounded(bar_drain + 8 * me, 0u, wd, kSiteDrain, false, kNapNs);
      }
      __syncwarp();
    }
  } else if (warp < 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // -------------------------------------------------- softmax warpgroup
    const int wr = warp;            // TMEM lanes 32*wr..
    const int rr = wr * 32 + lane;  // row within the query tile
    const uint32_t lane_off = static_cast<uint32_t>(wr * 32) << 16;
    const uint32_t tS = tmem + lane_off;
    const uint32_t tO = tmem + lane_off + L::kColO;
    const uint32_t tP = tmem + lane_off + L::kColP;
    const float c = p.scale_log2;
    uint32_t s_phase = 0, o_phase = 0;
    uint32_t p_count = 0;  // P tiles published so far
    bool ok = true;
    SegCursor cur = first_cursor(p);
    Segment w;
    while (ok && next_segment<kCausal, kR>(cur, w, p)) {
      const int bh = w.bh / kNO, oc = w.bh % kNO;
      const int row = w.q0 + rr;
      const int limit = kCausal ? min(p.N, row + 1) : p.N;  // allowed keys: [0, limit)
      float m_raw = -CUDART_INF_F;  // running max of the raw scores seen so far
      float base = -CUDART_INF_F;   // exponent base (log2 units) that l and O are relative to
      float l = 0.f;    // sum of p (unrounded): LSE
      float l_o = 0.f;  // normaliser of O: l plus the 16-bit rounding of each tile's largest p
      for (int j = w.kv_begin; j < w.kv_end; ++j) {
        bool got = wait_bounded(bar_s_full, s_phase, wd, kSiteSoftmaxSFull);
        got = __all_sync(0xffffffffu, got);
        if (!got) { ok = false; break; }
        s_phase ^= 1u;
        tc_fence_after_sync();
        uint32_t sr[128];
        tmem_ld32x128_wait(tS, sr);
        // S is in registers: the issuer may compute the next scores.
        tc_fence_before_sync();
        mbar_arrive(bar_s_free);
        float s[128];
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i]);
        const int kv0 = j * kKeys;
        if (kv0 + kKeys > limit) {  // ragged tail and/or causal diagonal: mask disallowed keys
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (kv0 + i >= limit) s[i] = -CUDART_INF_F;
        }
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
        // The exponent base moves only when the max has grown by more than
        // kRescaleLog2 (or on the first tile with an allowed key); while a
        // row has seen no allowed key its base stays -inf and every p is 0.
        const float cand = m_raw * c;
        float alpha = 1.f;
        if (m_raw != -CUDART_INF_F && (base == -CUDART_INF_F || cand - base > kRescaleLog2)) {
          alpha = ex2_approx(base - cand);
          base = cand;
        }
        const float nb = (base == -CUDART_INF_F) ? 0.f : -base;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float x0, x1;
          ffma2_bcast(x0, x1, s[2 * i], s[2 * i + 1], c, nb);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          fadd2_acc(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], p0, p1);
          pk[i] = pack2(p0, p1, kBf16);
        }
        // The previous P.V must be complete before P is overwritten and
        // before O is rescaled.
        if (p_count > 0) {
          bool fr = wait_bounded(bar_p_free, (p_count - 1) & 1u, wd, kSiteSoftmaxPFree);
          fr = __all_sync(0xffffffffu, fr);
          if (!fr) { ok = false; break; }
          tc_fence_after_sync();
        }
        tmem_st32x32(tP, *reinterpret_cast<const uint32_t(*)[32]>(pk));
        tmem_st32x32(tP + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
        if (j > w.kv_begin && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < kDtileOutCols; cc += 32) {
            uint32_t o[32];
            tmem_ld32x32_wait(tO + cc, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32x32(tO + cc, o);
          }
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(bar_p_full);
        ++p_count;
        const float lt = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
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
      bool got = wait_bounded(bar_o_full, o_phase, wd, kSiteSoftmaxOFull);
      got = __all_sync(0xffffffffu, got);
      if (!got) break;
      o_phase ^= 1u;
      tc_fence_after_sync();
      const float inv = (l > 0.f) ? __frcp_rn(l_o) : 0.f;
      const bool live = row < p.N;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      ((static_cast<size_t>(bh) * p.N + (live ? row : 0)) * D + kDtileOutCols * oc) * 2;
#pragma unroll 1
      for (int cc = 0; cc < kDtileOutCols; cc += 32) {
        uint32_t o[32];
        tmem_ld32x32_wait(tO + cc, o);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv, kBf16);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 2);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (live && oc == 0) {
        p.lse[static_cast<size_t>(bh) * p.N + row] =
            (l > 0.f) ? (base + __log2f(l)) * 0.69314718055994530942f : CUDART_INF_F;
      }
      // O is read out; the next segment's first P.V may overwrite it once
      // this warpgroup publishes that segment's first P (ordered by p_full).
      tc_fence_before_sync();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd_dtile(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const CUtensorMap& /*o: stored directly*/, const Params& p, int grid,
                             cudaStream_t stream) {
  auto kern = fa2_fwd_dtile_kernel<D, kBf16, kCausal>;
  const int smem = DtileLayout<D>::kSmemBytes;
  if (p.stream_k) return cudaErrorInvalidValue;  // round schedule only
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
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, p);
}

}  // namespace fa2
