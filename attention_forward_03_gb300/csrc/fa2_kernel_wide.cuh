// FlashAttention-2 forward for GB300 (sm_103a) at head dimension 256.
//
// The operation is the one of fa2_kernel.cuh (the pages' FlashAttention-2
// forward: "FlashAttention-2 MMA 代码学习", steps 0-1; yangyitao.com CUDA
// book ch. 15, sections 15.1 and 15.3); the head dims above 128 are the ones
// the tiling_qk page's launcher adds. What changes at D = 256 is the budget:
// a 128-row fp32 O accumulator takes 256 of the 512 tensor-memory columns,
// so a CTA holds ONE 128-row query sub-tile per work unit instead of two.
// The other 256 columns hold two S buffers, used by alternate K/V tiles, so
// the next tile's scores are computed while the softmax works on the current
// ones (with two sub-tiles the same overlap came from the other sub-tile).
//
// Layout of one CTA (one per SM, persistent over work units of 128 rows of
// one (batch, head)):
//   warps 0-3  softmax warpgroup (thread = query row = TMEM lane)
//   warps 4-7  idle (they keep the launch's register split of the other
//              forward kernel; the softmax of one sub-tile is one warpgroup)
//   warp  8    S issuer: S(j) = Q K_j^T into S buffer n mod 2, n the number
//              of tiles the CTA has taken so far (16 K-steps); owns the TMEM
//              allocation
//   warp  9    P.V issuer: O (+)= P(j) V_j (8 K-steps of N = 256)
//   warp 10    TMA producer; warp 11 idle
// Tensor memory: [0,128) S buffer 0, [128,256) S buffer 1, [256,512) O.
// Shared memory: Q (64 KB, resident for the segment), P (32 KB, 16-bit,
// K-major), and a four-slot ring of K/V half tiles (32 KB each); all
// 128-byte swizzled in 64-element-wide panels, the layout the MMAs read. The
// ring's load order per segment [b, e) is K_b, then for each j: K_{j+1},
// V_j, each tile as two halves: K split along the head dimension (the first
// and last 8 K-steps of Q.K^T), V along the keys (the first and last 4
// K-steps of P.V). Each half is released as soon as the MMAs that read it
// have completed, so the next tile's first half loads while the second half
// is still in use (with whole-tile slots the loads of a type and its MMAs
// ran one after the other).
//
// Both schedules of the other forward kernel are supported (rounds of whole
// units; stream-K shares of K/V-tile steps with a cross-CTA (m, l) merge of
// fp32 partials), with one partial slot per CTA.
#pragma once
#include "fa2_fwd_common.cuh"

namespace fa2 {

template <int D>
struct WideLayout {
  static_assert(D == 256, "the wide kernel is built for head dimension 256");
  static constexpr int kPanels = D / 64;
  static constexpr int kTileBytes = kPanels * kPanelBytes;  // 128 rows x 256 (Q, K or V tile): 64 KB
  // The ring holds half tiles: a K half is 128 keys x 128 head-dim columns
  // (two 16 KB panels, the operand of 8 of the 16 K-steps of Q.K^T); a V half
  // is 64 keys x 256 columns (four 8 KB panels of 64 rows, the operand of 4
  // of the 8 K-steps of P.V).
  static constexpr int kHalfBytes = kTileBytes / 2;
  static constexpr int kVPanelBytes = kHalfBytes / kPanels;  // 64 rows x 64 elements
  static constexpr int kStages = 4;
  static constexpr int kQBytes = kTileBytes;
  static constexpr int kPOffset = kQBytes;
  static constexpr int kRingOffset = kPOffset + kPTileBytes;
  static constexpr int kBarOffset = kRingOffset + kStages * kHalfBytes;
  // barriers: q_full, q_empty, ring full (K tile)[S], ring full (V tile)[S], ring empty[S],
  // s_full[2], s_free[2], p_full, p_free, o_full, drain[2], part_done
  static constexpr int kNumBars = 2 + 3 * kStages + 2 + 2 + 3 + 2 + 1;
  static constexpr int kMiscOffset = kBarOffset + kNumBars * 8;
  static constexpr int kSmemBytes = kMiscOffset + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kColO = 2 * kKeys;                 // O at 256
  static_assert(kColO + D <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    fa2_fwd_wide_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Params p) {
  using L = WideLayout<D>;
  constexpr int kR = 1;  // sub-tiles per work unit
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
  // Per slot one "full" barrier per tile type (each issuer takes one type
  // and so consumes every phase of the barriers it waits on) and a shared
  // "empty" one.
  auto bar_full = [&](int s, uint32_t is_v) { return bars + 16 + 8u * (is_v * L::kStages + s); };
  auto bar_empty = [&](int s) { return bars + 16 + 8u * (2 * L::kStages + s); };
  const uint32_t bar_s_full0 = bars + 16 + 24u * L::kStages;  // [S buffer]
  const uint32_t bar_s_free0 = bar_s_full0 + 16;              // [S buffer]
  const uint32_t bar_p_full = bar_s_free0 + 16;
  const uint32_t bar_p_free = bar_p_full + 8;
  const uint32_t bar_o_full = bar_p_free + 8;
  const uint32_t bar_drain = bar_o_full + 8;                  // [issuer]
  const uint32_t bar_part = bar_drain + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOffset);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOffset + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_empty, 1);  // released by the S issuer after the segment's last S
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_full(s, 0u), 1);
      mbar_init(bar_full(s, 1u), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s_full0 + 8 * b, 1);
      mbar_init(bar_s_free0 + 8 * b, 4 * 32);
      mbar_init(bar_drain + 8 * b, 1);
    }
    mbar_init(bar_p_full, 4 * 32);
    mbar_init(bar_p_free, 1);
    mbar_init(bar_o_full, 1);
    mbar_init(bar_part, 4 * 32);
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

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
    if (warp == kLoadWarp) {
      // ---------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        const uint64_t keep = l2_policy_evict_last();          // K/V: re-read by every query tile of the head
        const uint64_t stream_once = l2_policy_evict_first();  // Q: read once
        int slot = 0;
        uint32_t ring_ph = 0, issued = 0, q_round = 0;
        uint32_t types = 0, kbits = 0, vbits = 0;  // per slot: latest tile's type; next K / V full parity
        bool ok = true;
        SegCursor cur = first_cursor(p);
        Segment w;
        // Loads both halves of tile j, each into the next ring slot.
        auto load_tile = [&](const CUtensorMap* map, int j, uint32_t is_v) -> bool {
          for (int h = 0; h < 2; ++h) {
            if (!wait_bounded(bar_empty(slot), ring_ph ^ 1u, wd, kSiteLoadRingEmpty, true, kNapNs)) return false;
            const uint32_t full = bar_full(slot, is_v);
            const uint32_t dst = sRing + static_cast<uint32_t>(slot * L::kHalfBytes);
            if (!(p.test_withhold && issued == 0)) {  // test hook: the first half tile never arrives
              mbar_arrive_expect_tx(full, L::kHalfBytes);
              if (is_v) {  // keys [64h, 64h+64) of the tile, four 64-column panels (the V map's box is 64 rows)
                for (int pn = 0; pn < L::kPanels; ++pn)
                  tma_load_3d_hint(dst + pn * L::kVPanelBytes, map, full, pn * 64, j * kKeys + 64 * h, w.bh, keep);
              } else {     // head-dim columns [128h, 128h+128): two panels of 128 keys
                for (int pn = 0; pn < 2; ++pn)
                  tma_load_3d_hint(dst + pn * kPanelBytes, map, full, 128 * h + 64 * pn, j * kKeys, w.bh, keep);
              }
            }
            types = (types & ~(1u << slot)) | (is_v << slot);
            if (is_v) vbits ^= 1u << slot; else kbits ^= 1u << slot;
            ++issued;
            if (++slot == L::kStages) {
              slot = 0;
              ring_ph ^= 1u;
            }
          }
          return true;
        };
        while (ok && next_segment<kCausal, kR>(cur, w, p)) {
          if (q_round > 0 && !wait_bounded(bar_q_empty, (q_round - 1) & 1u, wd, kSiteLoadQEmpty, true, kNapNs)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_q_full, L::kQBytes);
          for (int pn = 0; pn < L::kPanels; ++pn)
            tma_load_3d_hint(sQ + pn * kPanelBytes, &tmQ, bar_q_full, pn * 64, w.q0, w.bh, stream_once);
          ++q_round;
          ok = load_tile(&tmK, w.kv_begin, 0u);
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
        const int me = warp - kMmaWarp;  // 0 issues every S, 1 every P.V
        constexpr uint32_t idesc_s = make_idesc_f16(kBf16, kKeys, false);
        constexpr uint32_t idesc_o = make_idesc_f16(kBf16, D, true);
        constexpr uint32_t kHi = desc_hi_sw128(1024);  // 8-row (K-major) / 8-key (MN-major) groups 1 KB apart
        // Half h of S(buffer) = Q K^T: the 8 K-steps over head-dim columns
        // [128h, 128h+128), B from the K half tile in `slot`.
        auto issue_s_half = [&](int buf, int h, int slot) {
          const uint32_t qa = desc_lo_sw128(sQ, 16) + static_cast<uint32_t>((h * 2 * kPanelBytes) >> 4);
          const uint32_t ka = desc_lo_sw128(sRing, 16) + static_cast<uint32_t>(slot * (L::kHalfBytes >> 4));
          const uint32_t dt = tmem + static_cast<uint32_t>(buf * kKeys);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
            mma_ss_w(dt, qa + off, kHi, ka + off, kHi, idesc_s, (h > 0 || kk > 0) ? 1u : 0u);
          }
        };
        // Half h of O (+)= P V: keys [64h, 64h+64), 4 K-steps of 16 keys. P
        // is K-major in shared memory; V is MN-major, N = 256 across the half
        // tile's four 64-column panels 8 KB apart.
        auto issue_pv_half = [&](int h, int slot, bool acc) {
          const uint32_t pa = desc_lo_sw128(sP, 16) + static_cast<uint32_t>((h * kPanelBytes) >> 4);
          const uint32_t va = desc_lo_sw128(sRing, L::kVPanelBytes) + static_cast<uint32_t>(slot * (L::kHalfBytes >> 4));
          const uint32_t dt = tmem + L::kColO;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t vb = va + static_cast<uint32_t>((kk * 16 * 128) >> 4);
            const uint32_t po = static_cast<uint32_t>((kk * 32) >> 4);
            mma_ss_w(dt, pa + po, kHi, vb, kHi, idesc_o, (acc || h > 0 || kk > 0) ? 1u : 0u);
          }
        };
        // Ring index of half 0 of a tile: two halves per tile, in the load
        // order K_b, then for each j: K_{j+1}, V_j.
        auto k_index = [](int j, int b) { return 2 * (j == b ? 0 : 2 * (j - b) - 1); };
        auto v_index = [](int j, int b, int e) { return 2 * (j == e - 1 ? 2 * (j - b) + 1 : 2 * (j - b) + 2); };
        uint32_t bits[2] = {0u, 0u};
        auto take = [&](uint32_t idx, uint32_t is_v) -> int {
          const int s = static_cast<int>(idx % L::kStages);
          const uint32_t par = (bits[is_v] >> s) & 1u;
          bits[is_v] ^= 1u << s;
          return wait_bounded(bar_full(s, is_v), par, wd, kSiteMmaRingFull, true, kNapNs) ? s : -1;
        };
        uint32_t base_idx = 0;
        bool ok = true;
        SegCursor cur = first_cursor(p);
        Segment w;
        if (me == 0) {
          // S issuer: S(j) into buffer (tile count) mod 2 as soon as K_j has
          // landed and the softmax has loaded the buffer's previous S.
          // per S buffer (bit b): the parity of its next s_free phase, and
          // whether an S issued into it is still held by the softmax
          uint32_t q_round = 0, n_s = 0, s_free_ph = 0u, s_out = 0u;
          while (ok && next_segment<kCausal, kR>(cur, w, p)) {
            const int b = w.kv_begin, e = w.kv_end;
            if (!wait_bounded(bar_q_full, q_round & 1u, wd, kSiteMmaQFull, true, kNapNs)) { ok = false; break; }
            ++q_round;
            for (int j = b; j < e; ++j) {
              const int slot_k = take(base_idx + k_index(j, b), 0u);
              if (slot_k < 0) { ok = false; break; }
              const int buf = static_cast<int>(n_s & 1u);
              if ((s_out >> buf) & 1u) {
                if (!wait_bounded(bar_s_free0 + 8 * buf, (s_free_ph >> buf) & 1u, wd, kSiteMmaSFree, true, kNapNs)) {
                  ok = false;
                  break;
                }
                s_free_ph ^= 1u << buf;
              }
              tc_fence_after_sync();
              issue_s_half(buf, 0, slot_k);
              mma_commit(bar_empty(slot_k));
              const int slot_k1 = take(base_idx + k_index(j, b) + 1, 0u);
              if (slot_k1 < 0) { ok = false; break; }
              tc_fence_after_sync();
              issue_s_half(buf, 1, slot_k1);
              mma_commit(bar_s_full0 + 8 * buf);
              s_out |= 1u << buf;
              ++n_s;
              mma_commit(bar_empty(slot_k1));
              if (j == e - 1) mma_commit(bar_q_empty);
            }
            base_idx += 4u * static_cast<uint32_t>(e - b);
          }
        } else {
          // P.V issuer: O += P(j) V_j as soon as V_j has landed and the
          // softmax has published P(j).
          uint32_t p_full_ph = 0;
          while (ok && next_segment<kCausal, kR>(cur, w, p)) {
            const int b = w.kv_begin, e = w.kv_end;
            for (int j = b; j < e; ++j) {
              const int slot_v = take(base_idx + v_index(j, b, e), 1u);
              if (slot_v < 0) { ok = false; break; }
              if (!wait_bounded(bar_p_full, p_full_ph, wd, kSiteMmaPFull, true, kNapNs)) { ok = false; break; }
              p_full_ph ^= 1u;
              tc_fence_after_sync();
              issue_pv_half(0, slot_v, j > b);
              mma_commit(bar_empty(slot_v));
              const int slot_v1 = take(base_idx + v_index(j, b, e) + 1, 1u);
              if (slot_v1 < 0) { ok = false; break; }
              tc_fence_after_sync();
              issue_pv_half(1, slot_v1, true);
              mma_commit(bar_p_free);
              if (j == e - 1) mma_commit(bar_o_full);
              mma_commit(bar_empty(slot_v1));
            }
            base_idx += 4u * static_cast<uint32_t>(e - b);
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
    const int wr = warp;                     // TMEM lanes 32*wr..
    const int rr = wr * 32 + lane;           // row within the sub-tile
    const uint32_t lane_off = static_cast<uint32_t>(wr * 32) << 16;
    const uint32_t tS0 = tmem + lane_off;
    const uint32_t tO = tmem + lane_off + L::kColO;
    // this thread's P row: 128 bytes per 64 keys, 16-byte chunks placed by
    // the 128-byte swizzle (chunk c of row r at c ^ (r % 8))
    const uint32_t p_row = sP + static_cast<uint32_t>(rr * 128);
    const uint32_t p_xor = static_cast<uint32_t>(rr & 7);
    const float c = p.scale_log2;
    uint32_t s_phase = 0u, o_phase = 0, part_phase = 0;  // s_phase bit b: next s_full parity of buffer b
    uint32_t n_s = 0;      // S tiles taken so far (selects the buffer)
    uint32_t p_count = 0;  // P tiles published so far
    bool ok = true;
    SegCursor cur = first_cursor(p);
    Segment w;
    while (ok && next_segment<kCausal, kR>(cur, w, p)) {
      const int row = w.q0 + rr;
      const int limit = kCausal ? min(p.N, row + 1) : p.N;  // allowed keys: [0, limit)
      float m_raw = -CUDART_INF_F;
      float base = -CUDART_INF_F;
      float l = 0.f;
      float l_o = 0.f;
      for (int j = w.kv_begin; j < w.kv_end; ++j) {
        const int buf = static_cast<int>(n_s & 1u);
        ++n_s;
        bool got = wait_bounded(bar_s_full0 + 8 * buf, (s_phase >> buf) & 1u, wd, kSiteSoftmaxSFull);
        got = __all_sync(0xffffffffu, got);
        if (!got) { ok = false; break; }
        s_phase ^= 1u << buf;
        tc_fence_after_sync();
        uint32_t sr[128];
        tmem_ld32x128_wait(tS0 + static_cast<uint32_t>(buf * kKeys), sr);
        tc_fence_before_sync();
        mbar_arrive(bar_s_free0 + 8 * buf);
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
        // kRescaleLog2 (or on the first tile with an allowed key).
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
        // The previous P.V must be complete before its P buffer is
        // overwritten and before O is rescaled.
        if (p_count > 0) {
          bool fr = wait_bounded(bar_p_free, (p_count - 1) & 1u, wd, kSiteSoftmaxPFree);
          fr = __all_sync(0xffffffffu, fr);
          if (!fr) { ok = false; break; }
          tc_fence_after_sync();
        }
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint32_t addr = p_row + static_cast<uint32_t>((ch >> 3) * kPanelBytes) +
                                ((static_cast<uint32_t>(ch & 7) ^ p_xor) << 4);
          st_shared_v4(addr, pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        }
        if (j > w.kv_begin && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tmem_ld32x32_wait(tO + cc, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32x32(tO + cc, o);
          }
        }
        tmem_wait_st();
        fence_proxy_async_shared();
        tc_fence_before_sync();
        mbar_arrive(bar_p_full);
        ++p_count;
        const float lt = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        // O is normalised by l plus the rounding of each tile's largest p
        // (the 16-bit value P.V used), the LSE by the unrounded l.
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
      if (w.kv_begin > 0) {
        // Not the unit's first tiles: hand the unnormalised partial to the
        // owner through this CTA's workspace slot.
        const size_t slot = static_cast<size_t>(blockIdx.x);
        float* po = p.ws_o + slot * D * 128;
        float* ps = p.ws_stats + slot * 3 * 128;
#pragma unroll 1
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
        mbar_arrive(bar_part);
        if (rr < 32) {  // the first warp waits as a whole, so that it stays converged
          bool done = wait_bounded(bar_part, part_phase, wd, kSitePartialWrite);
          done = __all_sync(0xffffffffu, done);
          if (!done) break;
          if (rr == 0) store_release(p.ws_flags + slot, p.epoch);
        }
        part_phase ^= 1u;
        tc_fence_before_sync();
        continue;
      }
      // Owner (or whole unit): fold in the partials of the CTAs that took the
      // rest of this unit, then normalise and write O and LSE.
      float a_own = 1.f, nbase = base;
      int first_c = blockIdx.x + 1, last_c = blockIdx.x;
      if (p.stream_k && w.kv_end < w.nkv) {
        while (last_c + 1 < static_cast<int>(gridDim.x) && stream_k_begin(p, last_c + 1) < w.unit_end) ++last_c;
        bool fine = true;
        for (int cb = first_c; cb <= last_c && fine; ++cb)
          fine = wait_flag(p.ws_flags + static_cast<size_t>(cb), p.epoch, wd, kSitePartialFlag);
        fine = __all_sync(0xffffffffu, fine);
        if (!fine) break;
        for (int cb = first_c; cb <= last_c; ++cb)
          nbase = fmaxf(nbase, __ldcg(p.ws_stats + static_cast<size_t>(cb) * 3 * 128 + rr));
        a_own = ex2_approx(base - nbase);
        l *= a_own;
        l_o *= a_own;
        for (int cb = first_c; cb <= last_c; ++cb) {
          const float* ps = p.ws_stats + static_cast<size_t>(cb) * 3 * 128;
          const float a = ex2_approx(__ldcg(ps + rr) - nbase);
          l += a * __ldcg(ps + 128 + rr);
          l_o += a * __ldcg(ps + 256 + rr);
        }
        base = nbase;
      }
      const float inv = (l > 0.f) ? __frcp_rn(l_o) : 0.f;
      const bool live = row < p.N;
      uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                      (static_cast<size_t>(w.bh) * p.N + (live ? row : 0)) * (D * 2);
#pragma unroll 1
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t o[32];
        tmem_ld32x32_wait(tO + cc, o);
        float of[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) of[i] = __uint_as_float(o[i]) * a_own;
        for (int cb = first_c; cb <= last_c; ++cb) {
          const size_t slot = static_cast<size_t>(cb);
          const float a = ex2_approx(__ldcg(p.ws_stats + slot * 3 * 128 + rr) - nbase);
          const float* po = p.ws_o + slot * D * 128;
#pragma unroll
          for (int i = 0; i < 32; ++i) of[i] = fmaf(a, __ldcg(po + (cc + i) * 128 + rr), of[i]);
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2(of[2 * i] * inv, of[2 * i + 1] * inv, kBf16);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(orow + cc * 2);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (live) {
        p.lse[static_cast<size_t>(w.bh) * p.N + row] =
            (l > 0.f) ? (base + __log2f(l)) * 0.69314718055994530942f : CUDART_INF_F;
      }
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

// The stream-K schedule waits across CTAs, so it is launched cooperatively
// (the whole grid resident at once, or the launch fails).
template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd_wide(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& /*o: stored directly at this head dim*/, const Params& p, int grid,
                            cudaStream_t stream) {
  auto kern = fa2_fwd_wide_kernel<D, kBf16, kCausal>;
  const int smem = WideLayout<D>::kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, p);
}

}  // namespace fa2
