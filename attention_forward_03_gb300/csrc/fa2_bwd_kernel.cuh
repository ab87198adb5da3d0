// FlashAttention-2 backward for GB300 (sm_103a): persistent, warp-specialised,
// TMA-fed, tcgen05 tensor cores accumulating in tensor memory (TMEM).
//
// What it computes is the gradient of the forward pass for an upstream
// gradient dO, the way the yangyitao.com CUDA book, ch. 15, describes the
// FlashAttention-2 backward: only LSE = m + log l is kept from the forward
// (section 15.1, change 4) and S and P are recomputed from it; the outer loop
// runs over K/V tiles and the inner loop over query tiles, and dQ is
// accumulated across K/V tiles with atomic adds (the chapter's closing
// paragraph). Per K/V tile (128 keys) and query step i (64 rows):
//
//   S^T  = K Q_i^T            P^T  = 2^(S^T * scale*log2(e) - LSE_i*log2(e))
//   dP^T = V dO_i^T           dS^T = P^T * (dP^T - Delta_i),  Delta_i = <dO_i, O_i>
//   dV  += P^T dO_i           dK  += dS^T Q_i        (in TMEM for the whole tile)
//   dQ_i^T = K^T dS^T         added into an fp32 dQ accumulator in global memory
//                             (a TMA bulk reduce-add per warpgroup and step)
//
// and at the end of the tile dK *= scale; dQ = scale * accumulator is
// converted to the dtype by a separate elementwise kernel.
//
// Layout of one CTA (one per SM, persistent over work units = K/V tiles, or
// over segments of them, see below):
//   warps 0-7  two compute warpgroups; thread = key row = TMEM lane, warpgroup
//              g takes query columns [32g, 32g+32) of every step (and, in
//              the epilogue, the dK / dV row's 32-column chunks: the first
//              half of them, rounded up, for g = 0, the rest for g = 1)
//   warp  8    tcgen05 MMA issuer (one thread) of the score products S^T,
//              dP^T; owns the TMEM allocation
//   warp  9    tcgen05 MMA issuer (one thread) of the gradient products dV,
//              dK, dQ^T. Both issuers poll their barriers without sleeping;
//              with that, two issuers also pay on causal launches (long
//              causal rows +19.5 %, B4 H16 N4096 causal +13.5 % over one
//              issuer that computed the next step's scores before the
//              current step's gradients), where with sleeping waits they had
//              measured 1 % slower.
//   warp  10   TMA producer (one thread)
//   warp  11   (D = 96, 128) two threads that add the compute warpgroups'
//              staged dQ^T rows into the accumulator with TMA reduce-adds
// Head dims 32 and 96 run in the tiles of 64 and 128 (Dp below): their
// columns past D arrive as zeros from the copy engine, so they add nothing.
// Tensor memory (fp32 columns x 128 lanes):
//   [0, D)          dV accumulator        [Dp, Dp+D)     dK accumulator
//   [2Dp, 2Dp+SR)   S^T of the step       [2Dp+SR, 2Dp+2SR) dP^T of the step
//   [2Dp+2SR, ...)  Dp = 128: dQ^T of the step (lane = head-dim index; the
//                   MMA runs with M = 128 and the lanes from D on are
//                   discarded), then P^T and dS^T of the step (SR/2 packed
//                   columns each); Dp = 64: dQ of the step, untransposed
//                   (lane = query row, 64 columns), then P^T (64 packed
//                   columns)
// Shared memory (128-byte swizzled, 64-element panels): K and V of the tile
// (resident for the unit), a ring of query steps (Q_i, dO_i, and their
// -LSE*log2(e) and Delta values), the 16-bit dS^T of the step (written by
// the compute threads, read by the tensor core), and an fp32
// staging tile for dQ that TMA reduce-adds into the global accumulator: at
// Dp = 128 SR rows x D, 32 rows per compute warpgroup and reduce-add; at
// Dp = 64 SR rows x 32 columns per warpgroup, 128-byte swizzled.
//
// Schedules: whole units dealt to the CTAs in rounds (zig-zag when causal),
// or stream-K: every CTA takes an equal share of all query steps, so a unit
// may be cut between consecutive CTAs; the CTA holding a unit's first steps
// (for which it is the last segment of its share) adds the fp32 partial dV,
// dK that the following CTAs wrote (each as the first segment of its share)
// before it writes dV and dK. dQ needs no merge: every step adds into the
// accumulator whichever CTA runs it.
//
// Pipelining: the issuer computes S^T, dP^T of step i+1 as soon as the
// compute threads have loaded those of step i into registers, so the tensor
// core works on step i+1 while P^T and dS^T of step i are formed; the
// compute threads read dQ^T of step i-1 after publishing step i.
#pragma once
#include "fa2_kernel.cuh"

namespace fa2 {

// 11 warps, and at D = 96, 128 a twelfth (see kBwdDqWarp)
constexpr int bwd_threads(int d) { return d > 64 ? 384 : 352; }
constexpr int kBwdMmaWarp = 8;      // MMA issuer (all products, or S^T / dP^T); owns the TMEM allocation
constexpr int kBwdGradWarp = 9;     // second MMA issuer (dV, dK, dQ^T)
constexpr int kBwdLoadWarp = 10;
// D = 96, 128: two lanes of this warp add the compute warpgroups' staged
// dQ^T rows into the accumulator (a TMA reduce-add per 32 rows) and give
// the rows back once the copy engine has read them. At D <= 64 each
// warpgroup's first thread does it (measured: the extra warp is +1 to +6 %
// at D = 96, 128 and -2 % at D = 64).
constexpr int kBwdDqWarp = 11;
constexpr int kBwdComputeThreads = 256;

enum : int {
  kSiteBwdKvEmpty = 21,
  kSiteBwdStageEmpty = 22,
  kSiteBwdKvFull = 23,
  kSiteBwdStageFull = 24,
  kSiteBwdSFree = 25,
  kSiteBwdPFull = 26,
  kSiteBwdAccFree = 27,
  kSiteBwdDqFree = 28,
  kSiteBwdSFull = 29,
  kSiteBwdPFree = 30,
  kSiteBwdDqFull = 31,
  kSiteBwdAccFull = 32,
  kSiteBwdDrain = 33,
  kSiteBwdDqsFree = 34,
  kSiteBwdDqsReady = 35,
  kSiteBwdPartWrite = 36,
  kSiteBwdPartFlag = 37,
};

template <int D>
struct BwdLayout {
  static_assert(bwd_head_dim_ok(D), "head dimension");
  // D = 32 and 96 use the tiles of 64 and 128: their columns past D read as
  // zeros (the copy engine's out-of-bounds fill) and add nothing
  static constexpr int kPanels = (D + 63) / 64;
  static constexpr int kDp = kPanels * 64;                    // padded head dimension
  // N of the dV, dK products (the O columns accumulated). At D = 32 it stays
  // 64: a 32-wide MN-major operand would cover half of a 128-byte swizzle
  // row, a form the operand layouts do not describe.
  static constexpr int kNacc = (D == 32) ? 64 : D;
  // Query rows per step (SR): 128 where the tensor memory has room for
  // 128-column S^T, dP^T and dQ^T next to dV and dK (Dp = 64: 64 + 64 + 3 x
  // 128 = 512 columns), else 64. Each compute warpgroup takes SR/2 query
  // columns of a step, in halves of 32.
  static constexpr int kSR = bwd_step_rows(D);
  static constexpr int kR = kBwdKeys / kSR;                   // steps per 128 query rows
  static constexpr int kCW = kSR / 2;                         // query columns per warpgroup
  static constexpr int kHalves = kCW / 32;
  static constexpr int kKVBytes = kPanels * kPanelBytes;      // K or V tile: 128 rows x Dp
  static constexpr int kQPanelBytes = kSR * 128;              // SR rows x 64 16-bit elements
  static constexpr int kQBytes = kPanels * kQPanelBytes;      // Q or dO step: SR rows x Dp
  static constexpr int kPTileBytes = (kSR / 64) * kPanelBytes;  // dS^T: 128 keys x SR queries
  static constexpr int kStatBytes = 2 * kSR * 4;              // -LSE*log2(e) and Delta of one step
  static constexpr int kStages = (kSR == 128) ? 3 : (kPanels == 2 ? 3 : 6);
  // Epilogue: a key row's D columns in chunks of 32, the first kChunksWg for
  // compute warpgroup 0 and the rest for warpgroup 1.
  static constexpr int kChunks = D / 32;
  static constexpr int kChunksWg = (kChunks + 1) / 2;
  static_assert(32 * 2 * kChunksWg <= kDp, "epilogue chunks stay inside the padded dV / dK columns");
  static constexpr int kStageBytes = 2 * kQBytes;             // Q then dO
  static constexpr int kK = 0;
  static constexpr int kV = kKVBytes;
  static constexpr int kRing = 2 * kKVBytes;
  static constexpr int kDS = kRing + kStages * kStageBytes;  // dS^T (P^T lives in tensor memory)
  static constexpr int kDQS = kDS + kPTileBytes;              // dQ staging: SR rows x D fp32
  static constexpr int kStats = kDQS + kSR * D * 4;
  static constexpr int kBars = kStats + kStages * kStatBytes;
  // kv_full, kv_empty, stage_full[S], stage_empty[S], s_full, s_free, p_full,
  // p_free, dq_full, dq_free, acc_full, acc_free, drain, dqs_ready[2], dqs_free[2], drain2, part_done
  static constexpr int kNumBars = 2 + 2 * kStages + 15;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kSmemBytes = kMisc + 16 + 1024;  // + slack for 1 KB alignment
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = kDp;
  static constexpr uint32_t kColS = 2 * kDp;
  static constexpr uint32_t kColDP = 2 * kDp + kSR;
  static constexpr uint32_t kColDQ = 2 * kDp + 2 * kSR;
  static_assert(kColDQ + kSR <= kTmemCols, "TMEM budget");
  // With 64-row steps (Dp = 128) the 64 columns past dQ^T hold the step's
  // P^T and dS^T as packed 16-bit pairs: the A operands of dV += P^T dO and
  // dK += dS^T Q then come from tensor memory (the faster form of the MMA,
  // and no shared-memory operand reads for them). dS^T also goes to shared
  // memory, where dQ^T = K^T dS^T reads it as its B operand. Measured +1.8 %
  // (target) and +2.5 % (B4 H16 N8192 D128) non-causal, and, with two
  // non-sleeping issuers, +1 to +2 % on causal launches too (with one issuer
  // it had been -2.4 % on long causal rows).
  static constexpr bool kGradATmem = (kSR == 64);
  // At Dp = 64 the step's dQ is computed untransposed, dQ = dS K (M = the
  // 128 query rows, N = 64): the rows fill all 128 TMEM lanes, so every
  // compute warp stages a share (32 columns per warpgroup, 16-byte stores
  // into 128-byte-swizzled rows that one TMA reduce-add per warpgroup reads),
  // and an N = 64 product takes 8 x ~47 cycles against 8 x 64 for dQ^T's
  // N = 128. dQ^T (lanes = head-dim index) puts only D of the 128 lanes to
  // use, so half the warps staged everything.
  static constexpr bool kDqRows = (kDp == 64);
  // At Dp = 64 the untransposed dQ takes 64 of its region's 128 columns;
  // the other 64 hold the step's P^T (128 query columns as packed pairs), so
  // dV += P^T dO reads A from tensor memory at every head dimension (at Dp =
  // 64 measured +5 to +11 % over P^T in shared memory, bit-identical). dS^T
  // stays in shared memory only there: dK and dQ both read it from there.
  static constexpr uint32_t kColPT = kDqRows ? kColDQ + kDp : kColDQ + kSR;
  static constexpr uint32_t kColDST = kColPT + kSR / 2;
  static_assert(kGradATmem || kDqRows, "P^T has tensor-memory columns at every step height");
  static_assert(kColPT + kSR / 2 <= kTmemCols, "TMEM budget");
  static_assert(!kGradATmem || kColDST + kSR / 2 <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kRing % 1024 == 0 && kDS % 1024 == 0, "swizzled tiles need 1 KB alignment");
};

// Work unit u -> (head, K/V tile). Non-causal: the tiles of a head are
// consecutive (its Q and dO stay hot in L2). Causal: the tiles with the most
// query steps (lowest index) first, over all heads.
template <bool kCausal>
__device__ __forceinline__ void bwd_unit(int u, const BwdParams& p, int& bh, int& kv) {
  if (kCausal) {
    kv = u / p.BH;
    bh = u % p.BH;
  } else {
    bh = u / p.nkv;
    kv = u % p.nkv;
  }
}

// Query steps [first, nq) that see keys of tile kv (kR steps per 128 rows).
template <bool kCausal, int kR>
__device__ __forceinline__ int bwd_first_step(int kv) {
  return kCausal ? kv * kR : 0;
}

// Unit of this CTA in round r (zig-zag when causal, as in the forward).
template <bool kCausal>
__device__ __forceinline__ int bwd_round_unit(int r) {
  const int g = gridDim.x, b = blockIdx.x;
  return r * g + ((kCausal && (r & 1)) ? (g - 1 - b) : b);
}

// A segment: query steps [i_begin, i_end) of unit (bh, kv). With the round
// schedule every segment is a whole unit; with stream-K a unit may be cut
// between consecutive CTAs.
struct BwdSegment {
  int bh, kv;
  int i_begin, i_end;
  long long unit_end;  // stream-K: global step one past the unit's last step
};

struct BwdCursor {
  int round;
  long long step, end;
};

__device__ __forceinline__ long long bwd_share_begin(const BwdParams& p, int b) {
  return p.total_steps * b / gridDim.x;
}

__device__ __forceinline__ BwdCursor bwd_first_cursor(const BwdParams& p) {
  BwdCursor c;
  c.round = 0;
  c.step = p.stream_k ? bwd_share_begin(p, blockIdx.x) : 0;
  c.end = p.stream_k ? bwd_share_begin(p, blockIdx.x + 1) : 0;
  return c;
}

// First step of causal unit kv within its head: units k < kv have
// nq - kR*k steps each, kv*nq - kR*kv*(kv-1)/2 in all.
template <int kR>
__device__ __forceinline__ long long bwd_causal_start(int kv, int nq) {
  return static_cast<long long>(kv) * nq - static_cast<long long>(kR) * kv * (kv - 1) / 2;
}

// Next segment of this CTA. Every role walks the same sequence.
template <bool kCausal, int kR>
__device__ __forceinline__ bool bwd_next_segment(BwdCursor& c, BwdSegment& s, const BwdParams& p) {
  if (!p.stream_k) {
    const int u = bwd_round_unit<kCausal>(c.round++);
    if (u >= p.num_units) return false;
    bwd_unit<kCausal>(u, p, s.bh, s.kv);
    s.i_begin = bwd_first_step<kCausal, kR>(s.kv);
    s.i_end = p.nq;
    s.unit_end = 0;
    return true;
  }
  if (c.step >= c.end) return false;
  // Units in order: heads, then K/V tiles ascending.
  const long long bh = c.step / p.steps_per_head;
  const long long r = c.step - bh * p.steps_per_head;
  int kv;
  long long start;
  if (kCausal) {
    // the root of (kR/2) kv^2 - (nq + kR/2) kv + r = 0, then corrected
    const float a = static_cast<float>(p.nq) + 0.5f * kR;
    kv = static_cast<int>((a - sqrtf(fmaxf(a * a - 2.f * kR * static_cast<float>(r), 0.f))) / kR);
    kv = min(max(kv, 0), p.nkv - 1);
    while (kv > 0 && bwd_causal_start<kR>(kv, p.nq) > r) --kv;
    while (kv + 1 < p.nkv && bwd_causal_start<kR>(kv + 1, p.nq) <= r) ++kv;
    start = bwd_causal_start<kR>(kv, p.nq);
  } else {
    kv = static_cast<int>(r / p.nq);
    start = static_cast<long long>(kv) * p.nq;
  }
  const int first = bwd_first_step<kCausal, kR>(kv);
  s.bh = static_cast<int>(bh);
  s.kv = kv;
  s.i_begin = first + static_cast<int>(r - start);
  const long long left = c.end - c.step;
  s.i_end = static_cast<int>(min(static_cast<long long>(p.nq), s.i_begin + left));
  s.unit_end = c.step - (s.i_begin - first) + (p.nq - first);
  c.step += s.i_end - s.i_begin;
  return true;
}

template <int D, bool kBf16, bool kCausal>
__global__ void __launch_bounds__(bwd_threads(D), 1)
    fa2_bwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                   const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using L = BwdLayout<D>;
  constexpr bool kTwoIssuers = true;
  constexpr bool kATmem = L::kGradATmem;  // dS^T in TMEM for dK (P^T is there for dV at every D)
  constexpr bool kDqWarp = bwd_threads(D) > 352;  // staged dQ^T added by warp kBwdDqWarp
  constexpr uint32_t kReaders = kTwoIssuers ? 2 : 1;  // issuer threads reading a ring slot and K/V
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sK = base + L::kK;
  const uint32_t sV = base + L::kV;
  const uint32_t sRing = base + L::kRing;
  const uint32_t sDS = base + L::kDS;
  const uint32_t sStats = base + L::kStats;
  const float* stats = reinterpret_cast<const float*>(smem + L::kStats);
  const uint32_t bars = base + L::kBars;
  const uint32_t bar_kv_full = bars;
  const uint32_t bar_kv_empty = bars + 8;
  auto bar_stage_full = [&](int s) { return bars + 16 + 8u * s; };
  auto bar_stage_empty = [&](int s) { return bars + 16 + 8u * (L::kStages + s); };
  const uint32_t bar_s_full = bars + 16 + 16u * L::kStages;  // S^T, dP^T of a step in TMEM
  const uint32_t bar_s_free = bar_s_full + 8;                 // ... loaded by the compute threads
  const uint32_t bar_p_full = bar_s_full + 16;                // P^T, dS^T of a step written
  const uint32_t bar_p_free = bar_s_full + 24;                // ... read by the tensor core
  const uint32_t bar_dq_full = bar_s_full + 32;               // dQ^T of a step in TMEM
  const uint32_t bar_dq_free = bar_s_full + 40;               // ... loaded by the compute threads
  const uint32_t bar_acc_full = bar_s_full + 48;              // dV, dK of a unit complete
  const uint32_t bar_acc_free = bar_s_full + 56;              // ... loaded by the compute threads
  const uint32_t bar_drain = bar_s_full + 64;
  // per compute warpgroup: its 32 staged dQ rows are written / have been read by TMA
  auto bar_dqs_ready = [&](int w) { return bar_s_full + 72 + 8u * w; };
  auto bar_dqs_free = [&](int w) { return bar_s_full + 88 + 8u * w; };
  const uint32_t bar_drain2 = bar_s_full + 104;                // second issuer
  const uint32_t bar_part = bar_s_full + 112;                  // stream-K partial dV, dK written
  const uint32_t sDQS = base + L::kDQS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv_full, 1);
    mbar_init(bar_kv_empty, kReaders);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar_stage_full(s), 1);
      mbar_init(bar_stage_empty(s), kReaders);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, kBwdComputeThreads);
    mbar_init(bar_p_full, kBwdComputeThreads);
    mbar_init(bar_p_free, 1);
    mbar_init(bar_dq_full, 1);
    mbar_init(bar_dq_free, kBwdComputeThreads);
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_acc_free, kBwdComputeThreads);
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain2, 1);
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar_dqs_ready(w), 128);
      mbar_init(bar_dqs_free(w), 1);
    }
    mbar_init(bar_part, kBwdComputeThreads);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == kBwdMmaWarp) {
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

  if (warp == kBwdLoadWarp) {
    // ------------------------------------------------------------ producer
    // Per unit: K and V of the tile once, then every query step (Q_i, dO_i
    // and their 64 -LSE*log2(e) / Delta values) through the ring.
    if (lane == 0) {
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmDO);
      tma_prefetch_map(&tmDQ);
      const uint64_t once = l2_policy_evict_first();  // K, V: read by one unit
      const uint64_t keep = l2_policy_evict_last();   // Q, dO: read by every K/V tile of the head
      int slot = 0;
      uint32_t ph = 0, units = 0, loads = 0;
      bool ok = true;
      BwdCursor cur = bwd_first_cursor(p);
      BwdSegment sg;
      while (ok && bwd_next_segment<kCausal, L::kR>(cur, sg, p)) {
        const int bh = sg.bh, kv = sg.kv;
        if (units > 0 && !wait_bounded(bar_kv_empty, (units - 1) & 1u, wd, kSiteBwdKvEmpty, true, kNapNs)) {
          ok = false;
          break;
        }
        if (!(p.test_withhold && units == 0)) {  // test hook: the first K/V tile never arrives
          mbar_arrive_expect_tx(bar_kv_full, 2 * L::kKVBytes);
          for (int pn = 0; pn < L::kPanels; ++pn) {
            tma_load_3d_hint(sK + pn * kPanelBytes, &tmK, bar_kv_full, pn * 64, kv * kBwdKeys, bh, once);
            tma_load_3d_hint(sV + pn * kPanelBytes, &tmV, bar_kv_full, pn * 64, kv * kBwdKeys, bh, once);
          }
        }
        ++units;
        for (int i = sg.i_begin; i < sg.i_end; ++i) {
          if (!wait_bounded(bar_stage_empty(slot), ph ^ 1u, wd, kSiteBwdStageEmpty, true, kNapNs)) {
            ok = false;
            break;
          }
          const uint32_t full = bar_stage_full(slot);
          const uint32_t st = sRing + static_cast<uint32_t>(slot * L::kStageBytes);
          mbar_arrive_expect_tx(full, L::kStageBytes + L::kStatBytes);
          for (int pn = 0; pn < L::kPanels; ++pn) {
            tma_load_3d_hint(st + pn * L::kQPanelBytes, &tmQ, full, pn * 64, i * L::kSR, bh, keep);
            tma_load_3d_hint(st + L::kQBytes + pn * L::kQPanelBytes, &tmDO, full, pn * 64, i * L::kSR, bh, keep);
          }
          const size_t off = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(i) * L::kSR;
          const uint32_t sst = sStats + static_cast<uint32_t>(slot * L::kStatBytes);
          bulk_load(sst, p.neg_lse2 + off, L::kSR * 4, full);
          bulk_load(sst + L::kSR * 4, p.delta + off, L::kSR * 4, full);
          ++loads;
          if (++slot == L::kStages) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      // Drain: every copy issued must have landed before the CTA may exit.
      const uint32_t first = loads > static_cast<uint32_t>(L::kStages) ? loads - L::kStages : 0u;
      for (uint32_t x = first; x < loads; ++x)
        wait_bounded(bar_stage_full(static_cast<int>(x % L::kStages)), (x / L::kStages) & 1u, wd, kSiteBwdDrain,
                     false, kNapNs);
      if (units > 0) wait_bounded(bar_kv_full, (units - 1) & 1u, wd, kSiteBwdDrain, false, kNapNs);
    }
    __syncwarp();
  } else if (warp == kBwdMmaWarp || (kTwoIssuers && warp == kBwdGradWarp)) {
    // The issuers poll their barriers without sleeping: each step is a chain
    // of hand-offs between them and the compute warpgroups, and a sleeping
    // waiter wakes late (measured: 0 to +2.3 % across the backward workloads).
    // --------------------------------------------------------- MMA issuers
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_f16(kBf16, L::kSR, false);              // S^T, dP^T: N = SR
      constexpr uint32_t idesc_acc = make_idesc_f16(kBf16, L::kNacc, true);           // dV, dK: N = D (64 at D = 32)
      constexpr uint32_t idesc_dq = make_idesc_f16_ab(kBf16, L::kSR, true, true);     // dQ^T: N = SR
      constexpr uint32_t idesc_dqr = make_idesc_f16_ab(kBf16, L::kNacc, true, true);  // dQ (Dp = 64): N = 64
      constexpr uint32_t kHi = desc_hi_sw128(1024);  // 8-row (K-major) / 8-row-of-K (MN-major) groups 1 KB apart
      // S^T = K Q_i^T and dP^T = V dO_i^T: A = K / V (K-major, 128-row
      // panels), B = Q_i / dO_i (K-major, SR-row panels), N = SR, D/16 steps.
      auto issue_sdp = [&](int slot) {
        const uint32_t st = sRing + static_cast<uint32_t>(slot * L::kStageBytes);
        const uint32_t k_lo = desc_lo_sw128(sK, 16), v_lo = desc_lo_sw128(sV, 16);
        const uint32_t q_lo = desc_lo_sw128(st, 16), do_lo = desc_lo_sw128(st + L::kQBytes, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
          const uint32_t b = static_cast<uint32_t>(((kk >> 2) * L::kQPanelBytes + (kk & 3) * 32) >> 4);
          mma_ss_w(tmem + L::kColS, k_lo + a, kHi, q_lo + b, kHi, idesc_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
          const uint32_t b = static_cast<uint32_t>(((kk >> 2) * L::kQPanelBytes + (kk & 3) * 32) >> 4);
          mma_ss_w(tmem + L::kColDP, v_lo + a, kHi, do_lo + b, kHi, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      // dV += P^T dO_i and dK += dS^T Q_i: A = P^T from tensor memory, dS^T
      // from tensor memory (Dp = 128) or shared memory (K-major, panels of 64
      // query columns 16 KB apart), B = dO_i / Q_i (MN-major: rows are the
      // contraction index, 64-column panels of SR rows), SR/16 steps of 16
      // rows.
      auto issue_grads = [&](int slot, bool acc) {
        const uint32_t st = sRing + static_cast<uint32_t>(slot * L::kStageBytes);
        const uint32_t ds_lo = desc_lo_sw128(sDS, 16);
        const uint32_t q_mn = desc_lo_sw128(st, L::kQPanelBytes);
        const uint32_t do_mn = desc_lo_sw128(st + L::kQBytes, L::kQPanelBytes);
#pragma unroll
        for (int kk = 0; kk < L::kSR / 16; ++kk) {
          const uint32_t b = static_cast<uint32_t>((kk * 16 * 128) >> 4);
          const uint32_t acc_kk = (acc || kk > 0) ? 1u : 0u;
          // A = P^T in TMEM: 16 query columns = 8 packed columns per K-step
          mma_ts_w(tmem + L::kColDV, tmem + L::kColPT + 8u * kk, do_mn + b, kHi, idesc_acc, acc_kk);
        }
#pragma unroll
        for (int kk = 0; kk < L::kSR / 16; ++kk) {
          const uint32_t a = static_cast<uint32_t>(((kk >> 2) * kPanelBytes + (kk & 3) * 32) >> 4);
          const uint32_t b = static_cast<uint32_t>((kk * 16 * 128) >> 4);
          const uint32_t acc_kk = (acc || kk > 0) ? 1u : 0u;
          if constexpr (kATmem)
            mma_ts_w(tmem + L::kColDK, tmem + L::kColDST + 8u * kk, q_mn + b, kHi, idesc_acc, acc_kk);
          else
            mma_ss_w(tmem + L::kColDK, ds_lo + a, kHi, q_mn + b, kHi, idesc_acc, acc_kk);
        }
      };
      // dQ_i^T = K^T dS^T: A = K read MN-major (M = head-dim index, two
      // 64-row M panels 16 KB apart; at D = 64 the second panel is the V
      // tile and its rows are discarded), B = dS^T MN-major (N = SR query
      // columns, panels of 64 16 KB apart), 8 steps of 16 keys.
      auto issue_dq = [&]() {
        const uint32_t kt_lo = desc_lo_sw128(sK, kPanelBytes);
        const uint32_t ds_mn = desc_lo_sw128(sDS, kPanelBytes);
#pragma unroll
        for (int kk = 0; kk < kBwdKeys / 16; ++kk) {
          const uint32_t off = static_cast<uint32_t>((kk * 16 * 128) >> 4);
          if constexpr (L::kDqRows)  // dQ = dS K: A = dS^T's rows read MN-major (M = queries), B = K MN-major
            mma_ss_w(tmem + L::kColDQ, ds_mn + off, kHi, kt_lo + off, kHi, idesc_dqr, kk > 0 ? 1u : 0u);
          else
            mma_ss_w(tmem + L::kColDQ, kt_lo + off, kHi, ds_mn + off, kHi, idesc_dq, kk > 0 ? 1u : 0u);
        }
      };

      if constexpr (kTwoIssuers) {
        // Two issuers walk the same step sequence: warp 8 the scores, warp 9
        // the gradients. Each releases a ring slot and K/V after its own
        // MMAs that read them (a commit tracks only its thread's MMAs).
        const bool scores = warp == kBwdMmaWarp;
        int slot = 0;
        uint32_t ph = 0;
        uint32_t g = 0;
        uint32_t units = 0;
        bool ok = true;
        BwdCursor cur = bwd_first_cursor(p);
        BwdSegment sg;
        while (ok && bwd_next_segment<kCausal, L::kR>(cur, sg, p)) {
          const int n_steps = sg.i_end - sg.i_begin;
          if (!wait_bounded(bar_kv_full, units & 1u, wd, kSiteBwdKvFull, true, 0u)) {
            ok = false;
            break;
          }
          for (int t = 0; t < n_steps; ++t, ++g) {
            if (!wait_bounded(bar_stage_full(slot), ph, wd, kSiteBwdStageFull, true, 0u)) {
              ok = false;
              break;
            }
            if (scores) {
              if (g > 0 && !wait_bounded(bar_s_free, (g - 1) & 1u, wd, kSiteBwdSFree, true, 0u)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              issue_sdp(slot);
              mma_commit(bar_s_full);
              mma_commit(bar_stage_empty(slot));
            } else {
              if (!wait_bounded(bar_p_full, g & 1u, wd, kSiteBwdPFull, true, 0u)) {
                ok = false;
                break;
              }
              if (t == 0 && units > 0 &&
                  !wait_bounded(bar_acc_free, (units - 1) & 1u, wd, kSiteBwdAccFree, true, 0u)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              issue_grads(slot, t > 0);
              mma_commit(bar_stage_empty(slot));
              if (g > 0 && !wait_bounded(bar_dq_free, (g - 1) & 1u, wd, kSiteBwdDqFree, true, 0u)) {
                ok = false;
                break;
              }
              tc_fence_after_sync();
              issue_dq();
              mma_commit(bar_p_free);
              mma_commit(bar_dq_full);
            }
            if (++slot == L::kStages) {
              slot = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          if (!scores) mma_commit(bar_acc_full);
          mma_commit(bar_kv_empty);
          ++units;
        }
      } else {
        int slot = 0;
        uint32_t ph = 0;
        uint32_t g = 0;      // global query-step counter of this CTA
        uint32_t units = 0;
        bool ok = true;
        // Takes the next ring slot (Q_i, dO_i loaded) and, once the compute
        // threads hold the previous step's S^T / dP^T, issues this step's.
        auto start_step = [&](uint32_t step) -> int {
          const int s = slot;
          if (!wait_bounded(bar_stage_full(s), ph, wd, kSiteBwdStageFull, true, 0u)) return -1;
          if (step > 0 && !wait_bounded(bar_s_free, (step - 1) & 1u, wd, kSiteBwdSFree, true, 0u)) return -1;
          tc_fence_after_sync();
          issue_sdp(s);
          mma_commit(bar_s_full);
          if (++slot == L::kStages) {
            slot = 0;
            ph ^= 1u;
          }
          return s;
        };
        BwdCursor wcur = bwd_first_cursor(p);
        BwdSegment sg;
        while (ok && bwd_next_segment<kCausal, L::kR>(wcur, sg, p)) {
          const int n_steps = sg.i_end - sg.i_begin;
          if (!wait_bounded(bar_kv_full, units & 1u, wd, kSiteBwdKvFull, true, 0u)) {
            ok = false;
            break;
          }
          int cur = start_step(g);
          if (cur < 0) {
            ok = false;
            break;
          }
          for (int t = 0; t < n_steps; ++t, ++g) {
            // the next step's scores first: the tensor core computes them
            // while the compute threads form P^T and dS^T of this one
            int nxt = -1;
            if (t + 1 < n_steps) {
              nxt = start_step(g + 1);
              if (nxt < 0) {
                ok = false;
                break;
              }
            }
            if (!wait_bounded(bar_p_full, g & 1u, wd, kSiteBwdPFull, true, 0u)) {
              ok = false;
              break;
            }
            // the unit's first accumulation overwrites dV / dK: the previous
            // unit's epilogue must have loaded them
            if (t == 0 && units > 0 && !wait_bounded(bar_acc_free, (units - 1) & 1u, wd, kSiteBwdAccFree, true, 0u)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_grads(cur, t > 0);
            mma_commit(bar_stage_empty(cur));
            if (g > 0 && !wait_bounded(bar_dq_free, (g - 1) & 1u, wd, kSiteBwdDqFree, true, 0u)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_dq();
            mma_commit(bar_p_free);
            mma_commit(bar_dq_full);
            cur = nxt;
          }
          if (!ok) break;
          mma_commit(bar_acc_full);
          mma_commit(bar_kv_empty);
          ++units;
        }
      }
      // Drain: the CTA must not exit (or free TMEM) with MMAs in flight.
      const uint32_t drain = warp == kBwdMmaWarp ? bar_drain : bar_drain2;
      mma_commit(drain);
      wait_bounded(drain, 0u, wd, kSiteBwdDrain, false, kNapNs);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------- compute warps
    const int wg = warp >> 2;                 // query-column half of every step
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int rr = quarter * 32 + lane;       // key row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    // this warpgroup's query columns of a step: [kCW*wg, kCW*wg + kCW), in halves of 32
    const uint32_t tS = tmem + lane_off + L::kColS + static_cast<uint32_t>(L::kCW * wg);
    const uint32_t tDP = tmem + lane_off + L::kColDP + static_cast<uint32_t>(L::kCW * wg);
    const uint32_t tDQ = tmem + lane_off + L::kColDQ + static_cast<uint32_t>(L::kCW * wg);
    const uint32_t ds_row = sDS + static_cast<uint32_t>(rr * 128);
    const uint32_t xr = static_cast<uint32_t>(rr & 7);
    const bool dq_rows = quarter * 32 < D;    // warp-uniform: lanes >= D of dQ^T are discarded
    const float c = p.scale_log2;
    uint32_t g = 0, units = 0, ph = 0, part_phase = 0;
    int slot = 0;
    bool ok = true;
    int pend_bh = 0, pend_q0 = 0;  // head and first row of the step whose dQ^T is pending

    // dQ^T of global step `step` (head pend_bh, rows pend_q0 + kCW*wg +
    // [0, kCW)) from TMEM into the fp32 accumulator: this thread holds
    // head-dim index rr of those query rows. The warpgroup writes them into
    // its kCW x D staging rows (row-major, the accumulator's layout); each
    // block of 32 rows is added into global memory by one TMA reduce-add,
    // issued by the warpgroup's first thread (D <= 64) or by a lane of warp
    // kBwdDqWarp (D = 96, 128); the staging rows are rewritten once those
    // TMAs have read them.
    const bool leader = (threadIdx.x & 127) == 0;
    const uint32_t stage_rows = sDQS + static_cast<uint32_t>(wg * L::kCW * D * 4);
    uint32_t drains = 0;
    auto drain_dq = [&](uint32_t step) -> bool {
      bool got = wait_bounded(bar_dq_full, step & 1u, wd, kSiteBwdDqFull);
      got = __all_sync(0xffffffffu, got);
      if (!got) return false;
      tc_fence_after_sync();
      if constexpr (L::kDqRows) {
        // this thread's query row (TMEM lane rr) of dQ, columns [32 wg, 32 wg + 32)
        uint32_t v[32];
        tmem_ld32x32_wait(tmem + lane_off + L::kColDQ + 32u * wg, v);
        tc_fence_before_sync();
        mbar_arrive(bar_dq_free);
        if (drains > 0) {
          if (leader) {
            bulk_wait_read_all();
            mbar_arrive(bar_dqs_free(wg));
          }
          bool fr = wait_bounded(bar_dqs_free(wg), (drains - 1) & 1u, wd, kSiteBwdDqsFree);
          fr = __all_sync(0xffffffffu, fr);
          if (!fr) return false;
        }
        const bool has_cols = 32 * wg < D;  // warpgroup-uniform: at D = 32 the second half is padding
        const uint32_t box = sDQS + static_cast<uint32_t>(wg * 128 * 32 * 4);
        if (has_cols) {
          // 8 chunks of 4 columns into this row of the box, 128-byte swizzled
          const uint32_t row = box + static_cast<uint32_t>(rr * 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(row + ((static_cast<uint32_t>(ch) ^ xr) << 4), v[4 * ch], v[4 * ch + 1], v[4 * ch + 2],
                         v[4 * ch + 3]);
        }
        fence_proxy_async_shared();
        mbar_arrive(bar_dqs_ready(wg));
        if (quarter == 0) {  // the leader's warp waits as a whole, so its lanes agree on the outcome
          bool rd = wait_bounded(bar_dqs_ready(wg), drains & 1u, wd, kSiteBwdDqsReady);
          rd = __all_sync(0xffffffffu, rd);
          if (!rd) return false;
        }
        if (leader) {
          if (has_cols && pend_q0 < p.N)  // rows past N are outside the map and skipped
            tma_reduce_add_3d(&tmDQ, box, 32 * wg, pend_q0, pend_bh);
          bulk_commit_group();
        }
        ++drains;
        return true;
      }
      uint32_t v[L::kHalves][32];
      // every warp loads (lanes from D on hold the discarded rows; a load
      // guarded by dq_rows made the compiler spill at D = 32 and 96), only
      // the warps with real head-dim rows store below
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h) tmem_ld32x32_wait(tDQ + 32u * h, v[h]);
      tc_fence_before_sync();
      mbar_arrive(bar_dq_free);
      // the staging rows must have been read by the previous step's TMAs
      if (drains > 0) {
        if (!kDqWarp && leader) {
          bulk_wait_read_all();
          mbar_arrive(bar_dqs_free(wg));
        }
        bool fr = wait_bounded(bar_dqs_free(wg), (drains - 1) & 1u, wd, kSiteBwdDqsFree);
        fr = __all_sync(0xffffffffu, fr);
        if (!fr) return false;
      }
      if (dq_rows) {
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(stage_rows + static_cast<uint32_t>(((32 * h + i) * D + rr) * 4)),
                         "f"(__uint_as_float(v[h][i]))
                         : "memory");
        }
      }
      fence_proxy_async_shared();
      mbar_arrive(bar_dqs_ready(wg));
      if constexpr (kDqWarp) {
        ++drains;
        return true;
      }
      if (quarter == 0) {  // the leader's warp waits as a whole, so its lanes agree on the outcome
        bool rd = wait_bounded(bar_dqs_ready(wg), drains & 1u, wd, kSiteBwdDqsReady);
        rd = __all_sync(0xffffffffu, rd);
        if (!rd) return false;
      }
      if (leader) {
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
          const int q0 = pend_q0 + L::kCW * wg + 32 * h;
          if (q0 < p.N)  // rows past N are outside the map and skipped
            tma_reduce_add_3d(&tmDQ, stage_rows + static_cast<uint32_t>(32 * h * D * 4), 0, q0, pend_bh);
        }
        bulk_commit_group();
      }
      ++drains;
      return true;
    };

    BwdCursor cur = bwd_first_cursor(p);
    BwdSegment sg;
    while (ok && bwd_next_segment<kCausal, L::kR>(cur, sg, p)) {
      const int bh = sg.bh, kv = sg.kv;
      const int key = kv * kBwdKeys + rr;
      const bool key_ok = key < p.N;
      for (int i = sg.i_begin; i < sg.i_end; ++i, ++g) {
        bool got = wait_bounded(bar_s_full, g & 1u, wd, kSiteBwdSFull);
        got = got && wait_bounded(bar_stage_full(slot), ph, wd, kSiteBwdStageFull);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const float* neg_lse2_step = stats + slot * (L::kStatBytes / 4) + L::kCW * wg;
        const float* delta_step = neg_lse2_step + L::kSR;
        bool fr = true;
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
          uint32_t sr[32], dpr[32];
          tmem_ld32x32_nowait(tS + 32u * h, sr);
          tmem_ld32x32_nowait(tDP + 32u * h, dpr);
          tmem_wait_ld2(sr, dpr);
          if (h == L::kHalves - 1) {
            // S^T and dP^T are in registers: the issuer may compute the next ones.
            tc_fence_before_sync();
            mbar_arrive(bar_s_free);
          }
          // the step's -LSE*log2(e) and Delta values of these 32 query columns
          const float4* nl4 = reinterpret_cast<const float4*>(neg_lse2_step + 32 * h);
          const float4* dl4 = reinterpret_cast<const float4*>(delta_step + 32 * h);
          const int q0 = i * L::kSR + L::kCW * wg + 32 * h;  // query row of this thread's first column
          // masked: keys past N (ragged last tile) and, causal, keys after the query
          const bool masked = !key_ok || (kCausal && key > q0);
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 nl = nl4[j / 4];
            const float4 dl = dl4[j / 4];
            float e[4], pr[4], ds[4];
            ffma2(e[0], e[1], __uint_as_float(sr[j]), __uint_as_float(sr[j + 1]), c, nl.x, nl.y);
            ffma2(e[2], e[3], __uint_as_float(sr[j + 2]), __uint_as_float(sr[j + 3]), c, nl.z, nl.w);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              pr[t] = ex2_approx(e[t]);
              if (masked && (!key_ok || key > q0 + j + t)) pr[t] = 0.f;
            }
            fmul_sub2(ds[0], ds[1], pr[0], pr[1], __uint_as_float(dpr[j]), __uint_as_float(dpr[j + 1]), dl.x, dl.y);
            fmul_sub2(ds[2], ds[3], pr[2], pr[3], __uint_as_float(dpr[j + 2]), __uint_as_float(dpr[j + 3]), dl.z,
                      dl.w);
            pk[j / 2] = pack2(pr[0], pr[1], kBf16);
            pk[j / 2 + 1] = pack2(pr[2], pr[3], kBf16);
            dk[j / 2] = pack2(ds[0], ds[1], kBf16);
            dk[j / 2 + 1] = pack2(ds[2], ds[3], kBf16);
          }
          // the previous step's P^T / dS^T must have been read by the tensor core
          if (h == 0 && g > 0) {
            fr = wait_bounded(bar_p_free, (g - 1) & 1u, wd, kSiteBwdPFree);
            fr = __all_sync(0xffffffffu, fr);
            if (!fr) break;
          }
          // 4 chunks of 8 query columns into the 128-byte-swizzled key row of
          // the 64-column panel that holds them
          const int qc = L::kCW * wg + 32 * h;  // first query column of this half in the step
          const uint32_t panel = static_cast<uint32_t>((qc >> 6) * kPanelBytes);
          // P^T (and, at 64-row steps, dS^T) of these 32 query columns into
          // this thread's TMEM lane: 16 packed columns
          tmem_st32x16(tmem + lane_off + L::kColPT + static_cast<uint32_t>(qc / 2), pk);
          if constexpr (kATmem) tmem_st32x16(tmem + lane_off + L::kColDST + static_cast<uint32_t>(qc / 2), dk);
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint32_t col = panel + ((static_cast<uint32_t>(((qc & 63) >> 3) + ch) ^ xr) << 4);
            st_shared_v4(ds_row + col, dk[4 * ch], dk[4 * ch + 1], dk[4 * ch + 2], dk[4 * ch + 3]);
          }
        }
        if (!fr) {
          ok = false;
          break;
        }
        tmem_wait_st();
        fence_proxy_async_shared();
        tc_fence_before_sync();
        mbar_arrive(bar_p_full);
        if (g > 0 && !drain_dq(g - 1)) {
          ok = false;
          break;
        }
        pend_bh = bh;
        pend_q0 = i * L::kSR;
        if (++slot == L::kStages) {
          slot = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      // Epilogue: this thread's key row of dV and dK (half of the columns).
      bool got = wait_bounded(bar_acc_full, units & 1u, wd, kSiteBwdAccFull);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // This warpgroup's share of the key row: 32-column chunks [c0, c0 + n_my).
      constexpr int kMy = L::kChunksWg;
      const int c0 = wg * kMy;
      const int n_my = min(kMy, L::kChunks - c0);  // warp-uniform
      const size_t out_row = (static_cast<size_t>(bh) * p.N + (key_ok ? key : 0)) * (D * 2);
      // Writes 32 columns (chunk c) of this key row of dV and dK (dK scaled).
      auto store_chunk = [&](int c, const float (&a)[32], const float (&b)[32]) {
        uint4* dvp = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.dv) + out_row + c * 64);
        uint4* dkp = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.dk) + out_row + c * 64);
        const float sc = p.scale;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float* x = a + 8 * q;
          const float* y = b + 8 * q;
          dvp[q] = make_uint4(pack2(x[0], x[1], kBf16), pack2(x[2], x[3], kBf16), pack2(x[4], x[5], kBf16),
                              pack2(x[6], x[7], kBf16));
          dkp[q] = make_uint4(pack2(y[0] * sc, y[1] * sc, kBf16), pack2(y[2] * sc, y[3] * sc, kBf16),
                              pack2(y[4] * sc, y[5] * sc, kBf16), pack2(y[6] * sc, y[7] * sc, kBf16));
        }
      };
      if (p.stream_k && sg.i_begin > bwd_first_step<kCausal, L::kR>(kv)) {
        // Not the unit's first steps: hand this CTA's partial dV, dK to the
        // unit's owner through its workspace slot ([2][D][128], column-major
        // so that a warp's stores are contiguous), 32 columns at a time.
        float* pv = p.ws_part + static_cast<size_t>(blockIdx.x) * 2 * D * 128;
        float* pkk = pv + D * 128;
#pragma unroll 1
        for (int c = c0; c < c0 + n_my; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32x32_wait(tmem + lane_off + L::kColDV + 32 * c, a);
          tmem_ld32x32_wait(tmem + lane_off + L::kColDK + 32 * c, b);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            __stcg(pv + (32 * c + i) * 128 + rr, __uint_as_float(a[i]));
            __stcg(pkk + (32 * c + i) * 128 + rr, __uint_as_float(b[i]));
          }
        }
        tc_fence_before_sync();
        mbar_arrive(bar_acc_free);
        __threadfence();
        mbar_arrive(bar_part);
        if (warp == 0) {  // the whole warp waits, so that it stays converged
          bool done = wait_bounded(bar_part, part_phase, wd, kSiteBwdPartWrite);
          done = __all_sync(0xffffffffu, done);
          if (!done) {
            ok = false;
            break;
          }
          if (lane == 0) store_release(p.ws_flags + blockIdx.x, p.epoch);
        }
        part_phase ^= 1u;
        ++units;
        continue;
      }
      if (p.stream_k && sg.i_end < p.nq) {
        // Owner of a cut unit: add the partials of the CTAs that took the
        // rest of its steps, in CTA order (a fixed order: dV and dK do not
        // depend on timing), 32 columns at a time, then write dV and dK.
        int last_c = blockIdx.x;
        while (last_c + 1 < static_cast<int>(gridDim.x) && bwd_share_begin(p, last_c + 1) < sg.unit_end) ++last_c;
        bool fine = true;
        for (int cb = blockIdx.x + 1; cb <= last_c && fine; ++cb)
          fine = wait_flag(p.ws_flags + cb, p.epoch, wd, kSiteBwdPartFlag);
        fine = __all_sync(0xffffffffu, fine);
        if (!fine) {
          ok = false;
          break;
        }
#pragma unroll 1
        for (int c = c0; c < c0 + n_my; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32x32_wait(tmem + lane_off + L::kColDV + 32 * c, a);
          tmem_ld32x32_wait(tmem + lane_off + L::kColDK + 32 * c, b);
          float fa[32], fb[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            fa[i] = __uint_as_float(a[i]);
            fb[i] = __uint_as_float(b[i]);
          }
#pragma unroll 1
          for (int cb = blockIdx.x + 1; cb <= last_c; ++cb) {
            const float* pv = p.ws_part + static_cast<size_t>(cb) * 2 * D * 128 + (32 * c) * 128 + rr;
            const float* pkk = pv + D * 128;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              fa[i] += __ldcg(pv + i * 128);
              fb[i] += __ldcg(pkk + i * 128);
            }
          }
          if (key_ok) store_chunk(c, fa, fb);
        }
        tc_fence_before_sync();
        mbar_arrive(bar_acc_free);
        ++units;
        continue;
      }
      uint32_t dv[32 * kMy], dkr[32 * kMy];
#pragma unroll
      for (int c = 0; c < kMy; ++c) {
        // loads kMy chunks whatever n_my is: with an odd chunk count the
        // last one of warpgroup 1 lies past D but inside the dV / dK region
        // (columns [D, Dp), never stored), and an unguarded load keeps the
        // arrays in registers
        tmem_ld32x32_wait(tmem + lane_off + L::kColDV + 32 * (c0 + c), *reinterpret_cast<uint32_t(*)[32]>(dv + 32 * c));
        tmem_ld32x32_wait(tmem + lane_off + L::kColDK + 32 * (c0 + c), *reinterpret_cast<uint32_t(*)[32]>(dkr + 32 * c));
      }
      tc_fence_before_sync();
      mbar_arrive(bar_acc_free);
      if (key_ok) {
#pragma unroll
        for (int c = 0; c < kMy; ++c) {
          if (c < n_my)
            store_chunk(c0 + c, *reinterpret_cast<const float(*)[32]>(dv + 32 * c),
                        *reinterpret_cast<const float(*)[32]>(dkr + 32 * c));
        }
      }
      ++units;
    }
    // the last step's dQ^T; the staged blocks must be read (and added)
    // before the CTA's shared memory goes away
    if (ok && g > 0) drain_dq(g - 1);
    if (!kDqWarp && leader) bulk_wait_all();
  } else if (kDqWarp && warp == kBwdDqWarp) {
    // ------------------------------------------------------------- dQ adds
    // Lane w serves compute warpgroup w, walking the steps in the order
    // every role does: once the warpgroup has staged a step's dQ^T rows, one
    // TMA reduce-add per 32 rows into the fp32 accumulator; once the copy
    // engine has read them, the rows are given back. It polls without
    // sleeping.
    if (lane < 2) {
      const int w = lane;
      const uint32_t rows = sDQS + static_cast<uint32_t>(w * L::kCW * D * 4);
      uint32_t k = 0;  // steps whose rows were added
      bool ok = true;
      BwdCursor cur = bwd_first_cursor(p);
      BwdSegment sg;
      while (ok && bwd_next_segment<kCausal, L::kR>(cur, sg, p)) {
        for (int i = sg.i_begin; i < sg.i_end; ++i, ++k) {
          ok = wait_bounded(bar_dqs_ready(w), k & 1u, wd, kSiteBwdDqsReady, true, 0u);
          if (!ok) break;
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
            const int q0 = i * L::kSR + L::kCW * w + 32 * h;
            if (q0 < p.N)  // rows past N are outside the map and skipped
              tma_reduce_add_3d(&tmDQ, rows + static_cast<uint32_t>(32 * h * D * 4), 0, q0, sg.bh);
          }
          bulk_commit_group();
          bulk_wait_read_all();
          mbar_arrive(bar_dqs_free(w));
        }
      }
      // the adds in flight complete before the CTA's shared memory goes away
      bulk_wait_all();
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kBf16, bool kCausal>
cudaError_t launch_bwd(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const CUtensorMap& dout,
                       const CUtensorMap& dq_acc, const BwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fa2_bwd_kernel<D, kBf16, kCausal>;
  const int smem = BwdLayout<D>::kSmemBytes;
  // Once per device: the shared-memory opt-in.
  static PerDeviceOnce prepared;
  const cudaError_t e = once_per_device(
      prepared, [&]() { return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
  if (e != cudaSuccess) return e;
  // The stream-K schedule waits across CTAs, so it is launched cooperatively
  // (the whole grid resident at once, or the launch fails).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(bwd_threads(D));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = p.stream_k ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, k, v, q, dout, dq_acc, p);
}

}  // namespace fa2
