// Pieces shared by the forward kernels (fa2_kernel.cuh: head dims up to
// 128, two 128-row query sub-tiles per work unit; fa2_kernel_wide.cuh: head
// dim 256, one sub-tile per unit): the thread layout and register split, the
// work-unit walk of both schedules (rounds of whole units, or stream-K shares
// of K/V-tile steps), the bounded waits of the device watchdog, and 16-bit
// packing.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "fa2_launch.h"
#include "sm103_ptx.cuh"
#include "tmem_io.cuh"

namespace fa2 {

constexpr int kThreads = 384;     // 3 warpgroups
constexpr int kMmaWarp = 8;       // first MMA issuer warp
constexpr int kLoadWarp = 10;
// Two MMA issuers (one per sub-tile, or one per instruction type: every S
// and every P.V; each kernel says which): a thread issuing tcgen05.mma is
// held until the tensor core takes each instruction (~90-110 cycles for
// these M=128 x N=128 x K=16 steps), so one thread cannot keep the tensor
// core busy.
constexpr int kIssuers = 2;
// Registers: the launch gives every thread kLaunchRegs (= 65536 / 384 rounded
// down to 8); the softmax warpgroups then take kSoftmaxRegs and the third
// warpgroup gives back down to kControlRegs. The split must add up exactly.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 216;
constexpr int kControlRegs = 72;
static_assert(2 * kSoftmaxRegs + kControlRegs == 3 * kLaunchRegs, "register split must match the launch");
constexpr int kPanelBytes = 128 * 128;  // 128 rows x 64 16-bit elements
constexpr int kPTileBytes = 2 * kPanelBytes;  // P of one sub-tile: 128 rows x 128 keys
constexpr uint32_t kTmemCols = 512;
// The exponent base of a row moves only when its max exceeds the base by more
// than this many powers of two (so p <= 2^8 = 256, exact in the 16-bit P and
// far from overflow in the fp32 sums).
constexpr float kRescaleLog2 = 8.0f;
// Sleep between polls of the producer's and MMA issuers' waits (see wait_bounded).
constexpr unsigned kNapNs = 20;

// Watchdog codes written to the status word (site of the wait that gave up).
enum : int {
  kSiteLoadQEmpty = 1,
  kSiteLoadRingEmpty = 2,
  kSiteMmaQFull = 3,
  kSiteMmaRingFull = 4,
  kSiteMmaPFull = 5,
  kSiteSoftmaxSFull = 6,
  kSiteSoftmaxOFull = 7,
  kSiteDrain = 8,
  kSitePartialWrite = 9,
  kSitePartialFlag = 10,
  kSiteMmaSFree = 11,
  kSiteSoftmaxPFree = 12,
  kSiteOStaged = 13,
  kSiteOBufFree = 14,
};

// A work unit is kR 128-row query sub-tiles: kR = 2 (256 rows, head dims up
// to 128) or kR = 1 (128 rows, head dim 256).
// K/V tiles of query unit qt (rows from kR*128*qt).
template <bool kCausal, int kR = 2>
__device__ __forceinline__ int unit_nkv(int qt, const Params& p) {
  return kCausal ? min(kR * qt + kR, p.nkv_full) : p.nkv_full;
}

// First K/V-tile step of causal unit qt within its head: the sum of
// kR*(i+1) over the units i < qt (only the last unit of a head is ever
// clipped by nkv_full, so the sum is exact for every unit).
template <int kR>
__device__ __forceinline__ long long causal_unit_start(int qt) {
  return static_cast<long long>(kR) * qt * (qt + 1) / 2;
}

struct Segment {
  int bh;
  int q0;                // first query row of the unit
  int kv_begin, kv_end;  // K/V tiles processed in this segment
  int nkv;               // K/V tiles of the whole unit
  long long unit_end;    // stream-K: step one past the unit's last step
};

struct SegCursor {
  int round;             // round schedule
  long long step, end;   // stream-K schedule
};

__device__ __forceinline__ long long stream_k_begin(const Params& p, int b) {
  return p.total_steps * b / gridDim.x;
}

__device__ __forceinline__ SegCursor first_cursor(const Params& p) {
  SegCursor c;
  c.round = 0;
  c.step = p.stream_k ? stream_k_begin(p, blockIdx.x) : 0;
  c.end = p.stream_k ? stream_k_begin(p, blockIdx.x + 1) : 0;
  return c;
}

// Next segment of this CTA. Every role walks the same sequence.
template <bool kCausal, int kR = 2>
__device__ __forceinline__ bool next_segment(SegCursor& c, Segment& s, const Params& p) {
  if (!p.stream_k) {
    // Rounds of whole units. Non-causal: consecutive units share a head (K/V
    // reuse in L2). Causal: heaviest query tiles first, dealt in a zig-zag so
    // heavy and light ends of each round spread over the CTAs.
    const int g = gridDim.x, b = blockIdx.x, r = c.round++;
    const int u = r * g + ((kCausal && (r & 1)) ? (g - 1 - b) : b);
    if (u >= p.num_units) return false;
    int qt, bh;
    if (kCausal) {
      qt = p.n_qt - 1 - u / p.BH;
      bh = u % p.BH;
    } else {
      qt = u % p.n_qt;
      bh = u / p.n_qt;
    }
    s.bh = bh;
    s.q0 = qt * kR * kRows;
    s.nkv = unit_nkv<kCausal, kR>(qt, p);
    s.kv_begin = 0;
    s.kv_end = s.nkv;
    s.unit_end = 0;
    return true;
  }
  if (c.step >= c.end) return false;
  // Units in order (head, query tile ascending); unit qt of a head starts at
  // step qt*nkv_full (non-causal) or kR*qt*(qt+1)/2 (causal: nkv = kR*(qt+1)).
  const long long bh = c.step / p.steps_per_head;
  const int r = static_cast<int>(c.step - bh * p.steps_per_head);
  int qt, start;
  if (kCausal) {
    qt = static_cast<int>((sqrtf(8.f * r / kR + 1.f) - 1.f) * 0.5f);
    qt = min(max(qt, 0), p.n_qt - 1);
    while (qt > 0 && causal_unit_start<kR>(qt) > r) --qt;
    while (qt + 1 < p.n_qt && causal_unit_start<kR>(qt + 1) <= r) ++qt;
    start = static_cast<int>(causal_unit_start<kR>(qt));
  } else {
    qt = r / p.nkv_full;
    start = qt * p.nkv_full;
  }
  s.bh = static_cast<int>(bh);
  s.q0 = qt * kR * kRows;
  s.nkv = unit_nkv<kCausal, kR>(qt, p);
  s.kv_begin = r - start;
  const long long left = c.end - c.step;
  s.kv_end = static_cast<int>(min(static_cast<long long>(s.nkv), s.kv_begin + left));
  s.unit_end = c.step - s.kv_begin + s.nkv;
  c.step += s.kv_end - s.kv_begin;
  return true;
}

struct Watchdog {
  int* status;
  volatile int* abort_flag;
  unsigned long long limit_ns;
};

// Bounded wait. Returns false when the limit passes (recording `site` in the
// status word and raising the CTA's abort flag) or when another role of the
// CTA has already aborted. `honour_abort` = false is used while draining.
// `nap_ns` > 0 sleeps between polls: the single-thread roles (producer, MMA
// issuers) share each SM sub-partition with softmax warps, whose issue slots
// a tight polling loop would take (measured: 12 % on long causal work).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const Watchdog& wd, int site,
                                          bool honour_abort = true, unsigned nap_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (nap_ns) __nanosleep(nap_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (honour_abort && *wd.abort_flag) return false;
      if (global_timer_ns() - t0 > wd.limit_ns) {
        *wd.abort_flag = 1;
        atomicCAS(wd.status, 0, site);
        return false;
      }
    }
  }
}

// Bounded wait for a global flag to carry this launch's epoch (acquire).
__device__ __forceinline__ bool wait_flag(const unsigned long long* f, unsigned long long epoch, const Watchdog& wd,
                                          int site) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    if (v == epoch) return true;
    if (it == 0) t0 = global_timer_ns();
    if ((it & 15u) == 15u) {
      if (*wd.abort_flag) return false;
      if (global_timer_ns() - t0 > wd.limit_ns) {
        *wd.abort_flag = 1;
        atomicCAS(wd.status, 0, site);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void store_release(unsigned long long* f, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ float round16(float x, bool bf16) {
  return bf16 ? __bfloat162float(__float2bfloat16_rn(x)) : __half2float(__float2half_rn(x));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

}  // namespace fa2
