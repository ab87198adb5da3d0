// C ABI of the backward pass: argument validation, the workspace layout,
// the two elementwise kernels around the main one (prologue: Delta = rowsum
// of dO * O, LSE in log2 units, zeroed dQ accumulator; epilogue: dQ =
// scale * accumulator in the dtype), tensor maps and the persistent launch.
// Declarations and the contract of every entry point: include/fa2.h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "fa2.h"
#include "fa2_launch.h"

namespace fa2 {
namespace {

constexpr int kElemThreads = 256;
constexpr int kElemBlocksPerSm = 8;

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace: dQ accumulator | -LSE*log2(e) | Delta (rows padded to a multiple
// of the step rows) | stream-K partial dV, dK
// (one [2][D][128] fp32 slot per CTA, kBwdMaxCtas slots) | their flags.
struct BwdWorkspace {
  size_t dq_bytes, stat_bytes, part_bytes, flag_bytes, total;
};

BwdWorkspace workspace_layout(int64_t bh, int N, int D) {
  const int64_t sr = bwd_step_rows(D);
  const int64_t npad = (static_cast<int64_t>(N) + sr - 1) / sr * sr;
  BwdWorkspace w;
  w.dq_bytes = round256(static_cast<size_t>(bh) * N * D * sizeof(float));
  w.stat_bytes = round256(static_cast<size_t>(bh) * npad * sizeof(float));
  w.part_bytes = round256(static_cast<size_t>(kBwdMaxCtas) * 2 * D * 128 * sizeof(float));
  w.flag_bytes = round256(static_cast<size_t>(kBwdMaxCtas) * sizeof(unsigned long long));
  w.total = w.dq_bytes + 2 * w.stat_bytes + w.part_bytes + w.flag_bytes;
  return w;
}

// Cost of the busiest CTA in query steps under the round schedule (units
// dealt in rounds, zig-zag when causal: the kernel's bwd_round_unit and
// bwd_unit), or -1 when there are too many causal units to count on every
// call (the count is one pass over the units; past 2^15 units the zig-zag
// rounds are many and even, and the rounds are kept).
long long round_schedule_cost(long long units, int bh, int nkv, int nq, int steps_per_tile, bool causal, int grid) {
  if (!causal) return (units + grid - 1) / grid * nq;
  if (units > (1ll << 15)) return -1;
  long long worst = 0;
  for (int b = 0; b < grid; ++b) {
    long long sum = 0;
    for (long long r = 0;; ++r) {
      const long long u = r * grid + ((r & 1) ? (grid - 1 - b) : b);
      if (u >= units) break;
      const long long kv = u / bh;  // causal: K/V tile major over all heads
      sum += nq - steps_per_tile * kv;
    }
    worst = sum > worst ? sum : worst;
  }
  return worst;
}

// Partial-result write and merge of a cut unit, in query steps (its 2*128*D
// fp32 values go out once and are read once by the owner).
constexpr long long kBwdSplitCostSteps = 2;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8], bool bf16) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (bf16) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      f[2 * i] = __low2float(h);
      f[2 * i + 1] = __high2float(h);
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      f[2 * i] = __low2float(h);
      f[2 * i + 1] = __high2float(h);
    }
  }
}

__device__ __forceinline__ uint32_t pack_pair(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Per row (b, h, i) of the padded [B*H, Npad] grid: Delta_i = <dO_i, O_i>
// and -LSE_i * log2(e), the offset the main kernel adds to S * scale*log2(e)
// with one packed FMA per two scores (rows >= N: 0 and -inf, so that P is 0
// there), and zeroes the row of the fp32 dQ accumulator. D/8 threads per
// row, 8 elements (16 bytes) each, in groups of kLanes (D/8 rounded up to a
// power of two: the shuffle reduction's width; the extra lanes add zero);
// the loop bound is a multiple of 32 so that whole warps take part.
template <int D, bool kBf16>
__global__ void __launch_bounds__(kElemThreads) fa2_bwd_prologue(const uint4* __restrict__ O,
                                                                 const uint4* __restrict__ dO,
                                                                 const float* __restrict__ LSE,
                                                                 float* __restrict__ dq_acc, float* __restrict__ neg_lse2,
                                                                 float* __restrict__ delta, int N, int Npad,
                                                                 long long rows) {
  constexpr int kPer = D / 8;  // threads with data per row
  constexpr int kLanes = kPer <= 4 ? 4 : (kPer <= 8 ? 8 : (kPer <= 16 ? 16 : 32));
  static_assert(kPer <= 32, "head dimension");
  const long long items = rows * kLanes;
  const long long bound = (items + 31) / 32 * 32;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < bound; idx += stride) {
    const long long row = idx / kLanes;
    const int part = static_cast<int>(idx % kLanes);
    const bool live = idx < items;
    const long long bh = live ? row / Npad : 0;
    const int i = live ? static_cast<int>(row % Npad) : 0;
    const bool real = live && i < N && part < kPer;
    float acc = 0.f;
    if (real) {
      const long long e = (bh * N + i) * kPer + part;  // in 16-byte units
      float o[8], g[8];
      unpack8(O[e], o, kBf16);
      unpack8(dO[e], g, kBf16);
#pragma unroll
      for (int k = 0; k < 8; ++k) acc = fmaf(o[k], g[k], acc);
      float4* z = reinterpret_cast<float4*>(dq_acc + e * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = kLanes / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, kLanes);
    if (live && part == 0) {
      const bool in_range = i < N;
      delta[row] = in_range ? acc : 0.f;
      neg_lse2[row] = in_range ? -(LSE[bh * N + i] * 1.4426950408889634f) : -CUDART_INF_F;
    }
  }
}

// dQ = dtype(scale * accumulator), 8 elements per thread.
template <bool kBf16>
__global__ void __launch_bounds__(kElemThreads) fa2_bwd_dq_convert(const float4* __restrict__ acc,
                                                                   uint4* __restrict__ dq, float scale,
                                                                   long long n8) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n8; idx += stride) {
    const float4 a = acc[2 * idx], b = acc[2 * idx + 1];
    dq[idx] = make_uint4(pack_pair(a.x * scale, a.y * scale, kBf16), pack_pair(a.z * scale, a.w * scale, kBf16),
                         pack_pair(b.x * scale, b.y * scale, kBf16), pack_pair(b.z * scale, b.w * scale, kBf16));
  }
}

using BwdLaunchFn = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                    const CUtensorMap&, const BwdParams&, int, cudaStream_t);

template <int D>
BwdLaunchFn pick_bwd_d(bool bf, bool c) {
  if (bf) return c ? launch_bwd<D, true, true> : launch_bwd<D, true, false>;
  return c ? launch_bwd<D, false, true> : launch_bwd<D, false, false>;
}

BwdLaunchFn pick_bwd(int d, int dtype, int causal) {
  const bool bf = dtype == FA2_BF16, c = causal != 0;
  switch (d) {
    case 32: return pick_bwd_d<32>(bf, c);
    case 64: return pick_bwd_d<64>(bf, c);
    case 96: return pick_bwd_d<96>(bf, c);
    default: return pick_bwd_d<128>(bf, c);
  }
}

template <int D>
cudaError_t launch_prologue(bool bf16, const void* O, const void* dO, const float* LSE, float* dq_acc, float* neg_lse2,
                            float* delta, int N, int Npad, long long rows, int grid, cudaStream_t s) {
  const uint4* o = static_cast<const uint4*>(O);
  const uint4* g = static_cast<const uint4*>(dO);
  if (bf16)
    fa2_bwd_prologue<D, true><<<grid, kElemThreads, 0, s>>>(o, g, LSE, dq_acc, neg_lse2, delta, N, Npad, rows);
  else
    fa2_bwd_prologue<D, false><<<grid, kElemThreads, 0, s>>>(o, g, LSE, dq_acc, neg_lse2, delta, N, Npad, rows);
  return cudaGetLastError();
}

int grid_for(long long items, int sms) {
  const long long need = (items + kElemThreads - 1) / kElemThreads;
  const long long cap = static_cast<long long>(sms) * kElemBlocksPerSm;
  return static_cast<int>(need < cap ? (need > 0 ? need : 1) : cap);
}

}  // namespace
}  // namespace fa2

using namespace fa2;

extern "C" int fa2_bwd_workspace_bytes(int B, int H, int N, int D, size_t* bytes) {
  if (!bytes || B < 0 || H < 0 || N < 0) return FA2_ERR_INVALID_ARG;
  if (!bwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  *bytes = workspace_layout(static_cast<int64_t>(B) * H, N, D).total;
  return FA2_OK;
}

extern "C" int fa2_bwd_sched(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                             const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int D, float scale,
                             int is_causal, int dtype, void* workspace, size_t workspace_bytes, int schedule,
                             struct CUstream_st* stream) {
  if (B < 0 || H < 0 || N < 0) return FA2_ERR_INVALID_ARG;
  if (schedule != FA2_SCHED_AUTO && schedule != FA2_SCHED_UNITS && schedule != FA2_SCHED_BALANCED)
    return FA2_ERR_INVALID_ARG;
  if (!bwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  if (dtype != FA2_F16 && dtype != FA2_BF16) return FA2_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA2_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return FA2_OK;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace) return FA2_ERR_INVALID_ARG;
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int64_t nkv = (static_cast<int64_t>(N) + kBwdKeys - 1) / kBwdKeys;
  if (bh > INT32_MAX || bh * nkv > INT32_MAX) return FA2_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                        reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                        reinterpret_cast<uintptr_t>(dO) | reinterpret_cast<uintptr_t>(LSE) |
                        reinterpret_cast<uintptr_t>(dQ) | reinterpret_cast<uintptr_t>(dK) |
                        reinterpret_cast<uintptr_t>(dV);
  if (mis & 15u) return FA2_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA2_ERR_ALIGN;
  const BwdWorkspace wl = workspace_layout(bh, N, D);
  if (workspace_bytes < wl.total) return FA2_ERR_INVALID_ARG;
  const size_t tb = static_cast<size_t>(bh) * N * D * 2;
  const size_t lb = static_cast<size_t>(bh) * N * 4;
  const void* ins[6] = {Q, K, V, O, dO, LSE};
  const size_t in_bytes[6] = {tb, tb, tb, tb, tb, lb};
  const void* outs[4] = {dQ, dK, dV, workspace};
  const size_t out_bytes[4] = {tb, tb, tb, workspace_bytes};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (ranges_overlap(outs[a], out_bytes[a], ins[b], in_bytes[b])) return FA2_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (ranges_overlap(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA2_ERR_INVALID_ARG;
  }

  int sms = 0;
  int* status = nullptr;
  const int rc = current_device_facts(&sms, &status);
  if (rc != FA2_OK) return rc;

  CUtensorMap mk, mv, mq, mdo;
  if (!encode_tile_map(&mk, K, (int)bh, N, D, dtype, kBwdKeys) ||
      !encode_tile_map(&mv, V, (int)bh, N, D, dtype, kBwdKeys) ||
      !encode_tile_map(&mq, Q, (int)bh, N, D, dtype, static_cast<unsigned>(bwd_step_rows(D))) ||
      !encode_tile_map(&mdo, dO, (int)bh, N, D, dtype, static_cast<unsigned>(bwd_step_rows(D))))
    return record_cuda_error(cudaErrorInvalidValue);

  const int sr = bwd_step_rows(D);
  const int npad = (N + sr - 1) / sr * sr;
  char* ws = static_cast<char*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(ws);
  CUtensorMap mdq;  // the kernel adds blocks of 32 rows of dQ into the accumulator
  const bool mapped = D <= 64 ? encode_f32_cols_map_sw128(&mdq, dq_acc, (int)bh, N, D, 128)
                              : encode_f32_rows_map(&mdq, dq_acc, (int)bh, N, D, 32);
  if (!mapped) return record_cuda_error(cudaErrorInvalidValue);
  float* neg_lse2 = reinterpret_cast<float*>(ws + wl.dq_bytes);
  float* delta = reinterpret_cast<float*>(ws + wl.dq_bytes + wl.stat_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool bf = dtype == FA2_BF16;

  const long long rows = bh * npad;
  const int pgrid = grid_for(rows * (D / 8), sms);
  cudaError_t e;
  switch (D) {
    case 32: e = launch_prologue<32>(bf, O, dO, LSE, dq_acc, neg_lse2, delta, N, npad, rows, pgrid, s); break;
    case 64: e = launch_prologue<64>(bf, O, dO, LSE, dq_acc, neg_lse2, delta, N, npad, rows, pgrid, s); break;
    case 96: e = launch_prologue<96>(bf, O, dO, LSE, dq_acc, neg_lse2, delta, N, npad, rows, pgrid, s); break;
    default: e = launch_prologue<128>(bf, O, dO, LSE, dq_acc, neg_lse2, delta, N, npad, rows, pgrid, s); break;
  }
  if (e != cudaSuccess) return record_cuda_error(e);

  BwdParams p = {};
  p.dk = dK;
  p.dv = dV;
  p.dq_acc = dq_acc;
  p.neg_lse2 = neg_lse2;
  p.delta = delta;
  p.status = status;
  p.watchdog_ns = watchdog_limit_ns();
  p.N = N;
  p.Npad = npad;
  p.BH = (int)bh;
  p.nkv = (int)nkv;
  p.nq = npad / sr;
  p.num_units = (int)(bh * nkv);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.scale = scale;
  // Query steps of one head: non-causal nkv * nq; causal, K/V tile kv sees
  // the steps from kv * (128 / step rows) on.
  const int steps_per_tile = kBwdKeys / sr;
  long long per_head = 0;
  for (int64_t kv = 0; kv < nkv; ++kv) per_head += is_causal ? p.nq - steps_per_tile * kv : p.nq;
  p.steps_per_head = per_head;
  p.total_steps = per_head * bh;
  const int round_grid = p.num_units < sms ? p.num_units : sms;
  const int sk_grid = static_cast<int>(std::min<long long>(std::min(sms, kBwdMaxCtas), p.total_steps));
  bool balanced = schedule == FA2_SCHED_BALANCED;
  if (schedule == FA2_SCHED_AUTO) {
    // the schedule whose busiest CTA has fewer steps, balanced only when it
    // saves at least 5 %
    const long long rounds =
        round_schedule_cost(p.num_units, p.BH, p.nkv, p.nq, steps_per_tile, is_causal != 0, round_grid);
    const long long split = (p.total_steps + sk_grid - 1) / sk_grid + kBwdSplitCostSteps;
    balanced = rounds > 0 && 100 * split < 95 * rounds;
  }
  p.test_withhold = take_test_withhold();
  int grid = round_grid;
  if (balanced) {
    p.stream_k = 1;
    grid = sk_grid;
    p.ws_part = reinterpret_cast<float*>(ws + wl.dq_bytes + 2 * wl.stat_bytes);
    p.ws_flags = reinterpret_cast<unsigned long long*>(ws + wl.dq_bytes + 2 * wl.stat_bytes + wl.part_bytes);
    p.epoch = next_launch_epoch();
  }
  e = pick_bwd(D, dtype, is_causal)(mk, mv, mq, mdo, mdq, p, grid, s);
  if (e != cudaSuccess) return record_cuda_error(e);

  const long long n8 = bh * N * (D / 8);
  const int cgrid = grid_for(n8, sms);
  if (bf)
    fa2_bwd_dq_convert<true><<<cgrid, kElemThreads, 0, s>>>(reinterpret_cast<const float4*>(dq_acc),
                                                             static_cast<uint4*>(dQ), scale, n8);
  else
    fa2_bwd_dq_convert<false><<<cgrid, kElemThreads, 0, s>>>(reinterpret_cast<const float4*>(dq_acc),
                                                              static_cast<uint4*>(dQ), scale, n8);
  e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda_error(e);
  return FA2_OK;
}

extern "C" int fa2_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, int B, int H, int N, int D, float scale, int is_causal,
                       int dtype, void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
  return fa2_bwd_sched(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, D, scale, is_causal, dtype, workspace,
                       workspace_bytes, FA2_SCHED_AUTO, stream);
}
