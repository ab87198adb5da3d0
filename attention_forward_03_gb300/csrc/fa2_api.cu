// C ABI of the forward library: argument validation, TMA descriptors, the
// persistent launch and the device watchdog word. Declarations and the
// contract of every entry point: include/fa2.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fa2.h"
#include "fa2_launch.h"

namespace fa2 {
namespace {

constexpr unsigned long long kDefaultWatchdogNs = 1000000000ull;

__device__ int g_watchdog_word;  // 0 = no timeout since last clear

std::atomic<unsigned long long> g_watchdog_ns{kDefaultWatchdogNs};
std::atomic<int> g_test_withhold{0};
thread_local char t_last_cuda_error[256] = "";

struct DeviceInfo {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  bool supported = false;  // compute capability 10.3, and this library's device code loaded there
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  int* status = nullptr;
};
DeviceInfo g_devices[kMaxDevices];

int record_cuda(cudaError_t e) {
  std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return FA2_ERR_CUDA;
}

// Device properties and the watchdog word's device address, once per device,
// queried with that device current. The compute capability comes first: on
// any other GPU this library's device code (sm_103a only) cannot load, so
// the symbol lookup is not attempted there and the device is "unsupported".
DeviceInfo* device_info(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& d = g_devices[dev];
  std::call_once(d.once, [&] {
    cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess && d.cc_major == 10 && d.cc_minor == 3) {
      e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_watchdog_word);
      d.supported = e == cudaSuccess;
    }
    d.err = e;
  });
  return &d;
}

// The current device's facts: FA2_OK, FA2_ERR_CUDA (recorded) or
// FA2_ERR_UNSUPPORTED (not an sm_103 GPU).
int current_device(DeviceInfo** out) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  DeviceInfo* info = device_info(dev);
  if (!info) return FA2_ERR_UNSUPPORTED;
  if (info->err != cudaSuccess) return record_cuda(info->err);
  if (!info->supported) return FA2_ERR_UNSUPPORTED;
  *out = info;
  return FA2_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Encoded tensor maps, cached by everything that goes into them (address,
// shape, element type, box height), so that repeated calls on the same
// buffers skip the encoding. A descriptor depends only on these values, so
// an entry stays valid after its buffer is freed (a later buffer at the same
// address with the same shape gets the same descriptor). Direct-mapped,
// guarded by one lock.
struct MapKey {
  const void* ptr;
  int bh, n, d, kind;  // kind: the 16-bit dtype code, 16 for fp32 rows, 17 for fp32 swizzled column boxes
  unsigned rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && bh == o.bh && n == o.n && d == o.d && kind == o.kind && rows == o.rows;
  }
};

constexpr int kMapCacheSlots = 512;
struct MapCache {
  std::mutex mu;
  bool used[kMapCacheSlots] = {};
  MapKey key[kMapCacheSlots];
  CUtensorMap map[kMapCacheSlots];
};
MapCache g_maps;

uint32_t map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.ptr);
  for (uint64_t v : {(uint64_t)k.bh, (uint64_t)k.n, (uint64_t)k.d, (uint64_t)k.kind, (uint64_t)k.rows})
    h = (h ^ v) * 0x9e3779b97f4a7c15ull;
  h ^= h >> 29;
  return static_cast<uint32_t>(h % kMapCacheSlots);
}

// Looks `key` up; on a miss encodes it with `enc_fn` and stores it.
template <typename F>
bool cached_map(CUtensorMap* out, const MapKey& key, F&& enc_fn) {
  const uint32_t slot = map_slot(key);
  {
    std::lock_guard<std::mutex> lock(g_maps.mu);
    if (g_maps.used[slot] && g_maps.key[slot] == key) {
      *out = g_maps.map[slot];
      return true;
    }
  }
  if (!enc_fn(out)) return false;
  std::lock_guard<std::mutex> lock(g_maps.mu);
  g_maps.used[slot] = true;
  g_maps.key[slot] = key;
  g_maps.map[slot] = *out;
  return true;
}

// [B*H, N, D] view of a [B,H,N,D] tensor; `rows` rows x 64 elements per box,
// 128-byte swizzle; rows past N, and columns past D (D = 32, or the second
// panel at D = 96), read as zeros.
bool make_rows_map(CUtensorMap* map, const void* ptr, int bh, int n, int d, int dtype, unsigned rows) {
  return cached_map(map, MapKey{ptr, bh, n, d, dtype, rows}, [&](CUtensorMap* m) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2};
    cuuint32_t box[3] = {64, rows, 1};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = enc(m, dtype == FA2_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                     const_cast<void*>(ptr), dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  });
}

bool make_map(CUtensorMap* map, const void* ptr, int bh, int n, int d, int dtype) {
  return make_rows_map(map, ptr, bh, n, d, dtype, 128);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

using LaunchFn = cudaError_t (*)(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                 const Params&, int, cudaStream_t);

template <int D>
LaunchFn pick_d(bool bf, bool c) {
  if (bf) return c ? launch_fwd<D, true, true> : launch_fwd<D, true, false>;
  return c ? launch_fwd<D, false, true> : launch_fwd<D, false, false>;
}

LaunchFn pick(int d, int dtype, int causal) {
  const bool bf = dtype == FA2_BF16, c = causal != 0;
  switch (d) {
    case 32: return pick_d<32>(bf, c);
    case 64: return pick_d<64>(bf, c);
    case 96: return pick_d<96>(bf, c);
    case 128: return pick_d<128>(bf, c);
    case 512:
      if (bf) return c ? launch_fwd_dtile<512, true, true> : launch_fwd_dtile<512, true, false>;
      return c ? launch_fwd_dtile<512, false, true> : launch_fwd_dtile<512, false, false>;
    case 1024:
      if (bf) return c ? launch_fwd_dtile<1024, true, true> : launch_fwd_dtile<1024, true, false>;
      return c ? launch_fwd_dtile<1024, false, true> : launch_fwd_dtile<1024, false, false>;
    default:
      if (bf) return c ? launch_fwd_wide<256, true, true> : launch_fwd_wide<256, true, false>;
      return c ? launch_fwd_wide<256, false, true> : launch_fwd_wide<256, false, false>;
  }
}

}  // namespace
}  // namespace fa2

using namespace fa2;

namespace {

std::atomic<unsigned long long> g_epoch{0};

// Launch tags: a per-process random high half and a counter, so a workspace
// flag left by any earlier launch (of this or another process) never matches.
unsigned long long next_epoch() {
  static const unsigned long long salt = [] {
    unsigned long long x = static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count());
    x ^= static_cast<unsigned long long>(getpid()) << 21;
    x ^= reinterpret_cast<uintptr_t>(&g_epoch);
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return (x ^ (x >> 31)) << 32;
  }();
  return salt | ((g_epoch.fetch_add(1, std::memory_order_relaxed) + 1) & 0xffffffffull);
}

// `schedule`: FA2_SCHED_UNITS (the workspace is ignored), FA2_SCHED_BALANCED
// (needs the workspace) or FA2_SCHED_AUTO (the cost model's choice, the
// rounds when there is no workspace).
int launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int D,
           float scale, int is_causal, int dtype, void* workspace, size_t workspace_bytes, int schedule,
           cudaStream_t stream) {
  if (schedule == FA2_SCHED_UNITS) {
    workspace = nullptr;
    workspace_bytes = 0;
  }
  if (B < 0 || H < 0 || N < 0) return FA2_ERR_INVALID_ARG;
  if (!fwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  if (dtype != FA2_F16 && dtype != FA2_BF16) return FA2_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA2_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return FA2_OK;
  if (!Q || !K || !V || !O || !LSE) return FA2_ERR_INVALID_ARG;
  const int64_t bh = static_cast<int64_t>(B) * H;
  const int unit_rows = fwd_unit_rows(D), unit_subtiles = fwd_unit_subtiles(D);
  const int64_t n_qt = (static_cast<int64_t>(N) + unit_rows - 1) / unit_rows;
  const int64_t bh_sched = bh * fwd_out_chunks(D);  // heads as the scheduler sees them
  if (bh > INT32_MAX || bh_sched * n_qt > INT32_MAX) return FA2_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                        reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                        reinterpret_cast<uintptr_t>(LSE) | reinterpret_cast<uintptr_t>(workspace);
  if (mis & 15u) return FA2_ERR_ALIGN;
  const size_t tbytes = static_cast<size_t>(bh) * N * D * 2;
  const size_t lbytes = static_cast<size_t>(bh) * N * 4;
  if (overlaps(O, tbytes, Q, tbytes) || overlaps(O, tbytes, K, tbytes) || overlaps(O, tbytes, V, tbytes) ||
      overlaps(LSE, lbytes, Q, tbytes) || overlaps(LSE, lbytes, K, tbytes) || overlaps(LSE, lbytes, V, tbytes) ||
      overlaps(LSE, lbytes, O, tbytes))
    return FA2_ERR_INVALID_ARG;
  if (workspace && (overlaps(workspace, workspace_bytes, Q, tbytes) || overlaps(workspace, workspace_bytes, K, tbytes) ||
                    overlaps(workspace, workspace_bytes, V, tbytes) || overlaps(workspace, workspace_bytes, O, tbytes) ||
                    overlaps(workspace, workspace_bytes, LSE, lbytes)))
    return FA2_ERR_INVALID_ARG;

  DeviceInfo* info = nullptr;
  const int rc = current_device(&info);
  if (rc != FA2_OK) return rc;
  if (workspace && workspace_bytes < stream_k_workspace_bytes(info->sms, D)) return FA2_ERR_INVALID_ARG;
  if (schedule == FA2_SCHED_AUTO && workspace &&
      fwd_auto_schedule(B, H, N, D, is_causal, info->sms) != FA2_SCHED_BALANCED)
    workspace = nullptr;  // the rounds win: run them, the workspace unused
  if (fwd_dtiled(D)) workspace = nullptr;  // head dims 512, 1024: round schedule only

  CUtensorMap mq, mk, mv, mo;
  // V boxes: 128 rows, or at head dims from 256 64 rows (the kernels stream V
  // in halves of 64 keys there); O: the kernel stores it through a map at
  // D = 96, 128
  if (!make_map(&mq, Q, (int)bh, N, D, dtype) || !make_map(&mk, K, (int)bh, N, D, dtype) ||
      !make_rows_map(&mv, V, (int)bh, N, D, dtype, D >= 256 ? 64u : 128u) || !make_map(&mo, O, (int)bh, N, D, dtype)) {
    std::snprintf(t_last_cuda_error, sizeof(t_last_cuda_error), "cuTensorMapEncodeTiled failed");
    return FA2_ERR_CUDA;
  }
  Params p = {};
  p.o = O;
  p.lse = LSE;
  p.status = info->status;
  p.watchdog_ns = g_watchdog_ns.load(std::memory_order_relaxed);
  p.N = N;
  p.BH = (int)bh_sched;
  p.n_qt = (int)n_qt;
  p.num_units = (int)(bh_sched * n_qt);
  p.nkv_full = (N + kKeys - 1) / kKeys;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.test_withhold = g_test_withhold.exchange(0, std::memory_order_relaxed);
  // K/V-tile steps of one head: non-causal n_qt * nkv_full; causal sum of
  // min(T*(qt+1), nkv_full) over the head's query units (T sub-tiles per unit).
  long long per_head = 0;
  if (is_causal) {
    for (int64_t qt = 0; qt < n_qt; ++qt)
      per_head += std::min<long long>(unit_subtiles * (qt + 1), p.nkv_full);
  } else {
    per_head = n_qt * static_cast<long long>(p.nkv_full);
  }
  p.steps_per_head = per_head;
  p.total_steps = per_head * bh_sched;
  int grid;
  if (workspace) {
    p.stream_k = 1;
    grid = static_cast<int>(std::min<long long>(info->sms, p.total_steps));
    const size_t slots = static_cast<size_t>(info->sms) * unit_subtiles;
    char* ws = static_cast<char*>(workspace);
    p.ws_o = reinterpret_cast<float*>(ws);
    p.ws_stats = p.ws_o + slots * D * 128;
    const size_t fbytes = (slots * (static_cast<size_t>(D) * 128 + 3 * 128) * sizeof(float) + 255) / 256 * 256;
    p.ws_flags = reinterpret_cast<unsigned long long*>(ws + fbytes);
    p.epoch = next_epoch();
  } else {
    p.stream_k = 0;
    grid = p.num_units < info->sms ? p.num_units : info->sms;
  }
  const cudaError_t e = pick(D, dtype, is_causal)(mq, mk, mv, mo, p, grid, stream);
  if (e != cudaSuccess) return record_cuda(e);
  return FA2_OK;
}

}  // namespace

namespace fa2 {
int record_cuda_error(cudaError_t e) { return record_cuda(e); }

unsigned long long next_launch_epoch() { return next_epoch(); }

int take_test_withhold() { return g_test_withhold.exchange(0, std::memory_order_relaxed); }

int current_device_facts(int* sms, int** status) {
  DeviceInfo* info = nullptr;
  const int rc = current_device(&info);
  if (rc != FA2_OK) return rc;
  *sms = info->sms;
  *status = info->status;
  return FA2_OK;
}

bool encode_tile_map(CUtensorMap* map, const void* ptr, int bh, int n, int d, int dtype, unsigned rows) {
  return make_rows_map(map, ptr, bh, n, d, dtype, rows);
}

bool encode_f32_cols_map_sw128(CUtensorMap* map, float* ptr, int bh, int n, int d, unsigned rows) {
  return cached_map(map, MapKey{ptr, bh, n, d, 17, rows}, [&](CUtensorMap* m) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)n * d * 4};
    cuuint32_t box[3] = {32, rows, 1};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  });
}

bool encode_f32_rows_map(CUtensorMap* map, float* ptr, int bh, int n, int d, unsigned rows) {
  return cached_map(map, MapKey{ptr, bh, n, d, 16, rows}, [&](CUtensorMap* m) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)bh};
    cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)n * d * 4};
    cuuint32_t box[3] = {(cuuint32_t)d, rows, 1};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estride,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
  });
}

unsigned long long watchdog_limit_ns() { return g_watchdog_ns.load(std::memory_order_relaxed); }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) { return overlaps(a, na, b, nb); }

int launch_forward(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int D,
                   float scale, int is_causal, int dtype, void* workspace, size_t workspace_bytes, bool balanced,
                   cudaStream_t stream) {
  return ::launch(Q, K, V, O, LSE, B, H, N, D, scale, is_causal, dtype, workspace, workspace_bytes,
                  balanced ? FA2_SCHED_BALANCED : FA2_SCHED_UNITS, stream);
}

// Cost of each schedule in K/V-tile steps of the busiest SM (a step: one
// work unit against one 128-key tile). Rounds: ceil(units / SMs) rounds of
// whole units. Balanced: total steps / SMs plus kSplitCostSteps for the
// partial-result write and merge of the units it cuts. Balanced is taken
// when at least 5 % cheaper, for non-causal work only: the heaviest-first
// zig-zag rounds measured faster than the split on every causal workload.
int fwd_auto_schedule(long long B, long long H, long long N, int D, int is_causal, int sms) {
  constexpr double kSplitCostSteps = 4.0;
  const long long rows = fwd_unit_rows(D);
  const long long units = B * H * ((N + rows - 1) / rows);
  if (is_causal || units <= 0 || sms <= 0 || fwd_dtiled(D)) return FA2_SCHED_UNITS;
  const long long nkv = (N + kKeys - 1) / kKeys;
  const double rounds_cost = static_cast<double>((units + sms - 1) / sms) * static_cast<double>(nkv);
  const double balanced_cost = static_cast<double>(units) * static_cast<double>(nkv) / sms + kSplitCostSteps;
  return balanced_cost < 0.95 * rounds_cost ? FA2_SCHED_BALANCED : FA2_SCHED_UNITS;
}
}  // namespace fa2

extern "C" int fa2_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                       int D, float scale, int is_causal, int dtype, struct CUstream_st* stream) {
  return launch(Q, K, V, O, LSE, B, H, N, D, scale, is_causal, dtype, nullptr, 0, FA2_SCHED_UNITS,
                reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fa2_fwd_schedule_for(int B, int H, int N, int D, int is_causal, int sms, int* schedule) {
  if (!schedule || B < 0 || H < 0 || N < 0 || sms < 1) return FA2_ERR_INVALID_ARG;
  if (!fwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  *schedule = fwd_auto_schedule(B, H, N, D, is_causal, sms);
  return FA2_OK;
}

extern "C" int fa2_fwd_sched(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                             int D, float scale, int is_causal, int dtype, void* workspace, size_t workspace_bytes,
                             int schedule, struct CUstream_st* stream) {
  if (schedule != FA2_SCHED_AUTO && schedule != FA2_SCHED_UNITS && schedule != FA2_SCHED_BALANCED)
    return FA2_ERR_INVALID_ARG;
  // the balanced schedule needs a workspace (none at head dims 512 and 1024,
  // which run the rounds)
  if (schedule == FA2_SCHED_BALANCED && !workspace && B > 0 && H > 0 && N > 0 && !fwd_dtiled(D))
    return FA2_ERR_INVALID_ARG;
  return launch(Q, K, V, O, LSE, B, H, N, D, scale, is_causal, dtype, workspace, workspace_bytes, schedule,
                reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fa2_fwd_workspace_bytes(int D, size_t* bytes) {
  if (!bytes) return FA2_ERR_INVALID_ARG;
  if (!fwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  DeviceInfo* info = device_info(dev);
  if (!info) return FA2_ERR_UNSUPPORTED;
  if (info->err != cudaSuccess) return record_cuda(info->err);
  *bytes = stream_k_workspace_bytes(info->sms, D);
  return FA2_OK;
}

extern "C" int fa2_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                          int D, float scale, int is_causal, int dtype, void* workspace, size_t workspace_bytes,
                          struct CUstream_st* stream) {
  return launch(Q, K, V, O, LSE, B, H, N, D, scale, is_causal, dtype, workspace, workspace_bytes,
                workspace ? FA2_SCHED_BALANCED : FA2_SCHED_UNITS, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fa2_device_status(struct CUstream_st* stream, int* status, int clear) {
  if (!status) return FA2_ERR_INVALID_ARG;
  DeviceInfo* info = nullptr;
  const int rc = current_device(&info);
  if (rc != FA2_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, info->status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) {
    e = cudaMemsetAsync(info->status, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  if (e != cudaSuccess) return record_cuda(e);
  *status = v;
  return v != 0 ? FA2_ERR_TIMEOUT : FA2_OK;
}

extern "C" int fa2_set_watchdog_ns(unsigned long long ns) {
  g_watchdog_ns.store(ns ? ns : kDefaultWatchdogNs, std::memory_order_relaxed);
  return FA2_OK;
}

extern "C" int fa2_test_withhold_next_load(int enable) {
  g_test_withhold.store(enable ? 1 : 0, std::memory_order_relaxed);
  return FA2_OK;
}

extern "C" const char* fa2_error_string(int code) {
  switch (code) {
    case FA2_OK: return "ok";
    case FA2_ERR_INVALID_ARG: return "invalid argument";
    case FA2_ERR_UNSUPPORTED: return "unsupported head dimension, dtype or device";
    case FA2_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
    case FA2_ERR_CUDA: return "CUDA call failed";
    case FA2_ERR_TIMEOUT: return "device watchdog timeout";
    default: return "unknown status";
  }
}

extern "C" const char* fa2_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int fa2_version(void) { return (1 << 16) | 1; }
