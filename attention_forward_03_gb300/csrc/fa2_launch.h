// Host-visible pieces of the forward and backward kernels: tile constants,
// the parameter blocks, and the launcher templates (instantiated in
// fa2_fwd_d32.cu, fa2_fwd_d64.cu, fa2_fwd_d96.cu, fa2_fwd_d128.cu,
// fa2_fwd_d256.cu and fa2_bwd_d{32,64,96,128}.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

#include <mutex>

namespace fa2 {

// Devices the library keeps per-device state for (set-up done once per device).
constexpr int kMaxDevices = 64;

// One-time, per-device preparation of a kernel (its function attributes):
// `prep` runs once for each device, with that device current, and its result
// is returned to every later call on the device. Devices past the table run
// `prep` on every call.
struct PerDeviceOnce {
  std::once_flag flag[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
};

template <typename F>
cudaError_t once_per_device(PerDeviceOnce& o, F&& prep) {
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return prep();
  std::call_once(o.flag[dev], [&] { o.err[dev] = prep(); });
  return o.err[dev];
}

constexpr int kRows = 128;          // query rows per sub-tile (= TMEM lanes)
constexpr int kSubTiles = 2;        // sub-tiles per work unit
constexpr int kKeys = 128;          // keys per K/V tile

// Head dimensions of the forward kernels. 64 and 128 are native; 32 and 96
// run in the layout of the next multiple of 64, the padded columns of every
// Q/K/V tile read as zeros (the copy engine's out-of-bounds fill), so they
// add nothing to Q.K^T and P.V. 256 has a kernel of its own with one
// 128-row query sub-tile per work unit (its O accumulator takes half of the
// tensor memory). 512 and 1024 tile the output's head dimension: a work unit
// is 128 query rows and one 256-column chunk of O (fa2_kernel_dtile.cuh).
constexpr int kDtileOutCols = 256;  // output columns per work unit at head dims 512 and 1024
constexpr bool fwd_head_dim_ok(int d) {
  return d == 32 || d == 64 || d == 96 || d == 128 || d == 256 || d == 512 || d == 1024;
}
constexpr bool fwd_dtiled(int d) { return d >= 512; }
constexpr int fwd_unit_subtiles(int d) { return d >= 256 ? 1 : kSubTiles; }
constexpr int fwd_unit_rows(int d) { return kRows * fwd_unit_subtiles(d); }
// Output chunks per query tile: the units of one query tile.
constexpr int fwd_out_chunks(int d) { return fwd_dtiled(d) ? d / kDtileOutCols : 1; }

struct Params {
  void* o;                  // [B,H,N,D] 16-bit
  float* lse;               // [B,H,N]
  int* status;              // device watchdog word
  unsigned long long watchdog_ns;
  int N;
  int BH;                   // heads B*H; at head dims 512 and 1024 B*H times the output chunks (each
                            // (head, chunk) pair is scheduled as a head of its own)
  int n_qt;                 // query work units per head = ceil(N / unit rows)
  int num_units;            // BH * n_qt
  int nkv_full;             // K/V tiles of a full row = ceil(N / 128)
  float scale_log2;         // scale * log2(e)
  // Schedule. 0: whole units dealt to CTAs in rounds. 1 (stream-K): CTA b
  // takes K/V-tile steps [total*b/G, total*(b+1)/G) of the unit sequence;
  // units cut between CTAs are merged through the workspace below.
  int stream_k;
  long long steps_per_head; // K/V-tile steps of all units of one head
  long long total_steps;    // BH * steps_per_head
  // (T = sub-tiles per unit: 2, or 1 at head dim 256)
  float* ws_o;              // [G][T][D][128] fp32 partial O (unnormalised)
  float* ws_stats;          // [G][T][3][128] base, l, l_o of each partial row
  unsigned long long* ws_flags;  // [G][T] = epoch once that partial is written
  unsigned long long epoch; // unique tag of this launch
  int test_withhold;        // test hook: the producer withholds its first K/V tile
};

constexpr int kBwdKeys = 128;       // keys per backward work unit (= TMEM lanes)
// Head dimensions of the backward kernel (32 and 96 in the tiles of 64 and 128).
constexpr bool bwd_head_dim_ok(int d) { return d == 32 || d == 64 || d == 96 || d == 128; }
// Query rows per backward step: 128 at head dims up to 64 (the tensor
// memory then holds 128-column S^T, dP^T and dQ^T beside dV and dK), else 64.
constexpr int bwd_step_rows(int d) { return d <= 64 ? 128 : 64; }

struct BwdParams {
  void* dk;                 // [B,H,N,D] 16-bit outputs
  void* dv;
  float* dq_acc;            // [B,H,N,D] fp32 dQ accumulator (zeroed by the prologue kernel; the
                            // kernel adds into it through a tensor map)
  const float* neg_lse2;    // [B*H, Npad] -LSE * log2(e) (the exponent's offset); -inf for rows >= N
  const float* delta;       // [B*H, Npad] <dO_i, O_i>; 0 for rows >= N
  int* status;              // device watchdog word
  unsigned long long watchdog_ns;
  int N;
  int Npad;                 // N rounded up to a multiple of the step rows
  int BH;
  int nkv;                  // K/V tiles (work units) per head = ceil(N / 128)
  int nq;                   // query steps per head = Npad / step rows
  int num_units;            // BH * nkv
  float scale_log2;         // scale * log2(e)
  float scale;
  // Schedule. 0: whole units dealt to CTAs in rounds. 1 (stream-K): CTA b
  // takes query steps [total*b/G, total*(b+1)/G) of the unit sequence
  // (heads in order, K/V tiles ascending); a unit cut between CTAs is
  // finished by the CTA holding its first steps, which adds the partial dK,
  // dV the following CTAs left in the workspace.
  int stream_k;
  long long steps_per_head; // query steps of all units of one head
  long long total_steps;    // BH * steps_per_head
  float* ws_part;           // [G][2][D][128] fp32 partial dV, dK (unscaled) of a cut unit
  unsigned long long* ws_flags;  // [G] = epoch once that partial is written
  unsigned long long epoch; // unique tag of this launch
  int test_withhold;        // test hook: the producer withholds its first K/V tile
};

// CTAs of the backward's stream-K schedule at most (its partial slots are
// part of the caller's workspace, which is sized without a device).
constexpr int kBwdMaxCtas = 160;

// Bytes of stream-K workspace for `grid` CTAs at head dimension d (none at
// head dims 512 and 1024, which run on the round schedule only).
constexpr size_t stream_k_workspace_bytes(int grid, int d) {
  return fwd_dtiled(d) ? 0
                       : (static_cast<size_t>(grid) * fwd_unit_subtiles(d) *
                              ((static_cast<size_t>(d) * 128 + 3 * 128) * sizeof(float)) +
                          255) / 256 * 256 +
                             static_cast<size_t>(grid) * fwd_unit_subtiles(d) * 8;
}

// The full forward call (validation, tensor maps, launch) with an optional
// stream-K workspace; the C entry points are thin wrappers around it. With
// `balanced` false the round schedule runs whatever the workspace.
int launch_forward(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int D,
                   float scale, int is_causal, int dtype, void* workspace, size_t workspace_bytes, bool balanced,
                   cudaStream_t stream);

// The forward schedule with less work on the busiest SM (FA2_SCHED_UNITS or
// FA2_SCHED_BALANCED) for a problem on a device with `sms` SMs; see
// fa2_fwd_schedule_for in include/fa2.h.
int fwd_auto_schedule(long long B, long long H, long long N, int D, int is_causal, int sms);

// Records `e` as the calling thread's last CUDA error (fa2_last_cuda_error)
// and returns FA2_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// A tag no earlier launch of this process (or of another one) has used, for
// the flags of cross-CTA partial results.
unsigned long long next_launch_epoch();

// The watchdog test hook's request (fa2_test_withhold_next_load), taken by
// the launch that calls this (one launch only).
int take_test_withhold();

// Shared with the backward pass: the current device's SM count and watchdog
// word (FA2_ERR_UNSUPPORTED unless it is a compute-capability 10.3 GPU; the
// capability is checked before anything that needs this library's device
// code on the device), a
// 128-byte-swizzled [B*H, N, D] tensor map with boxes of `rows` rows x 64
// elements, the watchdog limit, and an address-range overlap test.
int current_device_facts(int* sms, int** status);
bool encode_tile_map(CUtensorMap* map, const void* ptr, int bh, int n, int d, int dtype, unsigned rows);
unsigned long long watchdog_limit_ns();
// fp32 [B*H, N, D] map with boxes of `rows` whole rows (D elements), no swizzle.
bool encode_f32_rows_map(CUtensorMap* map, float* ptr, int bh, int n, int d, unsigned rows);
// fp32 [bh][n][d] in boxes of 32 columns x `rows` rows, 128-byte swizzled in
// shared memory (the backward's dQ staging at head dims up to 64).
bool encode_f32_cols_map_sw128(CUtensorMap* map, float* ptr, int bh, int n, int d, unsigned rows);
bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb);

template <int D, bool kBf16, bool kCausal>
cudaError_t launch_bwd(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const CUtensorMap& dout,
                       const CUtensorMap& dq_acc, const BwdParams& p, int grid, cudaStream_t stream);

// q, k, v: the input maps; o: the output's map (boxes of 128 rows x 64
// elements, 128-byte swizzle), through which the kernel stores O at D >= 96.
template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                       const Params& p, int grid, cudaStream_t stream);

// Head dim 256 (fa2_kernel_wide.cuh, instantiated in fa2_fwd_d256.cu).
template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd_wide(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                            const Params& p, int grid, cudaStream_t stream);

// Head dims 512 and 1024 (fa2_kernel_dtile.cuh, instantiated in
// fa2_fwd_d512.cu and fa2_fwd_d1024.cu); round schedule only.
template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd_dtile(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                             const Params& p, int grid, cudaStream_t stream);

}  // namespace fa2
