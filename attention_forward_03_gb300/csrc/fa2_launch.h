// Host-visible pieces of the forward kernel: tile constants, the parameter
// block, and the launcher template (instantiated in fa2_fwd_d64.cu and
// fa2_fwd_d128.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>

namespace fa2 {

constexpr int kRows = 128;          // query rows per sub-tile (= TMEM lanes)
constexpr int kSubTiles = 2;        // sub-tiles per work unit
constexpr int kUnitRows = kRows * kSubTiles;
constexpr int kKeys = 128;          // keys per K/V tile

struct Params {
  void* o;                  // [B,H,N,D] 16-bit
  float* lse;               // [B,H,N]
  int* status;              // device watchdog word
  unsigned long long watchdog_ns;
  int N;
  int BH;
  int n_qt;                 // query work units per head = ceil(N / 256)
  int num_units;            // BH * n_qt
  int nkv_full;             // K/V tiles of a full row = ceil(N / 128)
  float scale_log2;         // scale * log2(e)
  // Schedule. 0: whole units dealt to CTAs in rounds. 1 (stream-K): CTA b
  // takes K/V-tile steps [total*b/G, total*(b+1)/G) of the unit sequence;
  // units cut between CTAs are merged through the workspace below.
  int stream_k;
  long long steps_per_head; // K/V-tile steps of all units of one head
  long long total_steps;    // BH * steps_per_head
  float* ws_o;              // [G][2][D][128] fp32 partial O (unnormalised)
  float* ws_stats;          // [G][2][3][128] base, l, l_o of each partial row
  unsigned long long* ws_flags;  // [G][2] = epoch once that partial is written
  unsigned long long epoch; // unique tag of this launch
  int test_withhold;        // test hook: the producer withholds its first K/V tile
};

// Bytes of stream-K workspace for `grid` CTAs at head dimension d.
constexpr size_t stream_k_workspace_bytes(int grid, int d) {
  return (static_cast<size_t>(grid) * (2ull * (static_cast<size_t>(d) * 128 + 3 * 128) * sizeof(float)) + 255) /
             256 * 256 +
         static_cast<size_t>(grid) * 2 * 8;
}

// The full forward call (validation, tensor maps, launch) with an optional
// stream-K workspace; the C entry points are thin wrappers around it.
int launch_forward(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int D,
                   float scale, int is_causal, int dtype, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream);

// Records `e` as the calling thread's last CUDA error (fa2_last_cuda_error)
// and returns FA2_ERR_CUDA.
int record_cuda_error(cudaError_t e);

template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const Params& p,
                       int grid, cudaStream_t stream);

}  // namespace fa2
