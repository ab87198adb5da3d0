// Host-visible pieces of the forward kernel: tile constants, the parameter
// block, and the launcher template (instantiated in fa2_fwd_d64.cu and
// fa2_fwd_d128.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

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
  float scale_log2;         // scale * log2(e)
};

template <int D, bool kBf16, bool kCausal>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const Params& p,
                       int grid, cudaStream_t stream);

}  // namespace fa2
