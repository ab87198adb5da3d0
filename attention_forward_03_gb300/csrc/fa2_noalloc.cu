// A forward entry point that allocates nothing: the stream-K schedule of
// fa2_fwd_ws, with its scratch in a fixed device array of this library
// instead of caller memory. See fa2_fwd_noalloc in include/fa2.h.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "fa2.h"
#include "fa2_launch.h"

namespace {

// Largest configuration the static scratch covers: 160 CTAs (one per SM) at
// head dimension 128 (smaller head dimensions need less).
constexpr int kMaxCtas = 160;
constexpr size_t kScratchBytes = fa2::stream_k_workspace_bytes(kMaxCtas, 128);
static_assert(kScratchBytes == 21465600, "the size stated in fa2.h");
static_assert(fa2::stream_k_workspace_bytes(kMaxCtas, 256) <= kScratchBytes, "head dim 256 fits as well");

// Every GPU that loads this module holds this array until the process exits.
// In host code `g_scratch` is only a stand-in for the symbol: its device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct Setup {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  int sms = 0;
  void* ptr = nullptr;
};
Setup g_setup[fa2::kMaxDevices];

}  // namespace

extern "C" int fa2_fwd_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                               int N, int D, float scale, int is_causal, int dtype, struct CUstream_st* stream) {
  // the same argument checks fa2_fwd makes before it touches the device
  if (B < 0 || H < 0 || N < 0) return FA2_ERR_INVALID_ARG;
  if (!fa2::fwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  if (dtype != FA2_F16 && dtype != FA2_BF16) return FA2_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || N == 0) return FA2_OK;

  // The device must be one this library runs on (compute capability 10.3)
  // before anything below touches its device code.
  int sms = 0;
  int* status = nullptr;
  const int rc = fa2::current_device_facts(&sms, &status);
  if (rc != FA2_OK) return rc;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fa2::record_cuda_error(e);
  if (dev < 0 || dev >= fa2::kMaxDevices) return FA2_ERR_UNSUPPORTED;
  Setup& s = g_setup[dev];
  // Set-up on the first call on this device (with it current): the device
  // address of the static scratch. With lazy module loading (the CUDA 12+
  // default) this is also when the array's memory is committed on the device.
  std::call_once(s.once, [&] {
    s.sms = sms;
    s.err = cudaGetSymbolAddress(&s.ptr, g_scratch);
  });
  if (s.err != cudaSuccess) return fa2::record_cuda_error(s.err);
  if (s.ptr == nullptr) return fa2::record_cuda_error(cudaErrorInvalidSymbol);
  // The scratch holds one partial result per CTA; a device with more SMs
  // than it covers is refused rather than run with a cut-down grid.
  if (s.sms > kMaxCtas) return FA2_ERR_UNSUPPORTED;
  return fa2::launch_forward(Q, K, V, O, LSE, B, H, N, D, scale, is_causal, dtype, s.ptr, kScratchBytes, true,
                             reinterpret_cast<cudaStream_t>(stream));
}
