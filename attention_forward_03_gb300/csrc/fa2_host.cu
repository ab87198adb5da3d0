// End-to-end forward from host memory: the inputs are copied to the device,
// the forward pass runs and the outputs are copied back, in chunks of whole
// heads so that the copies of one chunk overlap the computation of another.
// Contract: fa2_fwd_host in include/fa2.h.
//
// Per chunk c of heads [h0, h0 + nh):
//   copy-in stream : Q, K, V rows of the chunk, host -> device
//   caller stream  : waits for them, then the forward kernel on the chunk
//   copy-out stream: waits for the kernel, then O and LSE rows, device -> host
// Every copy costs a few microseconds of the copy engine's time besides its
// bytes (measured on GB300: 48 MB host -> device in 24 copies 289.5 us, in 8
// two-dimensional copies 253.2 us, in one 240.6 us), so the call makes as
// few as the layout allows: when Q, K, V lie equally spaced in host memory
// (slices of one packed [3, B, H, N, D] buffer, for one) a chunk's three
// blocks move in one cudaMemcpy2DAsync, and when the device can address the
// host LSE buffer directly (page-locked memory under unified addressing)
// the kernels write LSE there and no LSE copy is made.
// The caller's stream is the ordering point: the copy streams wait for its
// work before the first copy, and it waits for the last copy before returning
// control of its queue, so the whole call behaves as stream-ordered work.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa2.h"
#include "fa2_launch.h"

namespace {

using fa2::kMaxDevices;

// Two non-blocking copy streams and four events per device, created on first
// use and kept for the life of the process. A stream wait binds to the event's
// latest record at the time it is enqueued, so one event can be re-recorded
// for every chunk; the per-device lock keeps another thread's records from
// interleaving with an enqueue in progress.
struct CopyPipes {
  std::mutex mu;
  bool ready = false;
  size_t max_pitch = 0;  // the device's limit on a 2-D copy's pitch
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t entry = nullptr, copied_in = nullptr, computed = nullptr, done = nullptr;
};
CopyPipes g_pipes[kMaxDevices];

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Device buffer layout: Q | K | V | O | LSE | stream-K workspace, each part
// starting on a 256-byte boundary. The LSE part holds each chunk's rows from
// a 16-byte boundary (the kernel's alignment rule), so it is sized for the
// worst case of one head per chunk: B*H*N floats plus 3 floats of padding
// per head (there are never more chunks than heads).
struct BufferLayout {
  size_t k, v, o, lse, ws, ws_bytes, total;
};

int buffer_layout(int B, int H, int N, int D, BufferLayout* L) {
  if (B < 0 || H < 0 || N < 0) return FA2_ERR_INVALID_ARG;
  if (!fa2::fwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  const int64_t bh = static_cast<int64_t>(B) * H;
  if (bh > INT32_MAX) return FA2_ERR_INVALID_ARG;
  const size_t t = round256(static_cast<size_t>(bh) * N * D * 2);
  const size_t l = round256(static_cast<size_t>(bh) * N * 4 + static_cast<size_t>(bh) * 12);
  size_t ws = 0;
  const int rc = fa2_fwd_workspace_bytes(D, &ws);
  if (rc != FA2_OK) return rc;
  L->k = t;
  L->v = 2 * t;
  L->o = 3 * t;
  L->lse = 4 * t;
  L->ws = 4 * t + l;
  L->ws_bytes = ws;
  L->total = L->ws + round256(ws);
  return FA2_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

cudaError_t make_pipes(CopyPipes& p, int dev) {
  int mp = 0;
  cudaError_t e = cudaDeviceGetAttribute(&mp, cudaDevAttrMaxPitch, dev);
  p.max_pitch = e == cudaSuccess && mp > 0 ? static_cast<size_t>(mp) : 0;
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
  for (cudaEvent_t* ev : {&p.entry, &p.copied_in, &p.computed, &p.done})
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  return e;
}

}  // namespace

extern "C" int fa2_fwd_host_buffer_bytes(int B, int H, int N, int D, size_t* bytes) {
  if (!bytes) return FA2_ERR_INVALID_ARG;
  BufferLayout L;
  const int rc = buffer_layout(B, H, N, D, &L);
  if (rc != FA2_OK) return rc;
  *bytes = L.total;
  return FA2_OK;
}

extern "C" int fa2_fwd_host(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                            int D, float scale, int is_causal, int dtype, int heads_per_chunk, int balanced,
                            void* dev_buffer, size_t dev_bytes, struct CUstream_st* stream_handle) {
  if (B < 0 || H < 0 || N < 0 || heads_per_chunk < 0) return FA2_ERR_INVALID_ARG;
  if (!fa2::fwd_head_dim_ok(D)) return FA2_ERR_UNSUPPORTED;
  if (dtype != FA2_F16 && dtype != FA2_BF16) return FA2_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA2_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return FA2_OK;
  if (!Q || !K || !V || !O || !LSE || !dev_buffer) return FA2_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(dev_buffer) & 255u) return FA2_ERR_ALIGN;
  const int64_t bh64 = static_cast<int64_t>(B) * H;
  if (bh64 > INT32_MAX) return FA2_ERR_INVALID_ARG;
  const int bh = static_cast<int>(bh64);
  const size_t head_elems = static_cast<size_t>(N) * D;
  const size_t tbytes = static_cast<size_t>(bh) * head_elems * 2;
  const size_t lbytes = static_cast<size_t>(bh) * N * 4;
  if (overlaps(O, tbytes, Q, tbytes) || overlaps(O, tbytes, K, tbytes) || overlaps(O, tbytes, V, tbytes) ||
      overlaps(LSE, lbytes, Q, tbytes) || overlaps(LSE, lbytes, K, tbytes) || overlaps(LSE, lbytes, V, tbytes) ||
      overlaps(LSE, lbytes, O, tbytes))
    return FA2_ERR_INVALID_ARG;
  BufferLayout L;
  int rc = buffer_layout(B, H, N, D, &L);
  if (rc != FA2_OK) return rc;
  if (dev_bytes < L.total) return FA2_ERR_INVALID_ARG;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fa2::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_UNSUPPORTED;
  CopyPipes& pp = g_pipes[dev];
  std::lock_guard<std::mutex> lock(pp.mu);
  if (!pp.ready) {
    e = make_pipes(pp, dev);
    if (e != cudaSuccess) return fa2::record_cuda_error(e);
    pp.ready = true;
  }

  // Q, K, V as three rows of one pitched block: equally spaced, in that
  // order, without overlap, and within the device's pitch limit. The driver
  // takes such a copy only when the block lies in one allocation (separately
  // allocated buffers can be equally spaced too); a 2-D copy it refuses is
  // refused at the call, nothing is enqueued, and the call falls back to
  // three copies per chunk.
  const char* hq = static_cast<const char*>(Q);
  const char* hk = static_cast<const char*>(K);
  const char* hv = static_cast<const char*>(V);
  const uintptr_t uq = reinterpret_cast<uintptr_t>(hq), uk = reinterpret_cast<uintptr_t>(hk),
                  uv = reinterpret_cast<uintptr_t>(hv);
  bool packed = uk > uq && uk - uq >= tbytes && uv > uk && uv - uk == uk - uq && uk - uq <= pp.max_pitch &&
                      L.k <= pp.max_pitch;
  // LSE straight from the kernels into host memory the device can address
  // (rows of a chunk must start on 16 bytes, as every LSE pointer of the
  // kernels).
  float* lse_direct = nullptr;
  {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, LSE) == cudaSuccess) {
      if (pa.type == cudaMemoryTypeHost && pa.devicePointer != nullptr && N % 4 == 0 &&
          (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15u) == 0)
        lse_direct = static_cast<float*>(pa.devicePointer);
    } else {
      cudaGetLastError();  // not an error of this call: the copy path is taken
    }
  }

  const int hpc = heads_per_chunk > 0 ? (heads_per_chunk < bh ? heads_per_chunk : bh) : (bh + 3) / 4;
  char* base = static_cast<char*>(dev_buffer);
  char* dq = base;
  char* dk = base + L.k;
  char* dv = base + L.v;
  char* dout = base + L.o;
  float* dlse = reinterpret_cast<float*>(base + L.lse);
  // The first chunk is half the size (so the first kernel starts sooner);
  // the others hold hpc heads, the last what remains (half a chunk when B*H
  // is a multiple of hpc, so the work after the last copy-in is short too).
  const int first = hpc >= 2 ? hpc / 2 : hpc;
  size_t lse_at = 0;  // device LSE rows of the next chunk start here (a multiple of 4 floats)
  void* ws = balanced ? static_cast<void*>(base + L.ws) : nullptr;
  char* hout = static_cast<char*>(O);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_handle);

  e = cudaEventRecord(pp.entry, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.in, pp.entry, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.out, pp.entry, 0);
  if (e != cudaSuccess) return fa2::record_cuda_error(e);
  rc = FA2_OK;
  for (int h0 = 0, nh = 0; h0 < bh && rc == FA2_OK; h0 += nh) {
    nh = h0 == 0 ? first : hpc;
    if (nh > bh - h0) nh = bh - h0;
    const size_t off = static_cast<size_t>(h0) * head_elems * 2;
    const size_t n = static_cast<size_t>(nh) * head_elems * 2;
    const size_t loff = static_cast<size_t>(h0) * N;  // host LSE rows of the chunk
    float* dl = lse_direct ? lse_direct + loff : dlse + lse_at;
    lse_at = (lse_at + static_cast<size_t>(nh) * N + 3) / 4 * 4;
    if (packed) {
      // rows Q, K, V of the chunk: host pitch = their spacing, device pitch = L.k
      e = cudaMemcpy2DAsync(dq + off, L.k, hq + off, uk - uq, n, 3, cudaMemcpyHostToDevice, pp.in);
      if (e == cudaErrorInvalidValue || e == cudaErrorInvalidPitchValue) {
        cudaGetLastError();
        packed = false;
      }
    }
    if (!packed) {
      e = cudaMemcpyAsync(dq + off, hq + off, n, cudaMemcpyHostToDevice, pp.in);
      if (e == cudaSuccess) e = cudaMemcpyAsync(dk + off, hk + off, n, cudaMemcpyHostToDevice, pp.in);
      if (e == cudaSuccess) e = cudaMemcpyAsync(dv + off, hv + off, n, cudaMemcpyHostToDevice, pp.in);
    }
    if (e == cudaSuccess) e = cudaEventRecord(pp.copied_in, pp.in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, pp.copied_in, 0);
    if (e != cudaSuccess) {
      rc = fa2::record_cuda_error(e);
      break;
    }
    rc = fa2::launch_forward(dq + off, dk + off, dv + off, dout + off, dl, 1, nh, N, D, scale, is_causal, dtype, ws,
                             ws ? L.ws_bytes : 0, ws != nullptr, s);
    if (rc != FA2_OK) break;
    e = cudaEventRecord(pp.computed, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.out, pp.computed, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hout + off, dout + off, n, cudaMemcpyDeviceToHost, pp.out);
    if (e == cudaSuccess && !lse_direct)
      e = cudaMemcpyAsync(LSE + loff, dl, static_cast<size_t>(nh) * N * 4, cudaMemcpyDeviceToHost, pp.out);
    if (e != cudaSuccess) rc = fa2::record_cuda_error(e);
  }
  // Whatever was enqueued, the caller's stream ends behind all of it.
  e = cudaEventRecord(pp.done, pp.out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, pp.done, 0);
  if (e == cudaSuccess) e = cudaEventRecord(pp.done, pp.in);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, pp.done, 0);
  if (e != cudaSuccess && rc == FA2_OK) rc = fa2::record_cuda_error(e);
  return rc;
}
